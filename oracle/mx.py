"""MX element/scale codecs and the MX block quantizer (CPU oracle, float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Formats (OCP MX v1.0; named on "Quantization on Ascend", MoE MXFP8 notes):

* e4m3fn element: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
  Exponent field 0 is subnormal (value m/8 * 2^-6), codes 0x7F/0xFF are NaN,
  there is no infinity, the largest finite magnitude is 448 (0x7E).
* UE8M0 (e8m0) scale: one unsigned byte b meaning 2^(b - 127) ("uint8 (e8m0,
  exponent + 127)" in the offline-path note).  Byte 0xFF is NaN and is never
  produced here.  There is no zero point (sglang PR #32266, commit note on the
  missing w13/w2 weight offset: "a pure scale format").
* A block is 32 consecutive elements along the contraction axis K.
* e2m1 (FP4) element, the MXFP4 weight format of the W4A8 path ("Quantization
  on Ascend", W4A8 notes: packed FP4 float4_e2m1fn_x2, two nibbles per byte,
  UE8M0 shared exponent per 32-element block): 1 sign bit, 2 exponent bits
  (bias 1), 1 mantissa bit; exponent field 0 is subnormal (value m/2); no
  NaN or infinity; the largest magnitude is 6.
"""

from __future__ import annotations

import math

import numpy as np

BLOCK = 32
E8M0_BIAS = 127
E4M3_MAX = 448.0
# largest power-of-two exponent of an e4m3 value (2^8 = 256 <= 448 < 512)
E4M3_EMAX = 8
E2M1_MAX = 6.0
# largest power-of-two exponent of an e2m1 value (2^2 = 4 <= 6 < 8)
E2M1_EMAX = 2


# ----------------------------------------------------------------------------
# e4m3fn codec
# ----------------------------------------------------------------------------

def _build_e4m3_table() -> np.ndarray:
    """Decode table for all 256 e4m3fn codes, from the bit-field definition."""
    t = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            t[code] = np.nan
        elif e == 0:
            t[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            t[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


E4M3_TABLE = _build_e4m3_table()
# non-negative finite codes 0x00..0x7E in increasing order of value
_E4M3_POS = E4M3_TABLE[:0x7F].copy()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 e4m3fn codes -> float64 values."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float64 -> e4m3fn code, round-to-nearest-even, saturating to +-448.

    The magnitude is first clamped to 448 (saturation: anything that would
    round above the largest finite value becomes 448), then rounded to the
    nearest point of the non-negative grid; an exact midpoint goes to the code
    with an even mantissa (the code's low bit is the mantissa's low bit).  The
    sign bit is kept, so a negative value that rounds to zero gives 0x80.
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3_encode: non-finite input is outside the contract")
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a, side="left")  # first grid point >= a
    hi = np.clip(hi, 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << 7
    return (mag | sign).astype(np.uint8)


# ----------------------------------------------------------------------------
# e2m1 codec (FP4)
# ----------------------------------------------------------------------------

def _build_e2m1_table() -> np.ndarray:
    """Decode table for the 16 e2m1 codes, from the bit-field definition."""
    t = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        if e == 0:
            t[code] = sign * (m / 2.0) * 2.0 ** (1 - 1)
        else:
            t[code] = sign * (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return t


E2M1_TABLE = _build_e2m1_table()
_E2M1_POS = E2M1_TABLE[:8].copy()   # codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """e2m1 codes (uint8 values 0..15) -> float64 values."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """float64 -> e2m1 code (0..15), round-to-nearest-even, saturating to +-6.

    As for e4m3: the magnitude is clamped to 6, rounded to the nearest point
    of the non-negative grid with an exact midpoint going to the even code
    (even mantissa bit), and the sign bit is kept (-0 -> 0x8).
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e2m1_encode: non-finite input is outside the contract")
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.clip(np.searchsorted(_E2M1_POS, a, side="left"), 0, 7)
    lo = np.clip(hi - 1, 0, 7)
    d_lo = a - _E2M1_POS[lo]
    d_hi = _E2M1_POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(take_hi, hi, lo).astype(np.uint8)
    return mag | (np.signbit(v).astype(np.uint8) << 3)


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """[..., K] e2m1 codes -> [..., K/2] bytes, element 2i in the low nibble
    and element 2i+1 in the high nibble (K even)."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    if c.shape[-1] % 2:
        raise ValueError("pack_fp4: K must be even")
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_fp4: [..., K/2] bytes -> [..., K] e2m1 codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def e4m3_ulp(a: np.ndarray) -> np.ndarray:
    """Spacing of the e4m3 grid at magnitude ``a`` (|a| <= 448)."""
    a = np.abs(np.asarray(a, dtype=np.float64))
    _, ex = np.frexp(np.maximum(a, 2.0 ** -6))  # a = f * 2^ex, f in [0.5, 1)
    return np.ldexp(1.0, ex - 1 - 3)


# ----------------------------------------------------------------------------
# bf16 (output dtype of GEMM2 and finalize)
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit pattern, round-to-nearest-even, directly from fp64.

    bf16 keeps 8 significant bits; for |v| >= 2^-126 the grid spacing is
    2^(floor(log2|v|) - 7), below that it is the subnormal step 2^-133.
    Rounding is done on the exact value (no intermediate fp32 rounding).
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("f64_to_bf16_bits: non-finite input")
    a = np.abs(v)
    _, ex = np.frexp(a)  # a = f * 2^ex, f in [0.5,1): floor(log2 a) = ex - 1
    step_exp = np.where(a >= 2.0 ** -126, ex - 1 - 7, -133)
    r = np.ldexp(np.round(np.ldexp(a, -step_exp)), step_exp)  # np.round: half-even
    r = np.where(np.signbit(v), -r, r)
    if np.any(np.abs(r) > 3.3895313892515355e38):
        raise OverflowError("bf16 overflow")
    f32 = r.astype(np.float32)  # exact: r is on the bf16 grid
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# UE8M0 block scale and the MX block quantizer
# ----------------------------------------------------------------------------

def e8m0_scale_exponent(amax: np.ndarray, emax: int = E4M3_EMAX) -> np.ndarray:
    """Shared-scale exponent s of a block from its amax (OCP MX v1.0 6.3).

    s = floor(log2(amax)) - emax, emax the element format's largest
    power-of-two exponent (8 for e4m3, 2 for e2m1), clamped to the e8m0 range
    [-127, 127]; an all-zero block (amax = 0) takes the smallest scale
    s = -127.  floor(log2) is read off the binary exponent (frexp), so it is
    exact for every fp64.
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    s = (ex - 1) - emax
    s = np.where(amax > 0, s, -127)
    return np.clip(s, -127, 127).astype(np.int64)


def mx_quantize(x: np.ndarray, block: int = BLOCK):
    """MX-quantize ``x`` along its last axis in blocks of ``block`` elements.

    Returns (q uint8 [..., K], scale uint8 [..., ceil(K/block)]).  The last
    block may be partial (K % 32 != 0): its amax is taken over the elements
    that exist, and its scale is one more entry of the ceil(K/32) scales
    (PR #32266 summary, "Offline partial MXFP8 block-scale layout").

    Per block: amax = max|x|; s = e8m0_scale_exponent(amax); the scale byte is
    s + 127; each element is q = e4m3_encode(x * 2^-s) (exact scaling).
    """
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("mx_quantize: non-finite input is outside the contract")
    K = x.shape[-1]
    nb = -(-K // block)
    pad = nb * block - K
    xp = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1) if pad else x
    xb = xp.reshape(x.shape[:-1] + (nb, block))
    amax = np.max(np.abs(xb), axis=-1)
    s = e8m0_scale_exponent(amax)
    scaled = np.ldexp(xb, -s[..., None])
    q = e4m3_encode(scaled).reshape(xp.shape)[..., :K]
    return np.ascontiguousarray(q), (s + E8M0_BIAS).astype(np.uint8)


def mxfp4_quantize(x: np.ndarray, block: int = BLOCK):
    """MXFP4 (e2m1 elements) quantization along the last axis; K % 32 == 0.

    Per block: amax = max|x|; s = e8m0_scale_exponent(amax, emax=2); scale
    byte s + 127; each element q = e2m1_encode(x * 2^-s).  Returns (packed
    uint8 [..., K/2] (pack_fp4), scale uint8 [..., K/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("mxfp4_quantize: non-finite input is outside the contract")
    K = x.shape[-1]
    if K % block:
        raise ValueError("mxfp4_quantize: K must be a multiple of the block")
    xb = x.reshape(x.shape[:-1] + (K // block, block))
    s = e8m0_scale_exponent(np.max(np.abs(xb), axis=-1), emax=E2M1_EMAX)
    codes = e2m1_encode(np.ldexp(xb, -s[..., None])).reshape(x.shape)
    return pack_fp4(codes), (s + E8M0_BIAS).astype(np.uint8)


def mxfp4_dequantize(packed: np.ndarray, scale: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """Inverse of mxfp4_quantize: dec(q) * 2^(scale - 127), float64 [..., K]."""
    codes = unpack_fp4(packed)
    s = np.asarray(scale, dtype=np.int64) - E8M0_BIAS
    return np.ldexp(e2m1_decode(codes), np.repeat(s, block, axis=-1)[..., :codes.shape[-1]])


def mx_dequantize(q: np.ndarray, scale: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """Inverse of ``mx_quantize``: dec(q) * 2^(scale - 127), float64."""
    q = np.asarray(q, dtype=np.uint8)
    K = q.shape[-1]
    s = np.asarray(scale, dtype=np.int64) - E8M0_BIAS
    s_full = np.repeat(s, block, axis=-1)[..., :K]
    return np.ldexp(e4m3_decode(q), s_full)


# ----------------------------------------------------------------------------
# pair-split scale layout
# ----------------------------------------------------------------------------

def pair_split_scales(scale: np.ndarray) -> np.ndarray:
    """Flat [..., ceil(K/32)] scales -> pair-split [..., ceil(K/64), 2].

    Consecutive scales are paired (contiguous pairing: the reshape is a view
    of the same bytes when the count is even).  An odd count gets one zero
    byte as the synthetic partner of the final partial block (PR #32266
    summary: K=4304 has 135 scales -> 136 -> 68 pairs; the padding "does not
    replace or alter any checkpoint scale").
    """
    scale = np.asarray(scale, dtype=np.uint8)
    n = scale.shape[-1]
    if n % 2:
        scale = np.concatenate([scale, np.zeros(scale.shape[:-1] + (1,), np.uint8)], axis=-1)
    return scale.reshape(scale.shape[:-1] + (scale.shape[-1] // 2, 2))


def n_scales(K: int, block: int = BLOCK) -> int:
    """Number of block scales along K: ceil(K / 32)."""
    return math.ceil(K / block)
