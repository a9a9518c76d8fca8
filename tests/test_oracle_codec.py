"""Pins for the oracle's codecs and MX block quantizer (CPU only).

Each check ties the oracle to something other than itself: torch's own
float8_e4m3fn and bfloat16 casts (library routines), brute-force nearest-grid
search, closed forms of the scale rule, the hand-worked golden blocks, and the
error bound the format implies.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_blocks.txt")


# ---------------------------------------------------------------- e4m3 codec

def test_e4m3_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = mx.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], ours[fin])
    # sign of zero: 0x80 is -0
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_e4m3_known_codes():
    assert mx.E4M3_TABLE[0x7E] == 448.0
    assert mx.E4M3_TABLE[0x01] == 2.0 ** -9          # smallest subnormal
    assert mx.E4M3_TABLE[0x08] == 2.0 ** -6          # smallest normal
    assert mx.E4M3_TABLE[0x38] == 1.0
    assert np.isnan(mx.E4M3_TABLE[0x7F]) and np.isnan(mx.E4M3_TABLE[0xFF])


def _all_finite_bf16_in_range(limit):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = mx.bf16_bits_to_f64(bits)
    keep = np.isfinite(v) & (np.abs(v) <= limit)
    return v[keep]


def test_e4m3_encode_matches_torch_on_every_bf16_value_in_range():
    # torch's cast is RNE but does not saturate above 464; compare where both define it
    v = _all_finite_bf16_in_range(448.0)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mx.e4m3_encode(v), ref)


def test_e4m3_encode_midpoints_go_to_even():
    grid = mx.E4M3_TABLE[:0x7F]
    mids = (grid[:-1] + grid[1:]) / 2.0          # exact in fp64 and fp32
    ours = mx.e4m3_encode(mids)
    even = np.where(np.arange(0, 0x7E) % 2 == 0, np.arange(0, 0x7E), np.arange(1, 0x7F))
    assert np.array_equal(ours, even.astype(np.uint8))
    ref = torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    assert np.array_equal(mx.e4m3_encode(-mids), ours | 0x80)


def test_e4m3_encode_brute_force_nearest():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.normal(0, 40, 4000), rng.normal(0, 0.01, 2000),
                        rng.uniform(-448, 448, 2000)])
    grid_codes = np.array([c for c in range(256) if not np.isnan(mx.E4M3_TABLE[c])])
    grid = mx.E4M3_TABLE[grid_codes]
    got = mx.e4m3_encode(v)
    for val, code in zip(v, got):
        d = np.abs(grid - val)
        best = np.flatnonzero(d == d.min())
        cands = grid_codes[best]
        # among equally near codes: the even mantissa, with the input's sign for zero
        if len(cands) > 1:
            cands = cands[(cands & 1) == 0]
        if mx.E4M3_TABLE[cands[0]] == 0.0:
            cands = np.array([0x80 if np.signbit(val) else 0x00])
        assert code == cands[0], (val, code, cands)


def test_e4m3_saturation():
    v = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, -500.0, -1e30])
    assert mx.e4m3_encode(v).tolist() == [0x7E] * 6 + [0xFE, 0xFE]


def test_e4m3_negative_underflow_keeps_sign():
    assert mx.e4m3_encode(np.array([-1e-9, 1e-9, -0.0, 0.0])).tolist() == [0x80, 0x00, 0x80, 0x00]


def test_e4m3_rejects_non_finite():
    with pytest.raises(ValueError):
        mx.e4m3_encode(np.array([np.nan]))


# ---------------------------------------------------------------- bf16 rounding

def test_f64_to_bf16_matches_torch_for_fp32_inputs():
    rng = np.random.default_rng(2)
    v32 = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 5000),
                          rng.normal(0, 1e30, 1000)]).astype(np.float32)
    # add exact ties: bf16 grid points plus half a bf16 ulp
    base = np.array([1.0, 1.0078125, 3.0, -2.5, 1e-20], np.float32)
    ulp = np.array([2 ** -7, 2 ** -7, 2 ** -6, 2 ** -6, 0], np.float32)
    ulp[4] = np.float32(2.0 ** (math.floor(math.log2(1e-20)) - 7))
    ties = (base + ulp / 2).astype(np.float32)
    v32 = np.concatenate([v32, ties])
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mx.f64_to_bf16_bits(v32.astype(np.float64)), ref)


def test_bf16_roundtrip_exact():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = mx.bf16_bits_to_f64(bits)
    fin = np.isfinite(v)
    back = mx.f64_to_bf16_bits(v[fin])
    # -0 and +0 keep their sign; every finite pattern maps back to itself
    assert np.array_equal(back, bits[fin])


# ---------------------------------------------------------------- scale rule

def test_scale_closed_form_powers_of_two():
    for e in range(-133, 128):
        amax = 2.0 ** e
        want = min(max(e - 8, -127), 127)
        assert mx.e8m0_scale_exponent(np.array([amax]))[0] == want
        # anything in [2^e, 2^(e+1)) has the same floor(log2)
        just_below_next = np.nextafter(2.0 ** (e + 1), 0)
        assert mx.e8m0_scale_exponent(np.array([just_below_next]))[0] == want
    assert mx.e8m0_scale_exponent(np.array([0.0]))[0] == -127


def test_scale_puts_block_amax_in_256_512():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (500, 64)) * np.exp2(rng.integers(-60, 60, (500, 1)))
    q, s = mx.mx_quantize(x)
    amax = np.abs(x.reshape(500, 2, 32)).max(-1)
    r = amax / np.exp2(s.astype(np.int64) - 127)
    assert np.all((r >= 256) & (r < 512))


# ---------------------------------------------------------------- golden blocks

def _golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, K, xs, sc, codes = [p.strip() for p in line.split("|")]
            K = int(K)
            x = np.zeros(K)
            vals = [float(v) for v in xs.split(",")]
            x[:len(vals)] = vals
            scales = [int(v) for v in sc.split(",")]
            q = np.zeros(K, np.uint8)
            cl = [int(c, 16) for c in codes.split(",")]
            q[:len(cl)] = cl
            cases.append((name, x, np.array(scales, np.uint8), q))
    return cases


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c[0])
def test_golden_blocks(case):
    name, x, scales, q = case
    gq, gs = mx.mx_quantize(x[None, :])
    assert gs[0].tolist() == scales.tolist(), name
    assert gq[0].tolist() == q.tolist(), name


GOLDEN_FP4 = os.path.join(os.path.dirname(__file__), "golden", "mxfp4_blocks.txt")


def _num(v):
    v = v.strip()
    return float.fromhex(v) if "p" in v.lower() else float(v)


def _golden_fp4():
    cases = []
    with open(GOLDEN_FP4) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, K, xs, sc, packed = [p.strip() for p in line.split("|")]
            K = int(K)
            x = np.zeros(K)
            vals = [_num(v) for v in xs.split(",")]
            x[:len(vals)] = vals
            q = np.zeros(K // 2, np.uint8)
            pl = [int(c, 16) for c in packed.split(",")]
            q[:len(pl)] = pl
            cases.append((name, x, np.array([int(v) for v in sc.split(",")], np.uint8), q))
    return cases


@pytest.mark.parametrize("case", _golden_fp4(), ids=lambda c: c[0])
def test_golden_mxfp4_blocks(case):
    """Hand-worked MXFP4 blocks: scale rule, ties to even, saturation, the
    e8m0 clamps and the nibble order of the packed bytes."""
    name, x, scales, q = case
    assert np.array_equal(mx.bf16_bits_to_f64(mx.f64_to_bf16_bits(x)), x), name  # bf16 inputs
    gq, gs = mx.mxfp4_quantize(x[None, :])
    assert gs[0].tolist() == scales.tolist(), name
    assert gq[0].tolist() == q.tolist(), name


# ---------------------------------------------------------------- dequant error

def test_dequant_error_bound():
    rng = np.random.default_rng(4)
    x = rng.standard_t(3, (400, 256)) * np.exp2(rng.integers(-20, 20, (400, 1)))
    x = mx.bf16_bits_to_f64(mx.f64_to_bf16_bits(x))   # bf16-exact inputs, like the path
    q, s = mx.mx_quantize(x)
    d = mx.mx_dequantize(q, s)
    scale = np.exp2(np.repeat(s.astype(np.int64) - 127, 32, axis=-1))
    r = np.abs(x) / scale
    err = np.abs(x - d) / scale
    inside = r <= 448
    assert np.all(err[inside] <= 0.5 * mx.e4m3_ulp(r[inside]) + 0.0)
    # saturation band (448, 512): error below 64 scale units
    assert np.all(err[~inside] < 64)


def test_exact_roundtrip_of_representable_blocks():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, (300, 32)).astype(np.uint8)
    codes[codes == 0x7F] = 0x7E
    codes[:, 0] = rng.integers(0x78, 0x7F, 300)             # block max in [256, 448]
    codes |= (rng.integers(0, 2, (300, 32)) << 7).astype(np.uint8)
    s = rng.integers(-100, 100, 300)
    x = np.ldexp(mx.e4m3_decode(codes), s[:, None])
    q, sc = mx.mx_quantize(x)
    assert np.array_equal(sc.reshape(-1).astype(np.int64), s + 127)
    # -0 inputs come back as 0x80, so compare values and the sign bit of zeros
    assert np.array_equal(q, codes)


# ---------------------------------------------------------------- pair-split layout

def test_pair_split_is_a_view_for_even_counts():
    rng = np.random.default_rng(6)
    s = rng.integers(0, 255, (3, 5, 64)).astype(np.uint8)      # K = 2048 -> 64 scales
    p = mx.pair_split_scales(s)
    assert p.shape == (3, 5, 32, 2)
    assert p.tobytes() == s.tobytes()
    assert np.array_equal(p[..., 7, 1], s[..., 15])


def test_pair_split_padding_k4304():
    # the pages' worked example: K=4304 -> 135 scales -> padded to 136 -> 68 pairs
    K = 4304
    assert mx.n_scales(K) == 135
    s = np.arange(135, dtype=np.uint8)[None, :]
    p = mx.pair_split_scales(s)
    assert p.shape == (1, 68, 2)
    assert p[0, 67, 0] == 134 and p[0, 67, 1] == 0
    assert p.reshape(1, -1)[0, :135].tolist() == list(range(135))
    assert math.ceil(K / 64) == 68


# ---------------------------------------------------------------- e2m1 (FP4) codec, W4A8 weights

def test_e2m1_value_set():
    """The 16 e2m1 codes decode to the FP4 value set {0, 0.5, 1, 1.5, 2, 3, 4, 6}
    and its negatives (codes 8..15 = sign bit set)."""
    vals = mx.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert list(vals[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(vals[8:], -vals[:8])
    assert np.signbit(vals[8]) and not np.signbit(vals[0])
    assert mx.E2M1_MAX == vals.max()


def test_e2m1_values_are_exact_e4m3_values_per_torch():
    """Every FP4 value is exactly representable in e4m3 (torch's cast is exact)."""
    v = torch.tensor(mx.E2M1_TABLE, dtype=torch.float32)
    back = v.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(back, mx.E2M1_TABLE)


def test_e2m1_encode_brute_force_nearest_even():
    grid = mx.e2m1_decode(np.arange(8, dtype=np.uint8))
    rng = np.random.default_rng(3)
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([rng.uniform(-9, 9, 20000), mids, -mids, grid, -grid,
                        np.nextafter(mids, 0), np.nextafter(mids, 10), [6.5, 7.9, 100.0, -1e9]])
    codes = mx.e2m1_encode(v)
    a = np.minimum(np.abs(v), 6.0)
    d = np.abs(a[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # ties (two candidates) go to the even code (mantissa bit 0)
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    ref = np.where(cand.sum(1) > 1, np.argmax(even, 1), np.argmax(cand, 1))
    assert np.array_equal(codes & 7, ref)
    assert np.array_equal(codes >> 3, np.signbit(v).astype(np.uint8))
    assert mx.e2m1_encode(np.array([5.0]))[0] == 6      # 5 = midpoint of 4 and 6 -> 4 (even)
    assert mx.e2m1_encode(np.array([-0.2]))[0] == 8     # rounds to zero, sign kept


def test_pack_fp4_nibble_order_and_roundtrip():
    assert mx.pack_fp4(np.array([1, 2], np.uint8))[0] == 0x21   # element 0 in the low nibble
    rng = np.random.default_rng(4)
    c = rng.integers(0, 16, (5, 64), dtype=np.uint8)
    assert np.array_equal(mx.unpack_fp4(mx.pack_fp4(c)), c)


def test_mxfp4_scale_closed_form_and_range():
    for e in range(-120, 120, 7):
        _, s = mx.mxfp4_quantize(np.full((1, 32), 2.0 ** e))
        assert int(s[0, 0]) - 127 == e - 2
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 32)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    _, s = mx.mxfp4_quantize(x)
    r = np.max(np.abs(x), axis=1) / np.exp2(s[:, 0].astype(np.int64) - 127)
    assert np.all((r >= 4) & (r < 8))
    _, s0 = mx.mxfp4_quantize(np.zeros((1, 32)))
    assert s0[0, 0] == 0


def test_mxfp4_dequant_error_bound_and_representable_roundtrip():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((256, 64))
    q, s = mx.mxfp4_quantize(x)
    d = mx.mxfp4_dequantize(q, s)
    sc = np.repeat(np.exp2(s.astype(np.int64) - 127), 32, axis=1)
    a = np.abs(x) / sc
    ulp = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    inside = a <= 6
    assert np.all(np.abs(d - x)[inside] <= (ulp * sc)[inside] / 2)
    assert np.all(np.abs(d - x)[~inside] < (2 * sc)[~inside])
    # blocks whose values are FP4 grid points times 2^s (amax in [4, 8)) come back exactly
    g = mx.e2m1_decode(rng.integers(0, 16, (16, 32), dtype=np.uint8))
    g[:, 0] = 6.0
    blk = g * np.exp2(rng.integers(-30, 30, (16, 1)))
    q2, s2 = mx.mxfp4_quantize(blk)
    assert np.array_equal(mx.mxfp4_dequantize(q2, s2), blk)


def test_mxfp4_gemm_equals_mxfp8_gemm_on_reencoded_weights():
    """W4A8 GEMM oracle == the pinned MXFP8 GEMM oracle fed the same weights
    re-encoded as e4m3 codes under the same scales (FP4 values are exact e4m3)."""
    from oracle import moe
    rng = np.random.default_rng(7)
    E, N, K, M = 3, 96, 128, 40
    w = rng.standard_normal((E, N, K)) * 0.02
    q4, s4 = mx.mxfp4_quantize(w)
    q8 = mx.e4m3_encode(mx.e2m1_decode(mx.unpack_fp4(q4)))
    assert np.array_equal(mx.mx_dequantize(q8, s4), mx.mxfp4_dequantize(q4, s4))
    aq, as_ = mx.mx_quantize(rng.standard_normal((M, K)))
    offs = np.array([0, 10, 10, M])
    y4 = moe.gmm2(aq, as_, q4, s4, offs, wfmt="e2m1")
    y8 = moe.gmm2(aq, as_, q8, s4, offs)
    assert np.array_equal(y4, y8)
