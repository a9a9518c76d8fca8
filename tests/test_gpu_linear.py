"""GPU parity of the dense MXFP8 linear (partial K blocks, ragged N).

Everything runs through the C ABI and is compared with the CPU oracle on the
same seeded bytes:

* the row quantizer for K % 32 == 16 (a partial last block of 16) and any
  K % 16 == 0: codes and scales bit-exact;
* the MMA-layout re-layout of weight scales for a ragged K slice and a ragged
  last row block: every byte against the layout's definition (pad = 127);
* exactness pins: lossless activations and integer-valued weights with
  scales in [2^-2, 2^2] keep every partial sum exact in fp32, so the output
  must equal the oracle bit for bit -- through 1-SM and 2-SM kernels, partial
  K and ragged N;
* the pages' shapes (Qwen3-VL vision MLP with K or N = 4304, Qwen3-8B
  projections): sampled outputs against the oracle within the bf16 bound;
* edge cases: M = 0, one row, argument errors, both entry points giving the
  same bytes, determinism.
"""

import math

import numpy as np
import pytest
import torch

from oracle import linear, mx
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import OUT_REL_FROB, bits16, rel_frob, to_bf16_tensor, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def mm():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_moe_gb300 as m
    return m


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("N,K", [(1, 16), (5, 48), (37, 336), (64, 4304), (3, 1040), (130, 208)])
def test_row_quant_partial_block_bit_exact(mm, N, K):
    rng = np.random.default_rng(N * 7 + K)
    x = rng.standard_t(4, (N, K)) * np.exp2(rng.integers(-30, 30, (N, 1)))
    x[0, -16:] = 0.0                       # an all-zero partial block
    if N > 1:
        x[1, -16:] *= 2.0 ** -120          # a subnormal-amax partial block
    xb = mx.f64_to_bf16_bits(x)
    q, s = mm.mx_quantize_3d(to_bf16_tensor(xb, DEV))
    torch.cuda.synchronize()
    qr, sr = mx.mx_quantize(mx.bf16_bits_to_f64(xb))
    assert s.shape == (N, math.ceil(K / 32))
    assert np.array_equal(u8(s), sr)
    assert np.array_equal(u8(q), qr)


def _tiled_expected(s, E, N, K):
    """The MMA layout by its definition: chunk (row block, K slice) of 512
    bytes, byte (r % 32) * 16 + (r / 32) * 4 + kb; 127 past the data."""
    KT, K32 = -(-K // 128), -(-K // 32)
    rows = -(-N // 128) * 128
    out = np.full((E, rows, KT * 4), 127, np.uint8)
    out[:, :N, :K32] = s
    flat = np.empty(E * rows * KT * 4, np.uint8)
    for e in range(E):
        for row in range(rows):
            rb, r = (e * rows + row) // 128, row % 128
            for j in range(KT * 4):
                flat[(rb * KT + j // 4) * 512 + (r % 32) * 16 + (r // 32) * 4 + j % 4] = out[e, row, j]
    return flat


@pytest.mark.parametrize("E,N,K", [(1, 200, 336), (1, 16, 48), (2, 256, 208), (1, 4304, 1152),
                                   (1, 1152, 4304)])
def test_scales_to_mma_layout_ragged(mm, E, N, K):
    rng = np.random.default_rng(E + N + K)
    s = rng.integers(100, 140, (E, N, -(-K // 32))).astype(np.uint8)
    out = mm.mx_scales_to_mma_layout(_t(s if E > 1 else s[0]), K)
    torch.cuda.synchronize()
    assert np.array_equal(u8(out).reshape(-1), _tiled_expected(s, E, N, K))


def _lossless_rows(rng, rows, K, lo=-8, hi=8, spread=1):
    """Rows that MX-quantize exactly: per block one element +-256 * 2^s (it
    fixes the scale at 2^s) and integers in [lo, hi] * 2^s elsewhere."""
    x = rng.integers(lo, hi + 1, (rows, K)).astype(np.float64)
    nb = -(-K // 32)
    s = rng.integers(-spread, spread + 1, (rows, nb))
    pos = rng.integers(0, 16, (rows, nb))
    sign = np.where(rng.random((rows, nb)) < 0.5, -1.0, 1.0)
    for j in range(nb):
        x[np.arange(rows), 32 * j + pos[:, j]] = 256.0 * sign[:, j]
    return x * np.exp2(np.repeat(s, 32, axis=1)[:, :K])


def _int_weights(rng, N, K):
    """Integer codes in [-2, 2] with scales 2^[-2, 2].  With the rows above
    every product is a multiple of 2^-3 and the sum of |products| over
    K = 4304 stays below 2^21, so any fp32 summation order is exact."""
    q = mx.e4m3_encode(rng.integers(-2, 3, (N, K)).astype(np.float64))
    s = (127 + rng.integers(-2, 3, (N, -(-K // 32)))).astype(np.uint8)
    return q, s


EXACT_SHAPES = [
    (200, 400, 336),     # tiny: ragged K slice, N = 3 row blocks + 16 (BN 128, ragged)
    (1, 16, 16),         # one row, one column sector, one partial block
    (129, 4304, 1152),   # N = 4304: 34 row blocks (BN 256), last one ragged
    (300, 1152, 4304),   # K = 4304: 135 scales, ragged last K slice
    (257, 272, 208),     # N = 272: odd row blocks (BN 128), 16-column tail
    (640, 512, 4304),    # enough rows for the 2-SM kernel
    (32, 4096, 1152),    # decode-sized M: split-K over 2 K ranges
    (20, 512, 4304),     # split-K over 7 K ranges, ragged last K slice
    (31, 8192, 256),     # 32 tiles of one partial m-tile, no split
]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("M,N,K", EXACT_SHAPES)
def test_linear_exact_structured(mm, M, N, K, mode):
    rng = np.random.default_rng(M + N + K)
    x = _lossless_rows(rng, M, K)
    wq, ws = _int_weights(rng, N, K)
    xb = mx.f64_to_bf16_bits(x)
    assert np.array_equal(mx.bf16_bits_to_f64(xb), x)
    mm.set_gemm_2sm(mode)
    try:
        y = mm.mxfp8_linear(to_bf16_tensor(xb, DEV), _t(wq), _t(ws))
        torch.cuda.synchronize()
    finally:
        mm.set_gemm_2sm("auto")
    assert mm.device_status() == 0
    ref = linear.mxfp8_linear(xb, wq, ws)
    got = bits16(y)
    mism = np.argwhere(got != ref)
    assert mism.shape[0] == 0, f"{mism.shape[0]} mismatches, first at {mism[:5].tolist()}"


def _sampled_check(mm, shape, n_rows=48, n_cols=256, layer=None):
    x, w = workloads.make_linear(shape, DEV)
    lin = layer or mm.MXFP8Linear.from_bf16(w)
    y = lin(x)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    rng = np.random.default_rng(shape.seed)
    rows = np.unique(np.concatenate([[0, shape.M - 1], rng.integers(0, shape.M, n_rows)]))
    cols = np.unique(np.concatenate([[0, shape.N - 1], rng.integers(0, shape.N, n_cols)]))
    wq, ws = mx.mx_quantize(mx.bf16_bits_to_f64(bits16(w[torch.from_numpy(cols).to(DEV)])))
    ref = linear.mxfp8_linear(bits16(x[torch.from_numpy(rows).to(DEV)]), wq, ws)
    got = bits16(y)[np.ix_(rows, cols)]
    assert rel_frob(got, ref) <= OUT_REL_FROB
    return y


def test_linear_tiny_full_vs_oracle(mm):
    shape = workloads.LINEAR_CONFIGS["linear_tiny"]
    x, w = workloads.make_linear(shape, DEV)
    y = mm.MXFP8Linear.from_bf16(w)(x)
    torch.cuda.synchronize()
    wq, ws = mx.mx_quantize(mx.bf16_bits_to_f64(bits16(w)))
    ref = linear.mxfp8_linear(bits16(x), wq, ws)
    assert rel_frob(bits16(y), ref) <= OUT_REL_FROB


@pytest.mark.parametrize("cfg", ["qwen3vl_vision_fc1", "qwen3vl_vision_fc2",
                                 "qwen3_8b_down_prefill", "qwen3_8b_gate_up_prefill",
                                 "qwen3_8b_down_decode"])
def test_linear_configs_sampled(mm, cfg):
    _sampled_check(mm, workloads.LINEAR_CONFIGS[cfg])


def test_linear_weight_quant_of_config_bit_exact(mm):
    shape = workloads.LINEAR_CONFIGS["qwen3vl_vision_fc2"]
    _, w = workloads.make_linear(shape, DEV)
    q, s = mm.mx_quantize_3d(w)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 511, shape.N - 1], device=DEV)
    qr, sr = mx.mx_quantize(mx.bf16_bits_to_f64(bits16(w[rows])))
    assert s.shape == (shape.N, 135)
    assert np.array_equal(u8(s[rows]), sr) and np.array_equal(u8(q[rows]), qr)


def test_linear_entry_points_agree_and_repeat(mm):
    shape = workloads.LINEAR_CONFIGS["linear_tiny"]
    x, w = workloads.make_linear(shape, DEV)
    wq, ws = mm.mx_quantize_3d(w)
    a = mm.mxfp8_linear(x, wq, ws)
    b = mm.mxfp8_linear_mma_scales(x, wq, mm.mx_scales_to_mma_layout(ws, shape.K))
    c = mm.mxfp8_linear(x, wq, ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_linear_leading_dims_and_empty(mm):
    shape = workloads.LINEAR_CONFIGS["linear_tiny"]
    x, w = workloads.make_linear(shape, DEV)
    lin = mm.MXFP8Linear.from_bf16(w)
    y2 = lin(x)
    y3 = lin(x.view(4, 50, shape.K))
    assert y3.shape == (4, 50, shape.N)
    assert torch.equal(y3.reshape(shape.M, shape.N).view(torch.int16), y2.view(torch.int16))
    y0 = lin(x[:0])
    torch.cuda.synchronize()
    assert y0.shape == (0, shape.N)


def test_linear_argument_errors(mm):
    from mxfp8_block_scaled_moe_gb300._lib import MXMoEError
    shape = workloads.LINEAR_CONFIGS["linear_tiny"]
    x, w = workloads.make_linear(shape, DEV)
    wq, ws = mm.mx_quantize_3d(w)
    with pytest.raises(MXMoEError) as ei:   # K % 16 != 0
        mm.mxfp8_linear(x[:, :328].contiguous(), wq[:, :328].contiguous(), ws)
    assert ei.value.code == 3
    with pytest.raises(MXMoEError) as ei:   # workspace too small
        mm.mxfp8_linear(x, wq, ws, workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert ei.value.code == 5
    buf = torch.empty(shape.M * shape.N + 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(MXMoEError) as ei:   # output not 32-byte aligned
        mm.mxfp8_linear(x, wq, ws, out=buf[8:8 + shape.M * shape.N].view(shape.M, shape.N))
    assert ei.value.code == 2
    torch.cuda.synchronize()
    assert mm.device_status() == 0
