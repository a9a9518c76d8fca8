"""GPU parity of the W4A4 path (MXFP4 weights and MXFP4 GEMM inputs).

Through the C ABI, against the CPU oracle on the same seeded bytes:

* the W4A4 dense linear: exactness pins (activations that MXFP4-quantize
  losslessly, e2m1 weights with scales 2^[-2, 2], every partial sum exact in
  fp32) bit-exact through the 1-SM and 2-SM kernels, with ragged K slices and
  ragged N; sampled outputs of the dense shapes within the bf16 bound;
* the W4A4 MoE layer against the oracle's W4A4 layer: the whole output for
  the small shapes, and at the prefill sizes the outputs of sampled tokens
  (a token's output depends only on its own row, its routing and its
  experts' weights, so the oracle runs on the sampled tokens alone);
* argument errors and the two linear entry points giving the same bytes.
"""

import numpy as np
import pytest
import torch

from oracle import linear, moe, mx
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


GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])


def _lossless_fp4_rows(rng, rows, K, spread=1):
    """Rows that MXFP4-quantize exactly: per block one element +-4 * 2^s (it
    fixes the scale at 2^s), e2m1 grid values * 2^s elsewhere."""
    x = GRID[rng.integers(0, 8, (rows, K))] * np.where(rng.random((rows, K)) < 0.5, -1.0, 1.0)
    nb = K // 32
    s = rng.integers(-spread, spread + 1, (rows, nb))
    pos = rng.integers(0, 32, (rows, nb))
    sign = np.where(rng.random((rows, nb)) < 0.5, -1.0, 1.0)
    for j in range(nb):
        x[np.arange(rows), 32 * j + pos[:, j]] = 4.0 * sign[:, j]
    return x * np.exp2(np.repeat(s, 32, axis=1))


def _fp4_weights(rng, N, K):
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    s = (127 + rng.integers(-2, 3, (N, K // 32))).astype(np.uint8)
    return mx.pack_fp4(codes), s


# the W4A4 linear takes K % 128 == 0; K % 256 == 128 leaves a packed k-slice
# with one scale chunk (two of its four K = 64 MMAs)
EXACT_SHAPES = [
    (200, 400, 384),     # N = 3 row blocks + 16 (128-wide tiles, ragged)
    (1, 16, 128),        # one row, one sector, one K slice
    (129, 4304, 1152),   # N = 4304: 34 row blocks (256-wide tiles), the last ragged
    (300, 1152, 4352),   # 34 K slices, N = 9 row blocks (128-wide tiles)
    (640, 512, 2048),    # enough rows for the 2-SM kernel
]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("M,N,K", EXACT_SHAPES)
def test_w4a4_linear_exact_structured(mm, M, N, K, mode):
    rng = np.random.default_rng(M + N + K + 7)
    x = _lossless_fp4_rows(rng, M, K)
    wp, ws = _fp4_weights(rng, N, K)
    w = mx.mxfp4_dequantize(wp, ws)
    # every product is a multiple of 2^-5 and the sum of |products| stays
    # below 2^24 of those units: any fp32 summation order is exact
    assert (np.abs(x) @ np.abs(w).T).max() * 32 < 2 ** 24
    xb = mx.f64_to_bf16_bits(x)
    assert np.array_equal(mx.bf16_bits_to_f64(xb), x)
    mm.set_gemm_2sm(mode)
    try:
        y = mm.mxfp4_linear(to_bf16_tensor(xb, DEV), _t(wp), _t(ws))
        torch.cuda.synchronize()
    finally:
        mm.set_gemm_2sm("auto")
    assert mm.device_status() == 0
    ref = linear.mxfp4_linear(xb, wp, ws)
    got = bits16(y)
    mism = np.argwhere(got != ref)
    assert mism.shape[0] == 0, f"{mism.shape[0]} mismatches, first at {mism[:5].tolist()}"


@pytest.mark.parametrize("cfg", ["qwen3vl_vision_fc1", "qwen3_8b_down_prefill",
                                 "qwen3_8b_gate_up_prefill", "qwen3_8b_down_decode"])
def test_w4a4_linear_configs_sampled(mm, cfg):
    shape = workloads.LINEAR_CONFIGS[cfg]
    x, w = workloads.make_linear(shape, DEV)
    lin = mm.MXFP4Linear.from_bf16(w)
    y = lin(x)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    rng = np.random.default_rng(shape.seed + 1)
    rows = np.unique(np.concatenate([[0, shape.M - 1], rng.integers(0, shape.M, 48)]))
    cols = np.unique(np.concatenate([[0, shape.N - 1], rng.integers(0, shape.N, 256)]))
    wp, ws = mx.mxfp4_quantize(mx.bf16_bits_to_f64(bits16(w[torch.from_numpy(cols).to(DEV)])))
    assert np.array_equal(u8(lin.wp[torch.from_numpy(cols).to(DEV)]), wp)
    ref = linear.mxfp4_linear(bits16(x[torch.from_numpy(rows).to(DEV)]), wp, ws)
    assert rel_frob(bits16(y)[np.ix_(rows, cols)], ref) <= OUT_REL_FROB


def test_w4a4_linear_entry_points_agree_and_errors(mm):
    from mxfp8_block_scaled_moe_gb300._lib import MXMoEError
    shape = workloads.LINEAR_CONFIGS["linear_tiny"]
    x, w = workloads.make_linear(shape, DEV)
    x, w = x[:, :256].contiguous(), w[:, :256].contiguous()
    wp, ws = mm.mx_quantize_fp4_3d(w)
    a = mm.mxfp4_linear(x, wp, ws)
    b = mm.mxfp4_linear_mma_scales(x, wp, mm.mx_scales_to_mma_layout(ws, 256))
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for kk in (192, 240):                   # K % 128 != 0
        with pytest.raises(MXMoEError) as ei:
            mm.mxfp4_linear(x[:, :kk].contiguous(), wp[:, :kk // 2].contiguous(), ws)
        assert ei.value.code == 3
    buf = torch.empty(wp.numel() + 64, dtype=torch.uint8, device=DEV)
    base = (-buf.data_ptr()) % 32 + 16
    wp16 = buf[base:base + wp.numel()].view(wp.shape)
    wp16.copy_(wp)
    with pytest.raises(MXMoEError) as ei:   # packed weights only 16-byte aligned
        mm.mxfp4_linear(x, wp16, ws)
    assert ei.value.code == 2
    torch.cuda.synchronize()
    assert mm.device_status() == 0


def _oracle_layer(mm, layer, x, logits, k, I):
    return moe.moe_forward(bits16(x), logits.cpu().numpy(), u8(layer.w13p), u8(layer.w13s),
                           u8(layer.w2p), u8(layer.w2s), k, I, wfmt="e2m1", afmt="e2m1")


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode"])
def test_w4a4_layer_matches_oracle(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.W4A4MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    out = layer(inp["x"], inp["logits"])
    out2 = layer(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out, out2)
    ref = _oracle_layer(mm, layer, inp["x"], inp["logits"], shape.k, shape.I)
    assert rel_frob(bits16(out), ref["out"]) <= OUT_REL_FROB


@pytest.mark.parametrize("cfg", ["qwen3_30b_prefill", "qwen3_30b_skewed"])
def test_w4a4_layer_prefill_sampled_tokens(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.W4A4MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    del inp["w13"], inp["w2"]
    out = layer(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    rng = np.random.default_rng(shape.seed + 2)
    tok = np.unique(np.concatenate([[0, shape.T - 1], rng.integers(0, shape.T, 22)]))
    ti = torch.from_numpy(tok).to(DEV)
    ref = _oracle_layer(mm, layer, inp["x"][ti], inp["logits"][ti], shape.k, shape.I)
    assert rel_frob(bits16(out[ti]), ref["out"]) <= OUT_REL_FROB
