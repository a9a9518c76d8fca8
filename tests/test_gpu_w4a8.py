"""GPU parity of the W4A8 path (MXFP4 e2m1 expert weights x MXFP8 activations)
through the C ABI: the load-time FP4 quantizer bit-exact against the oracle,
the layer against the oracle (small shapes), and, at the prefill size, the
W4A8 layer against the MXFP8 layer fed the same weight values as e4m3 codes
(every e2m1 value is an e4m3 value, so the two layers compute the same
thing)."""

import numpy as np
import pytest
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import OUT_REL_FROB, bits16, rel_frob, u8

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


def to_bf16_tensor(bits, dev):
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(dev)


@pytest.mark.parametrize("E,N,K", [(1, 1, 32), (3, 5, 96), (8, 256, 256), (2, 37, 2048)])
def test_mx_quantize_fp4_bit_exact(mm, E, N, K):
    rng = np.random.default_rng(E * 100 + N + K)
    x = rng.standard_t(4, (E, N, K)) * np.exp2(rng.integers(-30, 30, (E, N, 1)))
    x[0, 0, :4] = [6.0, -5.0, 0.25, -0.2]       # saturation-band tie, ties to even, -0
    if N > 1:
        x[0, 1] = 0.0                             # zero block
    xb = mx.f64_to_bf16_bits(x)
    q, s = mm.mx_quantize_fp4_3d(to_bf16_tensor(xb, DEV))
    torch.cuda.synchronize()
    qr, sr = mx.mxfp4_quantize(mx.bf16_bits_to_f64(xb))
    assert np.array_equal(u8(s), sr)
    assert np.array_equal(u8(q), qr)


def _reencode_e4m3(p):
    """Packed FP4 weights (device) -> the same values as e4m3 codes (device)."""
    lut = torch.from_numpy(mx.e4m3_encode(mx.E2M1_TABLE)).to(p.device)
    codes = torch.stack([p & 0xF, p >> 4], dim=-1).reshape(p.shape[:-1] + (2 * p.shape[-1],))
    return lut[codes.long()]


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode"])
def test_w4a8_layer_matches_oracle(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    layer = mm.W4A8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    out = layer(inp["x"], inp["logits"])
    out2 = layer(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out, out2)
    ref = moe.moe_forward(bits16(inp["x"]), inp["logits"].cpu().numpy(), u8(layer.w13p),
                          u8(layer.w13s), u8(layer.w2p), u8(layer.w2s), shape.k, shape.I,
                          wfmt="e2m1")
    assert rel_frob(bits16(out), ref["out"]) <= OUT_REL_FROB


@pytest.mark.parametrize("cfg", ["qwen3_30b_prefill", "qwen3_30b_skewed"])
def test_w4a8_layer_equals_mxfp8_layer_on_reencoded_weights(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    l4 = mm.W4A8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    l8 = mm.MXFP8MoELayer.from_quantized(_reencode_e4m3(l4.w13p), l4.w13s, _reencode_e4m3(l4.w2p),
                                         l4.w2s, shape.k)
    out4 = l4(inp["x"], inp["logits"])
    out8 = l8(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    # e4m3 x e2m1 and e4m3 x e4m3 products of the same values are the same
    # exact numbers, accumulated by the same tiles in the same order
    assert torch.equal(out4, out8), int((out4 != out8).sum().item())
