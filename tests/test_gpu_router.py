"""GPU parity of the router gate GEMM fused with softmax top-k.

Through the C ABI, against the CPU oracle and against the logits-input
routing kernel:

* exactness: integer-valued bf16 hidden states and gate make every logit an
  exact integer in fp32, so the device logits equal the oracle's exactly, and
  the many ties exercise the tie rule (lower expert id first);
* the config shapes: device logits within the fp32 accumulation bound of the
  oracle's exact fp64 logits; the top-k decision taken on the device's own
  logits equals the oracle's top-k on those logits (ids exact, weights within
  the routing tolerance) and the logits-input routing kernel's bytes;
* the layer from hidden states + gate equals the logits-input layer fed the
  device logits, byte for byte;
* the load-time dequant of an offline MXFP8 gate bit-exact against the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import TOPK_W_RTOL, bits16, to_bf16_tensor, u8

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


def _check_topk_against(mm, x, gate, k, renorm, r, logits):
    """ids / weights: equal to the oracle's top-k on the device logits and
    byte-identical to the logits-input routing kernel on the same logits."""
    ids, w = moe.route_topk(logits.cpu().numpy(), k, renorm)
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ids)
    wd = r["topk_w"].cpu().numpy().astype(np.float64)
    # relative tolerance of the fp32 softmax; a weight below fp32's normal range
    # (e^-100 against the top logit) keeps only its absolute size
    assert np.all(np.abs(wd - w) <= TOPK_W_RTOL * np.abs(w) + 2.0 ** -125)
    rr = mm.moe_route_quant_mxfp8(x, logits, k, renorm)
    assert torch.equal(rr["topk_ids"], r["topk_ids"])
    assert torch.equal(rr["topk_w"].view(torch.int32), r["topk_w"].view(torch.int32))


@pytest.mark.parametrize("T,H,E,k", [(1, 64, 16, 1), (200, 256, 128, 8), (1000, 2048, 128, 8),
                                     (333, 512, 256, 16), (64, 128, 48, 5), (77, 192, 8, 2),
                                     (130, 64, 6, 6), (257, 128, 64, 32)])
@pytest.mark.parametrize("renorm", [True, False])
def test_router_exact_integer_inputs(mm, T, H, E, k, renorm):
    rng = np.random.default_rng(T + H + E + k)
    xi = rng.integers(-8, 9, (T, H)).astype(np.float64)
    gi = rng.integers(-4, 5, (E, H)).astype(np.float64)
    xb, gb = mx.f64_to_bf16_bits(xi), mx.f64_to_bf16_bits(gi)
    x, gate = to_bf16_tensor(xb, DEV), to_bf16_tensor(gb, DEV)
    r = mm.moe_router_gate_topk(x, gate, k, renorm, logits=True)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    ref = moe.router_logits(xb, gb)
    assert np.array_equal(r["logits"].cpu().numpy().astype(np.float64), ref)
    _check_topk_against(mm, x, gate, k, renorm, r, r["logits"])


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode", "qwen3_30b_prefill"])
def test_router_configs(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    x = workloads.make_hidden(shape, DEV)
    gate = workloads.make_gate(shape, DEV)
    r = mm.moe_router_gate_topk(x, gate, shape.k, True, logits=True)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    rows = np.arange(shape.T) if shape.T <= 2048 else np.random.default_rng(1).choice(
        shape.T, 512, replace=False)
    ri = torch.from_numpy(rows).to(DEV)
    xb, gb = bits16(x[ri]), bits16(gate)
    ref = moe.router_logits(xb, gb)
    # fp32 accumulation of exact bf16 products: |error| <= H * 2^-24 * sum |x g|
    bound = shape.H * 2.0 ** -24 * (np.abs(mx.bf16_bits_to_f64(xb)) @
                                     np.abs(mx.bf16_bits_to_f64(gb)).T)
    dl = r["logits"][ri].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(dl - ref) <= bound)
    _check_topk_against(mm, x, gate, shape.k, True, r, r["logits"])


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode", "qwen3_30b_prefill"])
def test_gated_layer_equals_logits_layer(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV)
    gate = workloads.make_gate(shape, DEV)
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    logits = mm.moe_router_gate_topk(inp["x"], gate, shape.k, logits=True)["logits"]
    out_g = layer.forward_gated(inp["x"], gate)
    out_l = layer(inp["x"], logits)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out_g, out_l), int((out_g != out_l).sum().item())


def test_offline_gate_dequant_bit_exact(mm):
    rng = np.random.default_rng(3)
    E, H = 128, 2048
    codes = rng.integers(0, 256, (E, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x44          # NaN codes are outside the contract
    s = rng.integers(90, 150, (E, H // 32)).astype(np.uint8)
    s[0, 0], s[1, 1] = 0, 254                     # extreme scales: subnormal results, and
    codes[1, 32:64] = rng.choice(np.array([0x00, 0x30, 0x38, 0x3F, 0xB8, 0xBF], np.uint8), 32)
    # |values| < 2 in the 2^127 block, so every product is a finite bf16
    got = mm.mx_dequantize_bf16_2d(torch.from_numpy(codes).to(DEV), torch.from_numpy(s).to(DEV))
    torch.cuda.synchronize()
    ref = moe.dequantize_gate(codes, s)
    fin = np.isfinite(mx.bf16_bits_to_f64(ref))
    assert np.array_equal(bits16(got)[fin], ref[fin])


def test_offline_gate_layer(mm):
    """An MXFP8 gate (quantized at export) is dequantized with its block scale
    and then routes exactly like a bf16 gate holding those values."""
    shape = workloads.CONFIGS["tiny"]
    inp = workloads.make_layer(shape, DEV)
    gq, gs = mm.mx_quantize_3d(workloads.make_gate(shape, DEV))
    gate = mm.mx_dequantize_bf16_2d(gq, gs)
    torch.cuda.synchronize()
    assert np.array_equal(bits16(gate), moe.dequantize_gate(u8(gq), u8(gs)))
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    logits = mm.moe_router_gate_topk(inp["x"], gate, shape.k, logits=True)["logits"]
    assert torch.equal(layer.forward_gated(inp["x"], gate), layer(inp["x"], logits))


def test_router_argument_errors(mm):
    from mxfp8_block_scaled_moe_gb300._lib import MXMoEError
    x = torch.zeros(8, 128, dtype=torch.bfloat16, device=DEV)
    for E, k, H in ((128, 33, 128), (272, 2, 128), (128, 2, 96)):
        g = torch.zeros(E, H, dtype=torch.bfloat16, device=DEV)
        with pytest.raises(MXMoEError) as ei:
            mm.moe_router_gate_topk(x[:, :H].contiguous(), g, k)
        assert ei.value.code == 4
    assert mm.moe_router_gate_topk(x[:0], torch.zeros(16, 128, dtype=torch.bfloat16,
                                                        device=DEV), 2)["topk_ids"].shape == (0, 2)
