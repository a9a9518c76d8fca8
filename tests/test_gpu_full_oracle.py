"""Full-size parity of the MXFP8 layer against the oracle, every expert.

At the prefill sizes the layer runs as the benchmark runs it (the
``MXFP8MoELayer`` call: MMA-layout scales, the default 1-SM / 2-SM kernel
choice), and the same bytes must come out of the four per-step entry points
in a row; the per-step outputs are then compared with the oracle on every
row of every expert:

* routing and the fused activation quant: bit-exact;
* gmm1 (SwiGLU + requant) from the device's own xq / xs: the requant
  tolerance over all M rows;
* gmm2 from the device's own aq / as: relative Frobenius over all rows, and
  per expert;
* finalize from the device's own y: relative Frobenius and the element-wise
  bound.

The 16K-token 30B prefill also runs the whole oracle layer
(``moe.moe_forward``) end to end against the layer output, and the skewed
routing (Zipf(1.2) popularity, four empty experts) runs the whole oracle
layer at every T of its sweep below 16K tokens.
"""

import numpy as np
import pytest
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads

import _oracle_pool
from _util import (OUT_REL_FROB, REQUANT_MAX_FRAC, TOPK_W_RTOL, bits16, finalize_bound_ok,
                   rel_frob, requant_mismatch, u8)

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


def _layer(mm, shape, inp):
    if shape.offline:
        return mm.MXFP8MoELayer.from_quantized(inp["w13q"], inp["w13s"], inp["w2q"], inp["w2s"],
                                               shape.k)
    return mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)


def _run_both(mm, shape):
    """The benchmark's layer call and the four per-step entry points."""
    inp = workloads.make_layer(shape, DEV)
    layer = _layer(mm, shape, inp)
    for key in ("w13", "w2", "w13q", "w13s", "w2q", "w2s"):
        inp.pop(key, None)
    out = layer(inp["x"], inp["logits"])
    r = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(r["xq"], r["xs"], layer.w13q, layer.w13s,
                                                 r["expert_offsets"])
    y = mm.grouped_gemm_mxfp8(aq, as_, layer.w2q, layer.w2s, r["expert_offsets"])
    out_chain = mm.moe_finalize_routing(y, r["topk_w"], r["src_to_sorted"], shape.k)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out, out_chain)
    return inp, layer, r, aq, as_, y, out


def _check_route(r, xb, logits, k, E):
    ids, w = moe.route_topk(logits, k, True)
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ids)
    wg = r["topk_w"].cpu().numpy().astype(np.float64)
    assert np.max(np.abs(wg - w) / np.abs(w)) <= TOPK_W_RTOL
    xq, xs, counts, offsets, s2s, src2s = moe.route_quant(mx.bf16_bits_to_f64(xb), ids, E)
    assert np.array_equal(r["expert_counts"].cpu().numpy(), counts)
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["sorted_to_src"].cpu().numpy(), s2s)
    assert np.array_equal(r["src_to_sorted"].cpu().numpy(), src2s)
    assert np.array_equal(u8(r["xs"]), xs)
    assert np.array_equal(u8(r["xq"]), xq)
    return offsets


def _check_gmm2_and_finalize(shape, layer, r, aq_g, as_g, y, out, offs):
    y_g = bits16(y)
    y_ref = _oracle_pool.gmm2_all_experts(aq_g, as_g, u8(layer.w2q), u8(layer.w2s), offs)
    assert rel_frob(y_g, y_ref) <= OUT_REL_FROB
    for e in range(shape.E):
        r0, r1 = offs[e], offs[e + 1]
        if r1 > r0:
            assert rel_frob(y_g[r0:r1], y_ref[r0:r1]) <= OUT_REL_FROB, e
    w_g = r["topk_w"].cpu().numpy()
    s2s = r["src_to_sorted"].cpu().numpy()
    assert rel_frob(bits16(out), moe.finalize(y_g, w_g, s2s, shape.k)) <= OUT_REL_FROB
    assert finalize_bound_ok(bits16(out), y_g, w_g, s2s, shape.k) == 0.0


@pytest.mark.parametrize("cfg", ["qwen3_235b_prefill", "qwen3_30b_skewed"])
def test_prefill_every_expert_stagewise(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp, layer, r, aq, as_, y, out = _run_both(mm, shape)
    offs = _check_route(r, bits16(inp["x"]), inp["logits"].cpu().numpy(), shape.k, shape.E)
    if shape.zipf_s > 0:
        cnt = np.diff(offs)
        assert (cnt == 0).sum() >= shape.n_empty and cnt.max() > 0.10 * shape.M
    aq_g, as_g = u8(aq), u8(as_)
    aq_ref, as_ref = _oracle_pool.gmm1_all_experts(u8(r["xq"]), u8(r["xs"]), u8(layer.w13q),
                                                   u8(layer.w13s), offs, shape.I)
    frac, dist = requant_mismatch(aq_g, as_g, aq_ref, as_ref)
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0, (frac, dist)
    _check_gmm2_and_finalize(shape, layer, r, aq_g, as_g, y, out, offs)


def test_prefill_30b_whole_oracle_layer(mm):
    """The 16K-token Qwen3-30B-A3B-shaped prefill: the oracle's whole layer
    end to end against the layer output, and every stage on every expert."""
    shape = workloads.CONFIGS["qwen3_30b_prefill"]
    inp, layer, r, aq, as_, y, out = _run_both(mm, shape)
    xb = bits16(inp["x"])
    ref = moe.moe_forward(xb, inp["logits"].cpu().numpy(), u8(layer.w13q), u8(layer.w13s),
                          u8(layer.w2q), u8(layer.w2s), shape.k, shape.I)
    assert rel_frob(bits16(out), ref["out"]) <= OUT_REL_FROB
    # the oracle's own intermediates: routing and quant bit-exact, and its gmm1
    # ran on exactly the device's xq / xs, so its aq / as are the stage check
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ref["topk_ids"])
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(r["src_to_sorted"].cpu().numpy(), ref["src_to_sorted"])
    assert np.array_equal(u8(r["xq"]), ref["xq"]) and np.array_equal(u8(r["xs"]), ref["xs"])
    aq_g, as_g = u8(aq), u8(as_)
    frac, dist = requant_mismatch(aq_g, as_g, ref["aq"], ref["as_"])
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0, (frac, dist)
    assert rel_frob(bits16(y), ref["y"]) <= OUT_REL_FROB
    _check_gmm2_and_finalize(shape, layer, r, aq_g, as_g, y, out, ref["offsets"])


@pytest.mark.parametrize("T", [t for t in workloads.SKEW_SWEEP_T if t < 16384])
def test_skewed_sweep_whole_oracle_layer(mm, T):
    shape = workloads.CONFIGS["qwen3_30b_skewed"].with_tokens(T)
    inp, layer, r, aq, as_, y, out = _run_both(mm, shape)
    ref = moe.moe_forward(bits16(inp["x"]), inp["logits"].cpu().numpy(), u8(layer.w13q),
                          u8(layer.w13s), u8(layer.w2q), u8(layer.w2s), shape.k, shape.I)
    assert np.array_equal(r["topk_ids"].cpu().numpy(), ref["topk_ids"])
    assert np.array_equal(r["expert_offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(u8(r["xq"]), ref["xq"]) and np.array_equal(u8(r["xs"]), ref["xs"])
    frac, dist = requant_mismatch(u8(aq), u8(as_), ref["aq"], ref["as_"])
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0, (frac, dist)
    assert rel_frob(bits16(y), ref["y"]) <= OUT_REL_FROB
    assert rel_frob(bits16(out), ref["out"]) <= OUT_REL_FROB
