"""GPU parity of the tcgen05 block-scaled grouped GEMMs against the oracle.

* Exactness pins: integer-valued e4m3 operands with per-block scales in
  [2^-2, 2^2] make every partial sum exactly representable in fp32, so the
  device result must equal the oracle's exact product bit for bit (gmm2) --
  this pins the scale-factor mapping (row, 32-element block) -> element.
* Ragged grouping: empty experts, one-row experts, experts spanning several
  128-row tiles with a ragged tail, the last tile past M.
* Config shapes: every expert of the small layers (the prefill sizes are in
  test_gpu_full_oracle.py).
"""

import numpy as np
import pytest
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import OUT_REL_FROB, REQUANT_MAX_FRAC, bits16, rel_frob, requant_mismatch, u8

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


def _int_mx(rng, shape, lo=-4, hi=4, scale_spread=2):
    """Integer-valued e4m3 codes and per-block scales 2^[-spread, spread]."""
    v = rng.integers(lo, hi + 1, shape).astype(np.float64)
    q = mx.e4m3_encode(v)
    s = (127 + rng.integers(-scale_spread, scale_spread + 1,
                            shape[:-1] + (shape[-1] // 32,))).astype(np.uint8)
    return q, s


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


@pytest.mark.parametrize("M,E,I,H,counts", [
    (128, 1, 128, 256, None),
    (256, 1, 256, 256, None),
    (300, 1, 128, 384, None),
    (394, 6, 256, 256, [0, 1, 130, 0, 257, 6]),
    (394, 6, 128, 384, [0, 1, 130, 0, 257, 6]),
    (7, 4, 128, 128, [3, 0, 0, 4]),
])
def test_gmm2_exact_structured_scales(mm, M, E, I, H, counts):
    rng = np.random.default_rng(M + E + I + H)
    counts = counts or [M]
    offs = _offsets(counts)
    aq, as_ = _int_mx(rng, (M, I))
    w2q, w2s = _int_mx(rng, (E, H, I))
    y = mm.grouped_gemm_mxfp8(_t(aq), _t(as_), _t(w2q), _t(w2s), _t(offs))
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    ref = moe.gmm2(aq, as_, w2q, w2s, offs)
    got = bits16(y)
    mism = np.argwhere(got != ref)
    assert mism.shape[0] == 0, f"{mism.shape[0]} mismatches, first at {mism[:5].tolist()}"


@pytest.mark.parametrize("M,E,H,I,counts", [
    (128, 1, 256, 128, None),
    (394, 6, 256, 256, [0, 1, 130, 0, 257, 6]),
    (260, 3, 384, 384, [129, 0, 131]),
])
def test_gmm1_swiglu_quant_structured(mm, M, E, H, I, counts):
    rng = np.random.default_rng(M * 3 + H + I)
    counts = counts or [M]
    offs = _offsets(counts)
    xq, xs = _int_mx(rng, (M, H), -4, 4, 1)
    w13q, w13s = _int_mx(rng, (E, 2 * I, H), -4, 4, 1)
    # scale w13 down so SwiGLU sees values of order 1..10 (both signs)
    w13s = (w13s.astype(np.int64) - 6).astype(np.uint8)
    aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(_t(xq), _t(xs), _t(w13q), _t(w13s), _t(offs))
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    aq_ref, as_ref = moe.gmm1_swiglu_quant(xq, xs, w13q, w13s, offs, I)
    frac, dist = requant_mismatch(u8(aq), u8(as_), aq_ref, as_ref)
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0, (frac, dist)


def _layer_weights(mm, shape):
    w13, w2 = workloads.make_weights_bf16(shape, DEV)
    w13q, w13s = mm.mx_quantize_3d(w13)
    w2q, w2s = mm.mx_quantize_3d(w2)
    return w13q, w13s, w2q, w2s


@pytest.mark.parametrize("cfg", ["tiny", "qwen3_30b_decode"])
def test_gmm_chain_on_config(mm, cfg):
    shape = workloads.CONFIGS[cfg]
    inp = workloads.make_layer(shape, DEV, weights=False)
    w13q, w13s, w2q, w2s = _layer_weights(mm, shape)
    r = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(r["xq"], r["xs"], w13q, w13s, r["expert_offsets"])
    y = mm.grouped_gemm_mxfp8(aq, as_, w2q, w2s, r["expert_offsets"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    offs = r["expert_offsets"].cpu().numpy()
    experts = list(range(shape.E))   # every expert (the prefill sizes: test_gpu_full_oracle)
    rows = np.concatenate([np.arange(offs[e], offs[e + 1]) for e in experts]).astype(np.int64)
    xq_h, xs_h = u8(r["xq"]), u8(r["xs"])
    w13q_h = {e: u8(w13q[e]) for e in experts}
    w13s_h = {e: u8(w13s[e]) for e in experts}
    w2q_h = {e: u8(w2q[e]) for e in experts}
    w2s_h = {e: u8(w2s[e]) for e in experts}
    aq_g, as_g, y_g = u8(aq), u8(as_), bits16(y)
    aq_ref = np.zeros_like(aq_g)
    as_ref = np.zeros_like(as_g)
    y_ref = np.zeros_like(y_g)
    for e in experts:
        r0, r1 = offs[e], offs[e + 1]
        if r1 == r0:
            continue
        sub = np.array([0, r1 - r0])
        a_q, a_s = moe.gmm1_swiglu_quant(xq_h[r0:r1], xs_h[r0:r1], w13q_h[e][None], w13s_h[e][None],
                                         sub, shape.I)
        aq_ref[r0:r1], as_ref[r0:r1] = a_q, a_s
        # gmm2 from the device's own gmm1 output (stage-by-stage parity)
        y_ref[r0:r1] = moe.gmm2(aq_g[r0:r1], as_g[r0:r1], w2q_h[e][None], w2s_h[e][None], sub)
    frac, dist = requant_mismatch(aq_g[rows], as_g[rows], aq_ref[rows], as_ref[rows])
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0, (frac, dist)
    assert rel_frob(y_g[rows], y_ref[rows]) <= OUT_REL_FROB


def test_gmm_empty_and_all_in_one_expert(mm):
    rng = np.random.default_rng(9)
    E, H, I = 8, 256, 128
    w13q, w13s = mx.mx_quantize(rng.normal(0, 0.05, (E, 2 * I, H)))
    w2q, w2s = mx.mx_quantize(rng.normal(0, 0.05, (E, H, I)))
    # M == 0: nothing to do, no error
    z = torch.zeros(0, H, dtype=torch.uint8, device=DEV)
    zs = torch.zeros(0, H // 32, dtype=torch.uint8, device=DEV)
    offs0 = _t(np.zeros(E + 1, np.int64))
    aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(z, zs, _t(w13q), _t(w13s), offs0)
    assert aq.shape == (0, I)
    # every row in the last expert
    M = 200
    xq, xs = mx.mx_quantize(rng.normal(0, 1, (M, H)))
    offs = _offsets([0] * (E - 1) + [M])
    aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(_t(xq), _t(xs), _t(w13q), _t(w13s), _t(offs))
    y = mm.grouped_gemm_mxfp8(aq, as_, _t(w2q), _t(w2s), _t(offs))
    torch.cuda.synchronize()
    aq_ref, as_ref = moe.gmm1_swiglu_quant(xq, xs, w13q, w13s, offs, I)
    frac, dist = requant_mismatch(u8(aq), u8(as_), aq_ref, as_ref)
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0
    y_ref = moe.gmm2(u8(aq), u8(as_), w2q, w2s, offs)
    assert rel_frob(bits16(y), y_ref) <= OUT_REL_FROB


def test_gemm_is_deterministic(mm):
    shape = workloads.CONFIGS["tiny"]
    inp = workloads.make_layer(shape, DEV, weights=False)
    w13q, w13s, w2q, w2s = _layer_weights(mm, shape)
    r = mm.moe_route_quant_mxfp8(inp["x"], inp["logits"], shape.k)
    outs = []
    for _ in range(2):
        aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(r["xq"], r["xs"], w13q, w13s, r["expert_offsets"])
        y = mm.grouped_gemm_mxfp8(aq, as_, w2q, w2s, r["expert_offsets"])
        outs.append((aq, as_, y))
    torch.cuda.synchronize()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
