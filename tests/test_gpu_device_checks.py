"""Device-side failure detection through the C ABI, with no GPU fault.

* Consistency checks: the grouped GEMMs read the caller's expert offsets on
  the device; an array that is not {0 = o_0 <= o_1 <= ... <= o_E = M} would
  send tiles to rows outside [0, M), so the kernels check it while they build
  their tile schedule, record MXMOE_ERR_DEVICE_CHECK and write nothing.
  Finalize checks every src_to_sorted index against [0, T*k).  The malformed
  arrays are ordinary host-made inputs: the kernels only read them.
* Bounded waits: with a wait limit of one clock cycle, the first barrier
  wait that does not complete at once runs out; the kernel must record
  MXMOE_ERR_DEVICE_TIMEOUT, drain its copies and MMAs, free tensor memory and
  return, and the next call must be correct.
"""

import ctypes as C

import numpy as np
import pytest
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads

from _util import REQUANT_MAX_FRAC, bits16, finalize_bound_ok, requant_mismatch, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
ERR_DEVICE_TIMEOUT = 7
ERR_DEVICE_CHECK = 8
SENTINEL = 0x5A


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


def _p(t):
    return C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _int_mx(rng, shape, lo, hi, spread):
    q = mx.e4m3_encode(rng.integers(lo, hi + 1, shape).astype(np.float64))
    s = (127 + rng.integers(-spread, spread + 1, shape[:-1] + (shape[-1] // 32,))).astype(np.uint8)
    return q, s


M, E, H, I = 300, 4, 256, 128
BAD_OFFSETS = {
    "decreasing": [0, 200, 100, 250, M],
    "first_not_zero": [5, 100, 150, 200, M],
    "last_below_M": [0, 100, 150, 200, M - 1],
    "last_above_M": [0, 100, 150, 200, M + 128],
    "negative": [0, -128, 150, 200, M],
    "huge": [0, 100, 150, 1 << 40, M],
}


@pytest.fixture(scope="module")
def gemm_inputs():
    rng = np.random.default_rng(21)
    xq, xs = _int_mx(rng, (M, H), -4, 4, 1)
    w13q, w13s = _int_mx(rng, (E, 2 * I, H), -4, 4, 1)
    w13s = (w13s.astype(np.int64) - 6).astype(np.uint8)
    aq, as_ = _int_mx(rng, (M, I), -4, 4, 1)
    w2q, w2s = _int_mx(rng, (E, H, I), -4, 4, 1)
    return dict(xq=xq, xs=xs, w13q=w13q, w13s=w13s, aq=aq, as_=as_, w2q=w2q, w2s=w2s)


def _gmm1(mm, g, offs):
    lib = mm._lib.load()
    aq = torch.full((M, I), SENTINEL, dtype=torch.uint8, device=DEV)
    as_ = torch.full((M, I // 32), SENTINEL, dtype=torch.uint8, device=DEV)
    d = {k: _t(v) for k, v in g.items()}
    rc = lib.grouped_gemm_swiglu_quant_mxfp8(_p(d["xq"]), _p(d["xs"]), _p(d["w13q"]),
                                             _p(d["w13s"]), _p(offs), M, E, H, I, _p(aq), _p(as_),
                                             _stream())
    assert rc == 0
    return aq, as_


def _gmm2(mm, g, offs):
    lib = mm._lib.load()
    y = torch.full((M, H), SENTINEL * 257, dtype=torch.int16, device=DEV)
    d = {k: _t(v) for k, v in g.items()}
    rc = lib.grouped_gemm_mxfp8(_p(d["aq"]), _p(d["as_"]), _p(d["w2q"]), _p(d["w2s"]), _p(offs),
                                M, E, I, H, _p(y), _stream())
    assert rc == 0
    return y


@pytest.mark.parametrize("case", sorted(BAD_OFFSETS))
def test_grouped_gemms_reject_malformed_offsets(mm, gemm_inputs, case):
    assert mm.device_status(clear=True) == 0
    offs = _t(np.array(BAD_OFFSETS[case], np.int64))
    aq, as_ = _gmm1(mm, gemm_inputs, offs)
    assert mm.device_status(clear=True) == ERR_DEVICE_CHECK
    assert bool((aq == SENTINEL).all()) and bool((as_ == SENTINEL).all()), "gmm1 wrote rows"
    y = _gmm2(mm, gemm_inputs, offs)
    assert mm.device_status(clear=True) == ERR_DEVICE_CHECK
    assert bool((y == SENTINEL * 257).all()), "gmm2 wrote rows"


def test_grouped_gemms_correct_after_a_rejected_call(mm, gemm_inputs):
    g = gemm_inputs
    bad = _t(np.array(BAD_OFFSETS["decreasing"], np.int64))
    _gmm2(mm, g, bad)
    assert mm.device_status(clear=True) == ERR_DEVICE_CHECK
    counts = [0, 1, 170, 129]   # empty, one-row and multi-tile experts, ragged tails
    offs_h = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    offs = _t(offs_h)
    aq, as_ = _gmm1(mm, g, offs)
    y = _gmm2(mm, g, offs)
    torch.cuda.synchronize()
    assert mm.device_status(clear=True) == 0
    aq_ref, as_ref = moe.gmm1_swiglu_quant(g["xq"], g["xs"], g["w13q"], g["w13s"], offs_h, I)
    frac, dist = requant_mismatch(u8(aq), u8(as_), aq_ref, as_ref)
    assert frac <= REQUANT_MAX_FRAC and dist <= 1.0, (frac, dist)
    # integer operands with scales 2^[-1, 1]: every partial sum is exact in fp32
    assert np.array_equal(bits16(y), moe.gmm2(g["aq"], g["as_"], g["w2q"], g["w2s"], offs_h))


@pytest.mark.parametrize("bad_index", [-1, "T*k", 1 << 30])
def test_finalize_rejects_out_of_range_indices(mm, bad_index):
    rng = np.random.default_rng(22)
    T, k, Hf = 40, 4, 256
    Mf = T * k
    y = torch.from_numpy(rng.normal(0, 1, (Mf, Hf)).astype(np.float32)).to(DEV).to(torch.bfloat16)
    w = _t(rng.uniform(0.1, 1.0, (T, k)).astype(np.float32))
    idx_h = rng.permutation(Mf).astype(np.int32)
    idx_h[7] = Mf if bad_index == "T*k" else bad_index
    idx = _t(idx_h)
    out = torch.empty(T, Hf, dtype=torch.bfloat16, device=DEV)
    assert mm.device_status(clear=True) == 0
    rc = mm._lib.load().moe_finalize_routing(_p(y), _p(w), _p(idx), T, k, Hf, _p(out), _stream())
    assert rc == 0
    assert mm.device_status(clear=True) == ERR_DEVICE_CHECK
    # the bad slot contributes nothing; every token, that one included, is the
    # combine of its in-range slots
    idx_ok = idx_h.copy()
    idx_ok[7] = 0
    w_ok = w.cpu().numpy().copy()
    w_ok[7 // k, 7 % k] = 0.0
    assert finalize_bound_ok(bits16(out), bits16(y), w_ok, idx_ok, k) == 0.0


def test_device_wait_timeout_reports_and_recovers(mm):
    """A wait limit of one cycle: the epilogue waits for a 128-slice mainloop
    (K = 16384), far longer than any single barrier poll, so its wait must run
    out; the kernel returns MXMOE_ERR_DEVICE_TIMEOUT and the next call with
    the default limit is bit-exact again."""
    rng = np.random.default_rng(10)
    Mt, Et, It, Ht = 256, 1, 16384, 256
    offs = np.array([0, Mt], np.int64)
    # integers in [-2, 2], unit scales: every partial sum is an exact fp32 integer
    aq, as_ = _int_mx(rng, (Mt, It), -2, 2, 0)
    w2q, w2s = _int_mx(rng, (Et, Ht, It), -2, 2, 0)
    args = (_t(aq), _t(as_), _t(w2q), _t(w2s), _t(offs))
    assert mm.device_status(clear=True) == 0
    mm.set_wait_limit_cycles(1)
    try:
        mm.grouped_gemm_mxfp8(*args)
        status = mm.device_status(clear=True)
    finally:
        mm.set_wait_limit_cycles(0)
    assert status == ERR_DEVICE_TIMEOUT
    y = mm.grouped_gemm_mxfp8(*args)
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert np.array_equal(bits16(y), moe.gmm2(aq, as_, w2q, w2s, offs))


def test_small_batch_gemm_chain_wait_timeout_reports_and_recovers(mm):
    """The 32-token layer runs both grouped GEMMs as one kernel whose producer
    waits on other CTAs' gmm1 units; with a wait limit of one cycle its waits
    run out, the layer reports MXMOE_ERR_DEVICE_TIMEOUT, and the next call with
    the default limit gives the bytes of a call that never timed out."""
    shape = workloads.CONFIGS["qwen3_30b_decode"]
    inp = workloads.make_layer(shape, "cuda")
    layer = mm.MXFP8MoELayer.from_bf16(inp["w13"], inp["w2"], shape.k)
    ref = layer(inp["x"], inp["logits"]).clone()
    torch.cuda.synchronize()
    assert mm.device_status(clear=True) == 0
    mm.set_wait_limit_cycles(1)
    try:
        layer(inp["x"], inp["logits"])
        status = mm.device_status(clear=True)
    finally:
        mm.set_wait_limit_cycles(0)
    assert status == ERR_DEVICE_TIMEOUT
    out = layer(inp["x"], inp["logits"])
    torch.cuda.synchronize()
    assert mm.device_status() == 0
    assert torch.equal(out, ref)
