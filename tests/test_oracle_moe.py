"""Pins for the oracle's routing, permutation, GEMMs and finalize (CPU only).

Pinned by brute force on tiny inputs (pure-Python loops written from the
definitions), by library routines where a step reduces to one (scipy softmax
and expit, torch.topk, integer matmul), and by the invariants the pages state
(byte identity of fused and two-step routing quant, the identity layer).
"""

import itertools

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe, mx
from mxfp8_block_scaled_moe_gb300 import workloads


# ---------------------------------------------------------------- routing

def test_route_topk_matches_torch_topk_and_scipy_softmax():
    rng = np.random.default_rng(0)
    logits = rng.normal(0, 1, (200, 16)).astype(np.float32)
    ids, w = moe.route_topk(logits, 4, renormalize=False)
    tv, ti = torch.topk(torch.from_numpy(logits), 4, dim=1)
    assert np.array_equal(ids, ti.numpy())
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(p, ids.astype(np.int64), 1), rtol=1e-14)
    ids2, w2 = moe.route_topk(logits, 4, renormalize=True)
    assert np.array_equal(ids2, ids)
    assert np.allclose(w2.sum(1), 1.0, rtol=1e-14)
    assert np.allclose(w2, w / w.sum(1, keepdims=True), rtol=1e-14)


def test_route_topk_brute_force_with_ties():
    # small integer logits -> many ties; brute force over all k-subsets
    rng = np.random.default_rng(1)
    logits = rng.integers(-2, 3, (300, 6)).astype(np.float32)
    k = 3
    ids, _ = moe.route_topk(logits, k)
    for t in range(logits.shape[0]):
        best = None
        for subset in itertools.combinations(range(6), k):
            # rank: larger logits first, then lexicographically smaller ids
            key = (tuple(sorted((-logits[t, e], e) for e in subset)))
            if best is None or key < best[0]:
                best = (key, [e for _, e in key])
        assert ids[t].tolist() == best[1]


def test_route_topk_k_equals_e_and_one():
    logits = np.array([[0.5, -1.0, 2.0]], np.float32)
    ids, w = moe.route_topk(logits, 3)
    assert ids.tolist() == [[2, 0, 1]] and np.isclose(w.sum(), 1.0)
    ids, w = moe.route_topk(logits, 1)
    assert ids.tolist() == [[2]] and w.tolist() == [[1.0]]


# ---------------------------------------------------------------- permutation

def _permute_brute(ids, E):
    T, k = ids.shape
    rows = []
    counts = []
    for e in range(E):
        c = 0
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    rows.append(t * k + j)
                    c += 1
        counts.append(c)
    return counts, rows


def test_permute_brute_force():
    rng = np.random.default_rng(2)
    for T, E, k in [(1, 4, 2), (7, 5, 3), (33, 8, 2), (16, 3, 3)]:
        logits = rng.normal(0, 1, (T, E)).astype(np.float32)
        ids, _ = moe.route_topk(logits, k)
        counts, offsets, s2s, src2s = moe.permute(ids, E)
        bc, brows = _permute_brute(ids, E)
        assert counts.tolist() == bc
        assert s2s.tolist() == brows
        assert offsets[0] == 0 and offsets[-1] == T * k
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(src2s[s2s], np.arange(T * k))


def test_permute_empty_experts_and_order():
    ids = np.array([[3, 0], [3, 1], [0, 3]], np.int32)
    counts, offsets, s2s, src2s = moe.permute(ids, 5)
    assert counts.tolist() == [2, 1, 0, 3, 0]
    assert offsets.tolist() == [0, 2, 3, 3, 6, 6]
    assert s2s.tolist() == [1, 4, 3, 0, 2, 5]


# ---------------------------------------------------------------- fused route + quant

def test_fused_route_quant_is_byte_identical_to_two_step():
    """init_routing quant_mode=3 == (bf16 permute -> quant) == (quant -> permute)."""
    shape = workloads.CONFIGS["tiny"]
    inp = workloads.make_layer(shape, "cpu", weights=False)
    x = mx.bf16_bits_to_f64(inp["x"].view(torch.int16).numpy().view(np.uint16))
    ids, _ = moe.route_topk(inp["logits"].numpy(), shape.k)
    xq, xs, counts, offsets, s2s, src2s = moe.route_quant(x, ids, shape.E)
    xp = moe.permute_rows(x, s2s, shape.k)
    q2, s2 = mx.mx_quantize(xp)
    assert xq.tobytes() == q2.tobytes() and xs.tobytes() == s2.tobytes()
    qt, st = mx.mx_quantize(x)
    assert xq.tobytes() == qt[s2s // shape.k].tobytes()


# ---------------------------------------------------------------- GEMMs

def _rand_mx(rng, shape, int_valued=False):
    if int_valued:
        v = rng.integers(-8, 9, shape).astype(np.float64)
        q = mx.e4m3_encode(v)
        s = np.full(shape[:-1] + (shape[-1] // 32,), 127, np.uint8)
        return q, s
    return mx.mx_quantize(rng.normal(0, 1, shape))


def test_gmm2_integer_inputs_equal_integer_matmul():
    rng = np.random.default_rng(3)
    E, H, I = 3, 48, 64
    offsets = np.array([0, 5, 5, 12])
    aq, as_ = _rand_mx(rng, (12, I), int_valued=True)
    w2q, w2s = _rand_mx(rng, (E, H, I), int_valued=True)
    y = moe.gmm2(aq, as_, w2q, w2s, offsets, round_bf16=False)
    ai = mx.e4m3_decode(aq).astype(np.int64)
    wi = mx.e4m3_decode(w2q).astype(np.int64)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        assert np.array_equal(y[r0:r1], (ai[r0:r1] @ wi[e].T).astype(np.float64))


def test_gmm1_and_gmm2_brute_force():
    rng = np.random.default_rng(4)
    E, H, I = 2, 64, 32
    offsets = np.array([0, 3, 5])
    xq, xs = _rand_mx(rng, (5, H))
    w13q, w13s = _rand_mx(rng, (E, 2 * I, H))
    w2q, w2s = _rand_mx(rng, (E, H, I))
    aq, as_ = moe.gmm1_swiglu_quant(xq, xs, w13q, w13s, offsets, I)
    a_exact = moe.gmm1_swiglu(xq, xs, w13q, w13s, offsets, I)
    # brute force: element loops over decoded values
    for e in range(E):
        for r in range(offsets[e], offsets[e + 1]):
            xr = [mx.E4M3_TABLE[xq[r, c]] * 2.0 ** (int(xs[r, c // 32]) - 127) for c in range(H)]
            for j in range(I):
                gate = sum(xr[c] * mx.E4M3_TABLE[w13q[e, j, c]] * 2.0 ** (int(w13s[e, j, c // 32]) - 127)
                           for c in range(H))
                up = sum(xr[c] * mx.E4M3_TABLE[w13q[e, I + j, c]] * 2.0 ** (int(w13s[e, I + j, c // 32]) - 127)
                         for c in range(H))
                a = gate * scipy.special.expit(gate) * up
                assert np.isclose(a_exact[r, j], a, rtol=1e-12, atol=1e-300)
        # requant of the fp32-rounded SwiGLU output
    q_ref, s_ref = mx.mx_quantize(a_exact.astype(np.float32).astype(np.float64))
    assert np.array_equal(aq, q_ref) and np.array_equal(as_, s_ref)
    y = moe.gmm2(aq, as_, w2q, w2s, offsets, round_bf16=False)
    for e in range(E):
        for r in range(offsets[e], offsets[e + 1]):
            ar = [mx.E4M3_TABLE[aq[r, c]] * 2.0 ** (int(as_[r, c // 32]) - 127) for c in range(I)]
            for n in range(H):
                want = sum(ar[c] * mx.E4M3_TABLE[w2q[e, n, c]] * 2.0 ** (int(w2s[e, n, c // 32]) - 127)
                           for c in range(I))
                assert np.isclose(y[r, n], want, rtol=1e-12, atol=1e-300)


def test_gmm_single_expert_is_dense_and_gate_up_order():
    rng = np.random.default_rng(5)
    H, I = 64, 32
    xq, xs = _rand_mx(rng, (4, H))
    w13q, w13s = _rand_mx(rng, (1, 2 * I, H))
    a = moe.gmm1_swiglu(xq, xs, w13q, w13s, np.array([0, 4]), I)
    X = mx.mx_dequantize(xq, xs)
    W = mx.mx_dequantize(w13q[0], w13s[0])
    g, u = X @ W[:I].T, X @ W[I:].T
    assert np.allclose(a, g * scipy.special.expit(g) * u, rtol=1e-12)
    # swapping gate and up changes the result (guards the order)
    assert not np.allclose(a, u * scipy.special.expit(u) * g)


def test_silu_special_values():
    g = np.array([0.0, 1000.0, -1000.0, 2.0])
    s = moe.silu(g)
    assert s[0] == 0.0 and s[1] == 1000.0 and s[2] == 0.0
    assert np.isclose(s[3], 2.0 / (1.0 + np.exp(-2.0)))


# ---------------------------------------------------------------- finalize

def test_identity_layer_k1():
    """k=1, weight 1, identity expert: finalize(permute(x)) == x bit-exact."""
    rng = np.random.default_rng(6)
    T, H, E = 37, 64, 5
    xb = mx.f64_to_bf16_bits(rng.normal(0, 1, (T, H)))
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    ids, w = moe.route_topk(logits, 1)
    assert np.all(w == 1.0)
    counts, offsets, s2s, src2s = moe.permute(ids, E)
    y = xb[s2s // 1]
    out = moe.finalize(y, w.astype(np.float32), src2s, 1)
    assert np.array_equal(out, xb)


def test_finalize_convex_combination_of_equal_rows():
    rng = np.random.default_rng(7)
    T, H, E, k = 20, 32, 6, 3
    xb = mx.f64_to_bf16_bits(rng.normal(0, 1, (T, H)))
    ids, w = moe.route_topk(rng.normal(0, 1, (T, E)).astype(np.float32), k)
    counts, offsets, s2s, src2s = moe.permute(ids, E)
    y = xb[s2s // k]
    out = moe.finalize(y, w, src2s, k)
    # sum_j w_j * x = x * sum_j w_j = x (weights renormalised to 1)
    assert np.array_equal(out, xb)


def test_finalize_brute_force():
    rng = np.random.default_rng(8)
    T, H, k = 6, 8, 2
    y = mx.f64_to_bf16_bits(rng.normal(0, 1, (T * k, H)))
    w = rng.uniform(0, 1, (T, k))
    src2s = rng.permutation(T * k).astype(np.int32)
    out = moe.finalize(y, w, src2s, k, round_bf16=False)
    yv = mx.bf16_bits_to_f64(y)
    for t in range(T):
        for h in range(H):
            want = sum(w[t, j] * yv[src2s[t * k + j], h] for j in range(k))
            assert np.isclose(out[t, h], want, rtol=1e-14)


# ---------------------------------------------------------------- whole layer

def test_moe_forward_tiny_layer_runs_and_is_consistent():
    shape = workloads.CONFIGS["tiny"]
    inp = workloads.make_layer(shape, "cpu")
    xb = inp["x"].view(torch.int16).numpy().view(np.uint16)
    w13 = mx.bf16_bits_to_f64(inp["w13"].view(torch.int16).numpy().view(np.uint16))
    w2 = mx.bf16_bits_to_f64(inp["w2"].view(torch.int16).numpy().view(np.uint16))
    w13q, w13s = mx.mx_quantize(w13)
    w2q, w2s = mx.mx_quantize(w2)
    r = moe.moe_forward(xb, inp["logits"].numpy(), w13q, w13s, w2q, w2s, shape.k, shape.I)
    assert r["out"].shape == (shape.T, shape.H)
    assert r["offsets"][-1] == shape.M
    # the bf16 output is close to the unquantized fp64 layer (MXFP8 error only)
    x = mx.bf16_bits_to_f64(xb)
    ids, w = r["topk_ids"], r["topk_w"]
    ref = np.zeros((shape.T, shape.H))
    for t in range(shape.T):
        for j in range(shape.k):
            e = ids[t, j]
            h = w13[e] @ x[t]
            a = moe.silu(h[:shape.I]) * h[shape.I:]
            ref[t] += w[t, j] * (w2[e] @ a)
    got = mx.bf16_bits_to_f64(r["out"])
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.1, rel


def test_w4a8_layer_equals_mxfp8_layer_on_reencoded_weights():
    """The W4A8 layer (MXFP4 expert weights) is the MXFP8 layer fed the same
    weight values as e4m3 codes under the same scales."""
    rng = np.random.default_rng(11)
    T, H, E, k, I = 24, 64, 4, 2, 32
    x = mx.f64_to_bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w13 = rng.standard_normal((E, 2 * I, H)) * 0.05
    w2 = rng.standard_normal((E, H, I)) * 0.05
    q13, s13 = mx.mxfp4_quantize(w13)
    q2, s2 = mx.mxfp4_quantize(w2)
    r4 = moe.moe_forward(x, logits, q13, s13, q2, s2, k, I, wfmt="e2m1")
    e8 = lambda q: mx.e4m3_encode(mx.e2m1_decode(mx.unpack_fp4(q)))
    r8 = moe.moe_forward(x, logits, e8(q13), s13, e8(q2), s2, k, I)
    for key in ("aq", "as_", "y", "out"):
        assert np.array_equal(r4[key], r8[key]), key


def test_w4a4_layer_reduces_to_the_mxfp8_steps_on_reencoded_values():
    """The W4A4 layer (MXFP4 weights and expert inputs) is, step by step, the
    MXFP8 one fed the same values as e4m3 codes under the same scales: the
    routed inputs are the MXFP4 quant of the token rows, gmm1's pre-quant
    SwiGLU output equals the MXFP8 gmm1's on re-encoded operands, its
    requant is the MXFP4 quant of that output rounded to fp32, and gmm2
    equals the MXFP8 gmm2 on re-encoded operands."""
    rng = np.random.default_rng(12)
    T, H, E, k, I = 24, 64, 4, 2, 32
    xb = mx.f64_to_bf16_bits(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    q13, s13 = mx.mxfp4_quantize(rng.standard_normal((E, 2 * I, H)) * 0.05)
    q2, s2 = mx.mxfp4_quantize(rng.standard_normal((E, H, I)) * 0.05)
    r4 = moe.moe_forward(xb, logits, q13, s13, q2, s2, k, I, wfmt="e2m1", afmt="e2m1")
    e8 = lambda q: mx.e4m3_encode(mx.e2m1_decode(mx.unpack_fp4(q)))
    tok = r4["sorted_to_src"].astype(np.int64) // k
    xq_tok, xs_tok = mx.mxfp4_quantize(mx.bf16_bits_to_f64(xb))
    assert np.array_equal(r4["xq"], xq_tok[tok]) and np.array_equal(r4["xs"], xs_tok[tok])
    assert r4["xq"].shape == (T * k, H // 2) and r4["aq"].shape == (T * k, I // 2)
    offs = r4["offsets"]
    a8 = moe.gmm1_swiglu(e8(r4["xq"]), r4["xs"], e8(q13), s13, offs, I)
    a4 = moe.gmm1_swiglu(r4["xq"], r4["xs"], q13, s13, offs, I, wfmt="e2m1", afmt="e2m1")
    assert np.array_equal(a4, a8)
    aq, as_ = mx.mxfp4_quantize(a8.astype(np.float32).astype(np.float64))
    assert np.array_equal(r4["aq"], aq) and np.array_equal(r4["as_"], as_)
    y8 = moe.gmm2(e8(r4["aq"]), r4["as_"], e8(q2), s2, offs)
    assert np.array_equal(r4["y"], y8)


def test_router_logits_integer_brute_force():
    """Integer-valued bf16 inputs: the gate GEMM is an integer dot product."""
    rng = np.random.default_rng(21)
    T, H, E = 3, 40, 5
    xi = rng.integers(-9, 10, (T, H))
    gi = rng.integers(-5, 6, (E, H))
    got = moe.router_logits(mx.f64_to_bf16_bits(xi.astype(np.float64)),
                            mx.f64_to_bf16_bits(gi.astype(np.float64)))
    for t in range(T):
        for e in range(E):
            assert got[t, e] == sum(int(xi[t, h]) * int(gi[e, h]) for h in range(H))


def test_dequantize_gate_matches_torch_casts():
    """e4m3 decode (torch float8_e4m3fn) times 2^(s-127), cast to bf16 by torch."""
    rng = np.random.default_rng(22)
    E, H = 6, 96
    codes = rng.integers(0, 256, (E, H)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C          # NaN codes are outside the contract
    s = rng.integers(100, 140, (E, H // 32)).astype(np.uint8)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    val = dec * torch.from_numpy(np.exp2(np.repeat(s.astype(np.float64) - 127, 32, axis=1)))
    ref = val.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(moe.dequantize_gate(codes, s), ref)


def test_act_quant_and_deq_weight_dispatch_known_values():
    """The format dispatchers against hand-worked codes (OCP MX): a block of
    ones takes scale 2^(0 - 8) in MXFP8 (byte 119, e4m3 256 = 0x78) and
    2^(0 - 2) in MXFP4 (byte 125, e2m1 4 = code 6, two per byte); e4m3 0x38 is
    1.0, e2m1 codes 1 / 2 are 0.5 / 1.0 with the low nibble first."""
    ones = np.ones((2, 32))
    q, s = moe.act_quant(ones, "e4m3")
    assert q.dtype == np.uint8 and np.all(q == 0x78) and np.all(s == 119)
    q, s = moe.act_quant(ones, "e2m1")
    assert q.shape == (2, 16) and np.all(q == 0x66) and np.all(s == 125)
    w = moe.deq_weight(np.full((1, 32), 0x38, np.uint8), np.array([[128]], np.uint8), "e4m3")
    assert np.array_equal(w, np.full((1, 32), 2.0))
    w = moe.deq_weight(np.full((1, 16), 0x21, np.uint8), np.array([[126]], np.uint8), "e2m1")
    assert np.array_equal(w, np.tile([0.25, 0.5], 16)[None, :])
    with pytest.raises(ValueError):
        moe.act_quant(ones, "e5m2")
    with pytest.raises(ValueError):
        moe.deq_weight(q, s, "int4")


def _tiny_layer_q():
    shape = workloads.CONFIGS["tiny"]
    inp = workloads.make_layer(shape, "cpu")
    xb = inp["x"].view(torch.int16).numpy().view(np.uint16)
    w13q, w13s = mx.mx_quantize(mx.bf16_bits_to_f64(inp["w13"].view(torch.int16).numpy().view(np.uint16)))
    w2q, w2s = mx.mx_quantize(mx.bf16_bits_to_f64(inp["w2"].view(torch.int16).numpy().view(np.uint16)))
    return shape, xb, inp["logits"].numpy().astype(np.float64), w13q, w13s, w2q, w2s


def test_layer_invariant_under_expert_relabeling():
    """Renaming the experts (logit columns and weight slabs permuted together)
    leaves every token's output bit-identical: a wrong expert index or offset
    anywhere in the chain breaks it."""
    shape, xb, logits, w13q, w13s, w2q, w2s = _tiny_layer_q()
    E = w13q.shape[0]
    perm = np.random.default_rng(11).permutation(E)   # new id of expert e = perm[e]
    inv = np.argsort(perm)
    ref = moe.moe_forward(xb, logits, w13q, w13s, w2q, w2s, shape.k, shape.I)
    got = moe.moe_forward(xb, logits[:, inv], w13q[inv], w13s[inv], w2q[inv], w2s[inv],
                          shape.k, shape.I)
    assert np.array_equal(got["topk_ids"], perm[ref["topk_ids"]])
    # the softmax sums run over the experts in id order: fp64 rounding only
    np.testing.assert_allclose(got["topk_w"], ref["topk_w"], rtol=1e-13, atol=0)
    assert np.array_equal(got["counts"], ref["counts"][inv])
    for key in ("xq", "xs", "aq", "as_", "y"):   # expanded rows keep their order
        src = np.argsort(ref["sorted_to_src"])    # source slot -> sorted row (reference)
        rows_got = got[key][np.argsort(got["sorted_to_src"])]
        assert np.array_equal(rows_got, ref[key][src]), key
    # tokens whose fp32 combine weights agree have bit-identical outputs
    same = np.all(got["topk_w"].astype(np.float32) == ref["topk_w"].astype(np.float32), axis=1)
    assert same.mean() > 0.9
    assert np.array_equal(got["out"][same], ref["out"][same])


def test_layer_equivariant_under_token_permutation():
    """Tokens are independent: permuting them permutes the routing exactly and
    the outputs up to the summation order inside the library matmul."""
    shape, xb, logits, w13q, w13s, w2q, w2s = _tiny_layer_q()
    p = np.random.default_rng(12).permutation(shape.T)
    ref = moe.moe_forward(xb, logits, w13q, w13s, w2q, w2s, shape.k, shape.I)
    got = moe.moe_forward(xb[p], logits[p], w13q, w13s, w2q, w2s, shape.k, shape.I)
    assert np.array_equal(got["topk_ids"], ref["topk_ids"][p])
    assert np.array_equal(got["topk_w"], ref["topk_w"][p])
    a = mx.bf16_bits_to_f64(got["out"])
    b = mx.bf16_bits_to_f64(ref["out"][p])
    assert np.linalg.norm(a - b) <= 1e-3 * np.linalg.norm(b)
