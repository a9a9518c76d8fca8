"""MoE expert-forward steps of the MXFP8 path (CPU oracle, float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

The forward, as "Quantization on Ascend" (MoE MXFP8 notes, "Forward") and
sglang PR #32266 (commit note adding the fused experts kernel: "routing ->
act quant -> swiglu_quant_v2 -> grouped_matmul -> finalize_routing") describe
it:

1. top-k routing of each token over E experts (softmax, top-k, renormalise);
2. init_routing with quant_mode=3: the token rows are expanded k times,
   grouped by expert, and MX-quantized on the way (payload + e8m0 scale);
   per-expert token counts come out too;
3. gmm1: per expert, the grouped GEMM with w13 (gate rows then up rows),
   SwiGLU, and an MXFP8 requant that returns (payload, block scale);
4. gmm2: per expert, the grouped GEMM with w2, bf16 output;
5. finalize routing: the weighted top-k combine back to token order.

Shapes: T tokens, H hidden, E experts, k top-k, I moe_intermediate,
M = T*k expanded rows.  w13 is [E, 2I, H] and w2 is [E, H, I] (PR #32266,
note on the inherited create_weights), both K-contiguous and MX-quantized
along K.

Readings of points the pages leave open (each is one choice, stated once):

* top-k ties go to the lower expert id; the k slots of a token are in
  descending logit order;
* rows of one expert are ordered by the flat assignment index t*k + j (token
  order), which fixes the permutation uniquely;
* w13 rows [0, I) are the gate, rows [I, 2I) the up projection, and SwiGLU
  is silu(gate) * up with silu(g) = g / (1 + e^-g), no clamp;
* GEMM1 accumulates exactly (fp64 here); the SwiGLU output is rounded to
  fp32 before the requant, because the requant decision (block amax -> scale,
  element -> e4m3 code) is taken in the kernel's precision;
* GEMM2's output is bf16 (round-to-nearest-even of the exact product);
* the routing weights are applied in finalize, which accumulates exactly and
  rounds once to bf16; no token is dropped (no capacity limit);
* W4A8 (MXFP4 weights): the shared scale is floor(log2 amax) - 2 (2 = the
  largest power-of-two exponent of e2m1, as 8 is for e4m3), elements round to
  nearest-even and saturate at +-6, and a packed byte holds element 2i in its
  low nibble and element 2i+1 in its high nibble;
* W4A4 ("Quantization on Ascend", W4A4 MoE notes: each expert input is
  quantized to MXFP4 right before the grouped matmul): the routed hidden
  states and the SwiGLU output (the inputs of gmm1 and gmm2) are MXFP4 with
  the rule above, the SwiGLU output rounded to fp32 first as in the MXFP8
  requant.
"""

from __future__ import annotations

import numpy as np

from . import mx


# ----------------------------------------------------------------------------
# 0. router gate (upstream of the routing)
# ----------------------------------------------------------------------------

def router_logits(x_bf16_bits, gate_bf16_bits) -> np.ndarray:
    """The router gate, a plain linear layer without bias: logits[t, e] =
    sum_h x[t, h] * gate[e, h], exact (fp64) on the bf16 values.
    ("Quantization on Ascend", MoE MXFP8 notes: the gate is a
    ReplicatedLinear, bf16 on the online path.)"""
    return mx.bf16_bits_to_f64(x_bf16_bits) @ mx.bf16_bits_to_f64(gate_bf16_bits).T


def dequantize_gate(q, s) -> np.ndarray:
    """An offline MXFP8 router gate dequantized to bf16 bits: each element's
    decoded e4m3 value times its block's 2^(scale - 127), rounded once to
    bf16 (exact when the value is in bf16's range).  The pages: the offline
    gate must be dequantized with its block scale (PR #32266 router-gate
    note)."""
    return mx.f64_to_bf16_bits(mx.mx_dequantize(q, s))


# ----------------------------------------------------------------------------
# 1. routing
# ----------------------------------------------------------------------------

def route_topk(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k softmax routing.

    ``logits`` float32 [T, E] (the router output; both the oracle and the
    kernel read the same fp32 values, so the selection is an exact compare).
    Returns (topk_ids int32 [T, k], topk_w float64 [T, k]).

    p = softmax(logits[t]) in fp64; the k experts with the largest logits are
    chosen (ties -> lower id), in descending order; with ``renormalize`` the
    chosen probabilities are divided by their sum.
    """
    logits = np.asarray(logits, dtype=np.float32)
    if not np.all(np.isfinite(logits)):
        raise ValueError("route_topk: non-finite logits are outside the contract")
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("route_topk: need 1 <= k <= E")
    l64 = logits.astype(np.float64)
    ids_grid = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary -> sort by -logit, then by expert id
    order = np.lexsort((ids_grid, -l64), axis=1)
    topk_ids = order[:, :k].astype(np.int32)
    ex = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p = ex / ex.sum(axis=1, keepdims=True)
    w = np.take_along_axis(p, topk_ids.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return topk_ids, w


# ----------------------------------------------------------------------------
# 2. permutation (init_routing) and fused activation quant
# ----------------------------------------------------------------------------

def permute(topk_ids: np.ndarray, E: int):
    """Group the T*k assignments by expert.

    Returns (counts int64 [E], offsets int64 [E+1], sorted_to_src int32 [M],
    src_to_sorted int32 [M]).  counts is the dispatcher's COUNT group list,
    offsets its cumulative form with a leading 0 (gmm1 wants the cumulative
    form, gmm2 the count form: PR #30768 report, GroupedMatmulSwigluQuant
    excerpt).  Within an expert the rows keep flat-index order t*k + j.
    sorted_to_src[p] is the flat index of expanded row p, src_to_sorted is
    its inverse.
    """
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("permute: expert id out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    sorted_to_src = np.argsort(flat, kind="stable").astype(np.int32)
    src_to_sorted = np.empty_like(sorted_to_src)
    src_to_sorted[sorted_to_src] = np.arange(flat.size, dtype=np.int32)
    return counts, offsets, sorted_to_src, src_to_sorted


def act_quant(x: np.ndarray, afmt: str = "e4m3"):
    """MX-quantize activations along the last axis: MXFP8 (e4m3 codes) or,
    for W4A4, MXFP4 (packed e2m1, [..., K/2])."""
    if afmt == "e4m3":
        return mx.mx_quantize(x)
    if afmt == "e2m1":
        return mx.mxfp4_quantize(x)
    raise ValueError(f"unknown activation format {afmt!r}")


def route_quant(x: np.ndarray, topk_ids: np.ndarray, E: int, afmt: str = "e4m3"):
    """init_routing with quant_mode=3: permuted rows, MX-quantized along H.

    ``x`` float64 [T, H] (exact values of the bf16 hidden states).  Each token
    row is quantized (its blocks depend only on the row) and the result is
    placed in its k expanded rows.  Returns (xq uint8 [M, H] (packed [M, H/2]
    for ``afmt="e2m1"``), xs uint8 [M, ceil(H/32)], counts, offsets,
    sorted_to_src, src_to_sorted).
    """
    k = topk_ids.shape[1]
    counts, offsets, s2s, src2s = permute(topk_ids, E)
    q_tok, s_tok = act_quant(x, afmt)
    tok = s2s.astype(np.int64) // k
    return q_tok[tok], s_tok[tok], counts, offsets, s2s, src2s


def permute_rows(x: np.ndarray, sorted_to_src: np.ndarray, k: int) -> np.ndarray:
    """init_routing without quant: expanded row p is token sorted_to_src[p]//k."""
    return np.asarray(x)[np.asarray(sorted_to_src, dtype=np.int64) // k]


# ----------------------------------------------------------------------------
# 3. gmm1: grouped GEMM over w13 + SwiGLU + MXFP8 requant
# ----------------------------------------------------------------------------

def deq_weight(q, s, wfmt: str = "e4m3"):
    """Dequantize an MX matrix (one expert's weights, or activation rows):
    MXFP8 (e4m3 codes [N, K]) or, for the W4A8 / W4A4 paths ("Quantization on
    Ascend", W4A8 and W4A4 notes), MXFP4 (packed e2m1 [N, K/2]); e8m0 scales
    [N, K/32] either way."""
    if wfmt == "e4m3":
        return mx.mx_dequantize(q, s)
    if wfmt == "e2m1":
        return mx.mxfp4_dequantize(q, s)
    raise ValueError(f"unknown weight format {wfmt!r}")


def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + e^-g) in fp64 (e^-g may overflow to inf -> -0/+0)."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def gmm1_swiglu_quant(xq, xs, w13q, w13s, offsets, I: int, experts=None, wfmt: str = "e4m3",
                      afmt: str = "e4m3"):
    """Per expert e and its rows [off_e, off_{e+1}):

    h = deq(xq rows) @ deq(w13[e])^T (fp64, exact products), gate = h[:, :I],
    up = h[:, I:], a = silu(gate) * up, rounded to fp32, then MX-quantized
    along I (in ``afmt``: the activations' format is also gmm2's input
    format).  Returns (aq uint8 [M, I] (packed [M, I/2] for e2m1), as uint8
    [M, I/32]); rows of experts not listed in ``experts`` (default: all)
    stay zero.
    """
    M = xq.shape[0]
    E = w13q.shape[0]
    aq = np.zeros((M, I // 2 if afmt == "e2m1" else I), np.uint8)
    as_ = np.zeros((M, mx.n_scales(I)), np.uint8)
    for e in range(E) if experts is None else experts:
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        a_in = deq_weight(xq[r0:r1], xs[r0:r1], afmt)
        w = deq_weight(w13q[e], w13s[e], wfmt)
        h = a_in @ w.T
        a = silu(h[:, :I]) * h[:, I:]
        a32 = a.astype(np.float32).astype(np.float64)
        aq[r0:r1], as_[r0:r1] = act_quant(a32, afmt)
    return aq, as_


def gmm1_swiglu(xq, xs, w13q, w13s, offsets, I: int, experts=None, wfmt: str = "e4m3",
                afmt: str = "e4m3"):
    """The unquantized SwiGLU output a (fp64) of gmm1, for error reporting."""
    M = xq.shape[0]
    a_out = np.zeros((M, I))
    for e in range(w13q.shape[0]) if experts is None else experts:
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        h = deq_weight(xq[r0:r1], xs[r0:r1], afmt) @ deq_weight(w13q[e], w13s[e], wfmt).T
        a_out[r0:r1] = silu(h[:, :I]) * h[:, I:]
    return a_out


# ----------------------------------------------------------------------------
# 4. gmm2: grouped GEMM over w2, bf16 output
# ----------------------------------------------------------------------------

def gmm2(aq, as_, w2q, w2s, offsets, experts=None, round_bf16: bool = True,
         wfmt: str = "e4m3", afmt: str = "e4m3"):
    """Per expert: y = deq(aq rows) @ deq(w2[e])^T in fp64.

    Returns bf16 bit patterns uint16 [M, H] (``round_bf16``) or the exact
    fp64 product.  Rows of skipped experts stay zero.
    """
    M = aq.shape[0]
    E, H = w2q.shape[0], w2q.shape[1]
    y = np.zeros((M, H))
    for e in range(E) if experts is None else experts:
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        y[r0:r1] = deq_weight(aq[r0:r1], as_[r0:r1], afmt) @ deq_weight(w2q[e], w2s[e], wfmt).T
    return mx.f64_to_bf16_bits(y) if round_bf16 else y


# ----------------------------------------------------------------------------
# 5. finalize routing
# ----------------------------------------------------------------------------

def finalize(y_bf16_bits, topk_w, src_to_sorted, k: int, round_bf16: bool = True):
    """out[t] = sum_j topk_w[t, j] * y[src_to_sorted[t*k + j]].

    y is GEMM2's bf16 output; the weights are the fp32 routing weights the
    kernel stores.  The sum is exact (fp64) and rounded once to bf16.
    """
    y = mx.bf16_bits_to_f64(y_bf16_bits)
    w = np.asarray(topk_w, dtype=np.float64)
    T = w.shape[0]
    idx = np.asarray(src_to_sorted, dtype=np.int64).reshape(T, k)
    out = np.zeros((T, y.shape[1]))
    for j in range(k):
        out += w[:, j:j + 1] * y[idx[:, j]]
    return mx.f64_to_bf16_bits(out) if round_bf16 else out


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------

def moe_forward(x_bf16_bits, logits, w13q, w13s, w2q, w2s, k: int, I: int,
                renormalize: bool = True, wfmt: str = "e4m3", afmt: str = "e4m3"):
    """The whole MXFP8 expert forward; returns a dict of every intermediate.
    ``wfmt="e2m1"`` runs the W4A8 variant: MXFP4 (packed e2m1) expert weights
    with the same MXFP8 activations, routing, requant and finalize; adding
    ``afmt="e2m1"`` runs W4A4 (both grouped GEMMs' inputs MXFP4).

    The routing weights fed to finalize are rounded to fp32 first: the
    kernels carry them as fp32, and the rounding of the combine input is a
    property of the data path, not of the arithmetic.
    """
    x = mx.bf16_bits_to_f64(x_bf16_bits)
    E = w13q.shape[0]
    ids, w = route_topk(logits, k, renormalize)
    xq, xs, counts, offsets, s2s, src2s = route_quant(x, ids, E, afmt)
    aq, as_ = gmm1_swiglu_quant(xq, xs, w13q, w13s, offsets, I, wfmt=wfmt, afmt=afmt)
    y = gmm2(aq, as_, w2q, w2s, offsets, wfmt=wfmt, afmt=afmt)
    w32 = w.astype(np.float32)
    out = finalize(y, w32, src2s, k)
    return dict(topk_ids=ids, topk_w=w, xq=xq, xs=xs, counts=counts, offsets=offsets,
                sorted_to_src=s2s, src_to_sorted=src2s, aq=aq, as_=as_, y=y, out=out)
