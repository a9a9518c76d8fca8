"""Test helpers: tensor <-> numpy bit views and the parity comparators.

Tolerances (stated once, used by every parity test):

* quantization, scales, top-k ids, permutation indices, counts, offsets:
  bit-exact;
* routing weights: relative error <= 1e-6 (the device keeps the softmax's
  exponent arguments exact and its denominator compensated, so only the fp32
  exp error and a final rounding or two remain against the oracle's fp64);
* MXFP8 requant (gmm1 output): an element may differ from the oracle by at
  most one e4m3 grid step, on at most 0.1% of elements; a block whose scale
  byte differs counts as 32 mismatched elements;
* bf16 outputs (gmm2, finalize, the layer): relative Frobenius error <= 2e-3
  against the oracle's fp64-accumulated emulation of the same MXFP8 math.
"""

import numpy as np
import torch

from oracle import mx

REQUANT_MAX_FRAC = 1e-3
OUT_REL_FROB = 2e-3
TOPK_W_RTOL = 1e-6


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).cpu().numpy()


def to_bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def requant_mismatch(aq, as_, aq_ref, as_ref):
    """(fraction of mismatched elements, max grid-step distance) per the rule above."""
    aq, as_, aq_ref, as_ref = (np.asarray(v) for v in (aq, as_, aq_ref, as_ref))
    M, I = aq.shape
    nb = I // 32
    sdiff = (as_ != as_ref)
    bad = np.repeat(sdiff, 32, axis=1)
    same = ~bad
    v = mx.e4m3_decode(aq)
    vr = mx.e4m3_decode(aq_ref)
    step = mx.e4m3_ulp(np.maximum(np.abs(v), np.abs(vr)))
    dist = np.where(same, np.abs(v - vr) / step, 0.0)
    elem_bad = same & (aq != aq_ref) & ~((v == 0) & (vr == 0))
    n_bad = int(bad.sum() + elem_bad.sum())
    return n_bad / max(1, M * I), float(dist.max() if dist.size else 0.0)


def rel_frob(got_bits, want_bits) -> float:
    g = mx.bf16_bits_to_f64(got_bits)
    w = mx.bf16_bits_to_f64(want_bits)
    den = np.linalg.norm(w)
    return float(np.linalg.norm(g - w) / (den if den > 0 else 1.0))


def finalize_bound_ok(got_bits, y_bits, topk_w, src_to_sorted, k):
    """Elementwise: the device's fp32-accumulated, bf16-rounded combine lies
    within one bf16 rounding (2^-8 relative) of the exact fp64 sum, plus the
    fp32 accumulation error bound 2^-20 * sum_j |w_j| |y_j|.  Returns the
    fraction of elements outside that bound (expected 0)."""
    from oracle import moe as _moe
    y = mx.bf16_bits_to_f64(y_bits)
    w = np.asarray(topk_w, dtype=np.float64)
    T = w.shape[0]
    idx = np.asarray(src_to_sorted, dtype=np.int64).reshape(T, k)
    exact = _moe.finalize(y_bits, w, src_to_sorted, k, round_bf16=False)
    mag = np.zeros_like(exact)
    for j in range(k):
        mag += np.abs(w[:, j:j + 1]) * np.abs(y[idx[:, j]])
    got = mx.bf16_bits_to_f64(got_bits)
    bad = np.abs(got - exact) > 2.0 ** -8 * np.abs(exact) + 2.0 ** -20 * mag
    return float(bad.mean())
