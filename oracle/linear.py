"""Dense MXFP8 linear (CPU oracle, float64).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

"Quantization on Ascend" (MXFP8 implementation notes, online path): a dense
linear layer's bf16 weight is MX-quantized once at load along its input
dimension K, the activations are MX-quantized per token at inference, and a
block-scaled matmul with one e8m0 scale per 32 elements of K
(group_sizes [1, 1, 32]) gives the output.  The weight is kept [N, K]
(K contiguous); the pages' "pre-transposed [in, out]" weight is a view of
those bytes.

K may leave a partial last block: sglang PR #32266 summary, "Offline partial
MXFP8 block-scale layout" -- ceil(K/32) scales per row (135 for K = 4304),
the last block's scale taken over the elements that exist.

Readings (each one choice, stated once): the activation quant is the same
block rule as the weights' (``mx.mx_quantize``); the matmul is exact (fp64
here; the device accumulates in fp32) and its output is rounded once to bf16
(round-to-nearest-even).
"""

from __future__ import annotations

import numpy as np

from . import mx


def quantize_activations(x_bf16_bits: np.ndarray, fmt: str = "e4m3"):
    """Per-token MX quant of bf16 activations [M, K]: (q uint8 [M, K] (packed
    [M, K/2] MXFP4 for ``fmt="e2m1"``), scale uint8 [M, ceil(K/32)])."""
    x = mx.bf16_bits_to_f64(np.asarray(x_bf16_bits, dtype=np.uint16))
    return mx.mxfp4_quantize(x) if fmt == "e2m1" else mx.mx_quantize(x)


def _deq(q, s, fmt):
    return mx.mxfp4_dequantize(q, s) if fmt == "e2m1" else mx.mx_dequantize(q, s)


def linear(xq, xs, wq, ws, round_bf16: bool = True, fmt: str = "e4m3"):
    """out = deq(xq, xs) @ deq(wq, ws)^T, exact, then bf16 (``round_bf16``).

    xq [M, K], xs [M, ceil(K/32)], wq [N, K], ws [N, ceil(K/32)]; with
    ``fmt="e2m1"`` (W4A4) both payloads are packed MXFP4, [.., K/2].
    """
    y = _deq(xq, xs, fmt) @ _deq(wq, ws, fmt).T
    return mx.f64_to_bf16_bits(y) if round_bf16 else y


def mxfp8_linear(x_bf16_bits, wq, ws, round_bf16: bool = True):
    """The whole dense MXFP8 linear on bf16 activations: quant, then GEMM."""
    xq, xs = quantize_activations(x_bf16_bits)
    return linear(xq, xs, wq, ws, round_bf16)


def mxfp4_linear(x_bf16_bits, wp, ws, round_bf16: bool = True):
    """The W4A4 dense linear ("Quantization on Ascend", W4A4 notes, offline
    single-level path: both matmul inputs packed float4_e2m1fn_x2 with one
    UE8M0 scale per 32 elements of K): MXFP4 per-token activation quant,
    then the GEMM on packed MXFP4 weights [N, K/2].  K % 32 == 0 (the device
    path takes K % 128 == 0)."""
    xq, xs = quantize_activations(x_bf16_bits, "e2m1")
    return linear(xq, xs, wp, ws, round_bf16, fmt="e2m1")
