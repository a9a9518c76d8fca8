"""Seeded synthetic MoE-layer inputs.

The one module that serves both the CUDA path and the CPU oracle: it draws
random numbers and lays them out, and holds no step of the MXFP8 method (no
routing, quantization, GEMM or combine).  The router logits are produced here
by the upstream gate projection (or, for the skewed-load case, by Gumbel
sampling), because the path consumes logits as an input.

Shapes stand in for the MoE layers the pages target (Qwen3 MoE on
"Quantization on Ascend" and sglang PR #30768; the 16K-token random prefill of
sglang PR #40519): hidden states N(0,1) in bf16, expert weights N(0, 0.02) in
bf16 (quantized at load by the library), a bf16 router gate.

Generation uses a ``torch.Generator`` on the requested device, so a CPU run and
a CUDA run of the same seed give different (but each reproducible) bytes;
every test feeds the same bytes to both sides.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int            # tokens
    H: int            # hidden size (GEMM1 K, GEMM2 N)
    E: int            # experts
    k: int            # top-k
    I: int            # moe_intermediate size (GEMM1 N = 2I, GEMM2 K)
    seed: int
    gate_std: float = 0.02
    outlier_frac: float = 0.0   # fraction of hidden channels scaled x20
    offline: bool = False       # weights arrive as fp8 payload + e8m0 scales
    zipf_s: float = 0.0         # >0: skewed routing, expert share ~ rank^-s
    n_empty: int = 0            # experts forced to receive no token (skewed case)

    @property
    def M(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "LayerShape":
        return replace(self, T=T, name=f"{self.name}_T{T}")


CONFIGS = {
    # tiny layer: T=64, H=256, E=8, top-2, I=128
    "tiny": LayerShape("tiny", T=64, H=256, E=8, k=2, I=128, seed=0, gate_std=0.05),
    # Qwen3-30B-A3B-shaped layer, decode (32 tokens)
    "qwen3_30b_decode": LayerShape("qwen3_30b_decode", T=32, H=2048, E=128, k=8, I=768,
                                   seed=2, outlier_frac=0.01),
    # Qwen3-30B-A3B-shaped layer, 16K-token prefill
    "qwen3_30b_prefill": LayerShape("qwen3_30b_prefill", T=16384, H=2048, E=128, k=8, I=768,
                                    seed=3, outlier_frac=0.01),
    # Qwen3-235B-A22B-shaped layer, 8K-token prefill, offline fp8 + e8m0 weights
    "qwen3_235b_prefill": LayerShape("qwen3_235b_prefill", T=8192, H=4096, E=128, k=8, I=1536,
                                     seed=4, offline=True),
    # skewed load: Qwen3-30B-A3B shape, Zipf(1.2) expert popularity, 4 empty experts
    "qwen3_30b_skewed": LayerShape("qwen3_30b_skewed", T=16384, H=2048, E=128, k=8, I=768,
                                   seed=5, outlier_frac=0.01, zipf_s=1.2, n_empty=4),
}
SKEW_SWEEP_T = (1, 8, 128, 1024, 4096, 16384)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_hidden(shape: LayerShape, device="cpu") -> torch.Tensor:
    """Hidden states bf16 [T, H] ~ N(0,1); an outlier set of channels x20."""
    g = _gen(device, shape.seed * 1000 + 1)
    x = torch.randn(shape.T, shape.H, generator=g, device=device, dtype=torch.float32)
    n_out = round(shape.outlier_frac * shape.H)
    if n_out:
        ch = torch.randperm(shape.H, generator=g, device=device)[:n_out]
        x[:, ch] *= 20.0
    return x.to(torch.bfloat16)


def make_logits(shape: LayerShape, x: torch.Tensor, device="cpu") -> torch.Tensor:
    """Router logits fp32 [T, E].

    Default: the upstream gate projection fp32(x) @ fp32(gate), gate bf16
    [H, E] ~ N(0, gate_std).  Skewed case: Gumbel-perturbed log-popularities,
    log p_e + G with p_e ~ rank^-s over the non-empty experts (ranks mapped to
    experts by a seeded permutation); taking the top k of those is sampling k
    distinct experts by popularity.  The empty experts get logit -1e4.
    """
    g = _gen(device, shape.seed * 1000 + 2)
    if shape.zipf_s > 0:
        E = shape.E
        perm = torch.randperm(E, generator=g, device=device)
        n_live = E - shape.n_empty
        ranks = torch.arange(1, n_live + 1, device=device, dtype=torch.float64)
        logp_live = -shape.zipf_s * torch.log(ranks)
        logp = torch.full((E,), -1.0e4, device=device, dtype=torch.float64)
        logp[perm[:n_live]] = logp_live
        u = torch.rand(shape.T, E, generator=g, device=device, dtype=torch.float64)
        u = u.clamp_(1e-300, 1.0 - 1e-16)
        gumbel = -torch.log(-torch.log(u))
        return (logp[None, :] + gumbel).to(torch.float32)
    gate = _draw_gate(shape, g, device)
    return x.float() @ gate.float()


def _draw_gate(shape: LayerShape, g, device):
    return (torch.randn(shape.H, shape.E, generator=g, device=device, dtype=torch.float32)
            * shape.gate_std).to(torch.bfloat16)


def make_gate(shape: LayerShape, device="cpu") -> torch.Tensor:
    """The router gate bf16 [E, H] (out_features, in_features) whose product
    with the hidden states gives ``make_logits`` (the same seeded draw)."""
    if shape.zipf_s > 0:
        raise ValueError("the skewed-load shape draws its logits directly (no gate)")
    g = _gen(device, shape.seed * 1000 + 2)
    return _draw_gate(shape, g, device).t().contiguous()


def make_weights_bf16(shape: LayerShape, device="cpu"):
    """Expert weights bf16: w13 [E, 2I, H] (gate rows, then up rows), w2 [E, H, I]."""
    g = _gen(device, shape.seed * 1000 + 3)
    w13 = (torch.randn(shape.E, 2 * shape.I, shape.H, generator=g, device=device) * 0.02)
    w13 = w13.to(torch.bfloat16)
    w2 = (torch.randn(shape.E, shape.H, shape.I, generator=g, device=device) * 0.02)
    w2 = w2.to(torch.bfloat16)
    return w13, w2


def make_weights_offline(shape: LayerShape, device="cpu"):
    """A synthetic pre-quantized checkpoint: e4m3 payload + e8m0 scale bytes.

    Payload: N(0, 64^2) samples cast by torch to float8_e4m3fn (clamped to the
    finite range first) -- a library conversion used here only to draw
    realistic codes.  Scales: one byte per 32 K-elements, uniform in
    [113, 116], so the decoded weights have the N(0, ~0.02) magnitude of the
    online case.  Layout [E, N, K] payload, [E, N, K/32] scales (the
    [E, N, K/64, 2] pair-split view has the same bytes).
    """
    g = _gen(device, shape.seed * 1000 + 4)

    def one(N, K):
        v = torch.randn(shape.E, N, K, generator=g, device=device) * 64.0
        q = v.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        s = torch.randint(113, 117, (shape.E, N, math.ceil(K / 32)), generator=g,
                          device=device, dtype=torch.int32).to(torch.uint8)
        return q.contiguous(), s.contiguous()

    w13q, w13s = one(2 * shape.I, shape.H)
    w2q, w2s = one(shape.H, shape.I)
    return w13q, w13s, w2q, w2s


def make_layer(shape: LayerShape, device="cpu", weights=True) -> dict:
    """All inputs of one layer call as a dict of tensors on ``device``."""
    x = make_hidden(shape, device)
    out = dict(x=x, logits=make_logits(shape, x, device))
    if weights:
        if shape.offline:
            out["w13q"], out["w13s"], out["w2q"], out["w2s"] = make_weights_offline(shape, device)
        else:
            out["w13"], out["w2"] = make_weights_bf16(shape, device)
    return out


# ---------------------------------------------------------------------------
# dense linear layers
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class LinearShape:
    name: str
    M: int            # tokens
    N: int            # out_features
    K: int            # in_features (the contraction)
    seed: int
    w_std: float = 0.02


# Shapes of the dense layers the pages name: Qwen3-8B (the offline W8A8
# MXFP8 checkpoint of "Quantization on Ascend") and the Qwen3-VL vision MLP
# (sglang PR #32266: in_features 4304 gives 135 scales, a partial last block;
# its transpose has out_features 4304, a ragged last 128-row block).
LINEAR_CONFIGS = {
    "linear_tiny": LinearShape("linear_tiny", M=200, N=400, K=336, seed=20),
    "qwen3vl_vision_fc1": LinearShape("qwen3vl_vision_fc1", M=16384, N=4304, K=1152, seed=21),
    "qwen3vl_vision_fc2": LinearShape("qwen3vl_vision_fc2", M=16384, N=1152, K=4304, seed=22),
    "qwen3_8b_down_prefill": LinearShape("qwen3_8b_down_prefill", M=8192, N=4096, K=12288,
                                         seed=23),
    "qwen3_8b_gate_up_prefill": LinearShape("qwen3_8b_gate_up_prefill", M=8192, N=24576,
                                            K=4096, seed=24),
    "qwen3_8b_down_decode": LinearShape("qwen3_8b_down_decode", M=32, N=4096, K=12288, seed=25),
}


def make_linear(shape: LinearShape, device="cpu"):
    """(x bf16 [M, K] ~ N(0, 1), w bf16 [N, K] ~ N(0, w_std))."""
    g = _gen(device, shape.seed * 1000 + 5)
    x = torch.randn(shape.M, shape.K, generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn(shape.N, shape.K, generator=g, device=device) * shape.w_std)
    return x, w.to(torch.bfloat16)
