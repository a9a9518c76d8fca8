"""CPU oracle for the MXFP8 block-scaled fused-MoE expert forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table
or constant generator with the CUDA library; both sides only consume the same
seeded inputs from ``mxfp8_block_scaled_moe_gb300.workloads``.

Everything is plain NumPy in float64, written step by step in the order the
method defines it, with no blocking, fusion or reordering:

* ``oracle.mx``  -- the e4m3fn element codec, the bf16 rounding of outputs,
  the UE8M0 (e8m0) block-scale rule and the MX block quantizer, plus the
  pair-split scale view and its odd-count padding.
* ``oracle.moe`` -- top-k softmax routing, the expert permutation, the fused
  route+quant, the grouped GEMM1 + SwiGLU + requant, the grouped GEMM2, the
  finalize-routing combine and the whole layer.
* ``oracle.linear`` -- the dense MXFP8 linear (per-token activation quant,
  block-scaled GEMM, bf16 out), any K % 16 == 0.

Sources (cited per function):

* "Quantization on Ascend" (sglang docs), section "MXFP8 for LLM MoE models",
  implementation notes: online 3D weight quant, offline float8_e4m3fn payload
  with uint8 e8m0 scales (exponent + 127) reshaped [E,N,K/32] -> [E,N,K/64,2],
  the init_routing quant_mode=3 forward, gmm1 (gate/up + swiglu + requant)
  with a cumulative group list and gmm2 with a count group list.
* sglang PR #30768 report ("Add W8A8 MXFP8 quantization for Qwen3 MoE on
  Ascend NPU"), sections on the implementation breakdown and the
  GroupedMatmulSwigluQuant source excerpt.
* sglang PR #32266 ("Fix offline W8A8 MXFP8 quantization for Qwen3.5 on Ascend
  NPU"), commit notes on the fused experts path, quant_mode=3 byte identity,
  the w13 gate/up order, "no zero point", and the summary section
  "Offline partial MXFP8 block-scale layout" (ceil(K/32) scales, 135 -> 136 ->
  68 pairs for K=4304).
* OCP Microscaling Formats (MX) Specification v1.0: the shared scale of a
  32-element block is 2^(floor(log2(amax)) - emax_elem) with emax_elem = 8 for
  E4M3, stored as an E8M0 exponent; elements are cast with round-to-nearest-
  even and saturation.  The pages name the formats but do not print this
  rule; it is the plainest reading consistent with them.
"""

from . import mx, moe, linear  # noqa: F401
