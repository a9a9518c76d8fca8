/*
 * mxmoe.h -- C ABI of the MXFP8 (OCP MX, W8A8) block-scaled fused-MoE
 * expert forward for NVIDIA GB300 (sm_103a).
 *
 * The forward, as "Quantization on Ascend" (sglang docs, section "MXFP8 for
 * LLM MoE models", implementation notes "Forward", "Online path", "Offline
 * path") and sglang PR #32266 (commit note adding the fused experts kernel:
 * routing -> act quant -> swiglu_quant -> grouped_matmul -> finalize_routing)
 * describe it:
 *
 *   moe_route_quant_mxfp8           top-k routing + expert permutation with the
 *                                   per-token MX activation quant fused in
 *                                   (init_routing quant_mode=3)
 *   grouped_gemm_swiglu_quant_mxfp8 grouped GEMM over w13 (gate+up) + SwiGLU +
 *                                   MXFP8 requant (payload + block scale)
 *   grouped_gemm_mxfp8              grouped GEMM over w2, bf16 output
 *   moe_finalize_routing            weighted top-k combine back to token order
 *   moe_forward_mxfp8               the four above on one stream
 *   mx_quantize_3d                  load-time MX quant of [E, N, K] weights
 *   mx_quantize_fp4_3d, moe_forward_w4a8_mma_scales
 *                                   the W4A8 variant: MXFP4 (packed e2m1)
 *                                   expert weights x MXFP8 activations
 *   moe_forward_w4a4_mma_scales     the W4A4 variant: MXFP4 weights and MXFP4
 *                                   expert inputs
 *   mxfp8_linear, mxfp8_linear_mma_scales
 *                                   the dense MXFP8 linear (one group of the
 *                                   grouped GEMM), any K % 16 == 0
 *   mxfp4_linear, mxfp4_linear_mma_scales
 *                                   the W4A4 dense linear
 *   moe_router_gate_topk            the router gate GEMM fused with softmax top-k
 *   moe_forward_mxfp8_gated_mma_scales
 *                                   the layer from hidden states + router gate
 *   mx_dequantize_bf16_2d           load-time dequant of an MXFP8 router gate
 *
 * Formats.  An MX block is 32 consecutive elements along the contraction
 * axis K.  Payload: one float8_e4m3fn byte per element.  Scale: one UE8M0
 * (e8m0) byte per block, value 2^(byte - 127), chosen as
 * floor(log2(block amax)) - 8 clamped to [-127, 127] (all-zero block -> 0);
 * elements round to nearest-even and saturate at +-448 (OCP MX v1.0).
 * Scales are stored [rows, K/32] row-major; for K % 64 == 0 these are the
 * same bytes as the pair-split [rows, K/64, 2] view the pages use.
 *
 * Conventions (all entry points):
 *   - Every data pointer is a DEVICE pointer owned by the caller; the
 *     library never allocates, frees or keeps device memory it was given.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work
 *     is enqueued asynchronously on it; no call synchronizes the host.
 *   - Arguments are validated before anything is launched; on a non-OK
 *     status nothing was enqueued.  Pointers must be 16-byte aligned.
 *   - Kernels that wait on on-chip barriers give every wait a time limit;
 *     when one runs out the kernel records MXMOE_ERR_DEVICE_TIMEOUT in a
 *     device status word and returns.  mxmoe_get_device_status() reads it.
 *   - Not thread-safe across concurrent calls that share output buffers.
 */
#ifndef MXMOE_H_
#define MXMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXMOE_OK = 0,
  MXMOE_ERR_NULL = 1,            /* a required pointer is NULL              */
  MXMOE_ERR_ALIGN = 2,           /* a pointer is not 16-byte aligned        */
  MXMOE_ERR_SHAPE = 3,           /* a size is out of range or inconsistent  */
  MXMOE_ERR_UNSUPPORTED = 4,     /* valid but not supported by this build   */
  MXMOE_ERR_WORKSPACE = 5,       /* workspace missing or too small          */
  MXMOE_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed    */
  MXMOE_ERR_DEVICE_TIMEOUT = 7,  /* a device-side wait ran out of time      */
  MXMOE_ERR_DEVICE_CHECK = 8     /* a device-side consistency check failed  */
} mxmoe_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* mxmoe_status_string(mxmoe_status status);

/*
 * Load-time MX quantization of a 3D weight tensor (also any 2D tensor with
 * E = 1).  "Quantization on Ascend", MoE MXFP8 online path: bf16 expert
 * weights are quantized once at load, a 3D [E, N, K] input accepted directly.
 *
 *   w      bf16 [E, N, K] row-major (K contiguous)
 *   q      e4m3 [E, N, K]            (output)
 *   scale  e8m0 [E, N, ceil(K/32)]   (output)
 * Requires K % 16 == 0.  With K % 32 == 16 each row ends in a partial block
 * of 16 elements whose scale is taken over the elements that exist (sglang
 * PR #32266 summary, "Offline partial MXFP8 block-scale layout": ceil(K/32)
 * scales per row, e.g. 135 for K = 4304).  Empty (E*N == 0) is a no-op.
 */
mxmoe_status mx_quantize_3d(const uint16_t* w, int64_t E, int64_t N, int64_t K,
                            uint8_t* q, uint8_t* scale, void* stream);

/*
 * Load-time MXFP4 quantization (W4A8 weights, online path of the W4A8 notes:
 * bf16 weights -> MXFP4 at load): per 32-element block along K, scale byte
 * b = clamp(floor(log2 amax) - 2, -127, 127) + 127 (2 = the largest
 * power-of-two exponent of e2m1), elements e2m1 round-to-nearest-even,
 * saturating at +-6, packed two per byte (element 2i in the low nibble).
 *   w bf16 [E, N, K]; q uint8 [E, N, K/2]; scale uint8 [E, N, K/32].
 *   K % 32 == 0; w, q 16-byte aligned.
 */
mxmoe_status mx_quantize_fp4_3d(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint8_t* q,
                                uint8_t* scale, void* stream);

/*
 * Workspace bytes moe_route_quant_mxfp8 / moe_route_permute_bf16 need for
 * T tokens and E experts (per-block expert histograms).
 */
size_t moe_route_quant_mxfp8_workspace_size(int T, int E);

/*
 * Top-k routing with the per-token MX activation quant fused into the expert
 * permutation: init_routing with quant_mode=3 ("Quantization on Ascend",
 * MoE MXFP8 "Forward" note; PR #32266 commit note on quant_mode=3, whose
 * output is byte-identical to routing followed by a separate quant pass).
 *
 *   x              bf16 [T, H] hidden states
 *   logits         fp32 [T, E] router logits
 *   renormalize    nonzero: the k softmax weights are divided by their sum
 *   xq             e4m3 [M, H], M = T*k   expanded rows, grouped by expert
 *   xs             e8m0 [M, H/32]
 *   topk_ids       int32 [T, k]   experts of each token, descending logit,
 *                                 ties to the lower expert id
 *   topk_w         fp32 [T, k]    routing weights (softmax, optionally renormed)
 *   sorted_to_src  int32 [M]      expanded row p holds flat assignment
 *                                 sorted_to_src[p] = t*k + j (token t = /k)
 *   src_to_sorted  int32 [M]      inverse permutation
 *   expert_counts  int64 [E]      rows per expert (the COUNT group list)
 *   expert_offsets int64 [E+1]    exclusive prefix of counts, offsets[E] = M
 *                                 (the CUMULATIVE group list, leading 0)
 * Rows of one expert are in flat-index order (deterministic).
 * Requires 1 <= k <= min(E, 32), E <= 1024, H % 32 == 0, T >= 0.
 * T == 0 writes only counts/offsets (all zero).
 */
mxmoe_status moe_route_quant_mxfp8(const uint16_t* x, const float* logits, int T, int H,
                                   int E, int k, int renormalize, uint8_t* xq, uint8_t* xs,
                                   int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                                   int32_t* src_to_sorted, int64_t* expert_counts,
                                   int64_t* expert_offsets, void* ws, size_t ws_bytes,
                                   void* stream);

/*
 * moe_route_quant_mxfp8 for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point; it exists for callers
 * such as serving runtimes that pre-partition all device memory into their
 * own pool and forbid cudaMalloc while serving (an allocation there can
 * synchronize the device and fragments the pool), or plug-ins whose host
 * framework owns device memory and offers no workspace hook.
 *
 * Same arguments, results and layouts as moe_route_quant_mxfp8, minus the
 * workspace: the routing scratch (per-block expert histograms and their
 * scanned block bases) lives in a 2 MiB array inside the library that
 * every GPU loading the library keeps until the process exits.  Inputs and
 * outputs remain the caller's.
 *   - Limit: ceil(T / 64) * E <= 262144 (e.g. T = 131072 tokens at E = 128);
 *     larger calls return MXMOE_ERR_WORKSPACE and launch nothing.
 *   - The call allocates nothing (no cudaMalloc / cudaFree, no allocating
 *     library routine).  Its first call on a device looks up the array's
 *     device address with that device current; make that first call before
 *     any stream capture.  The address is kept per device and CUDA context:
 *     after cudaDeviceReset the next call (the first in the new context)
 *     looks it up again, and the array's contents start over.
 *   - Every call shares the one array.  Each call writes every scratch entry
 *     before it reads it, so nothing has to start at zero, but calls that
 *     overlap on the GPU (other streams, other threads) race on it.
 */
mxmoe_status moe_route_quant_mxfp8_noalloc(const uint16_t* x, const float* logits, int T, int H,
                                           int E, int k, int renormalize, uint8_t* xq,
                                           uint8_t* xs, int32_t* topk_ids, float* topk_w,
                                           int32_t* sorted_to_src, int32_t* src_to_sorted,
                                           int64_t* expert_counts, int64_t* expert_offsets,
                                           void* stream);

/*
 * The two-step comparator of moe_route_quant_mxfp8: the same routing and
 * permutation, but the expanded rows are written as bf16 (init_routing
 * without quant); a separate mx_quantize_3d(xp, 1, M, H) pass then gives the
 * same bytes as the fused call.  Arguments as above, xp bf16 [M, H].
 */
mxmoe_status moe_route_permute_bf16(const uint16_t* x, const float* logits, int T, int H,
                                    int E, int k, int renormalize, uint16_t* xp,
                                    int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                                    int32_t* src_to_sorted, int64_t* expert_counts,
                                    int64_t* expert_offsets, void* ws, size_t ws_bytes,
                                    void* stream);

/*
 * gmm1: grouped GEMM over w13 fused with SwiGLU and the MXFP8 requant
 * (PR #30768 report, GroupedMatmulSwigluQuant: returns quantized activations
 * and their block scale; "Quantization on Ascend": gmm1 fuses gate/up +
 * swiglu + requant and takes the cumulative group list).
 *
 * For expert e and rows r in [offsets[e], offsets[e+1]):
 *   h   = deq(xq[r]) . deq(w13[e])^T          fp32 accumulate, [2I]
 *   a   = silu(h[0:I]) * h[I:2I]              gate rows first, then up
 *   aq[r], as[r] = MX-quant(a) along I
 *
 *   xq, xs          e4m3 [M, H], e8m0 [M, H/32]
 *   w13q, w13s      e4m3 [E, 2I, H], e8m0 [E, 2I, H/32]
 *   expert_offsets  int64 [E+1] on the device, offsets[E] == M
 *   aq, as          e4m3 [M, I], e8m0 [M, I/32]   (outputs; aq 32-byte aligned)
 * Requires H % 128 == 0, I % 128 == 0, 1 <= E <= 256, M >= 0.
 */
mxmoe_status grouped_gemm_swiglu_quant_mxfp8(const uint8_t* xq, const uint8_t* xs,
                                             const uint8_t* w13q, const uint8_t* w13s,
                                             const int64_t* expert_offsets, int64_t M, int E,
                                             int H, int I, uint8_t* aq, uint8_t* as,
                                             void* stream);

/*
 * gmm2: grouped GEMM over w2 ("Quantization on Ascend", MoE MXFP8 "Forward":
 * npu_grouped_matmul with the count group list; the offsets here carry the
 * same information in cumulative form).
 *
 *   y[r] = deq(aq[r]) . deq(w2[e])^T, fp32 accumulate, rounded to bf16
 *
 *   aq, as      e4m3 [M, I], e8m0 [M, I/32]
 *   w2q, w2s    e4m3 [E, H, I], e8m0 [E, H, I/32]
 *   y           bf16 [M, H]   (output, 32-byte aligned)
 * Requires I % 128 == 0, H % 128 == 0, 1 <= E <= 256, M >= 0.
 */
mxmoe_status grouped_gemm_mxfp8(const uint8_t* aq, const uint8_t* as, const uint8_t* w2q,
                                const uint8_t* w2s, const int64_t* expert_offsets, int64_t M,
                                int E, int I, int H, uint16_t* y, void* stream);

/*
 * Finalize routing: weighted top-k combine back to token order
 * ("Quantization on Ascend", MoE layers use init_routing / finalize_routing;
 * PR #32266 fused experts note).
 *
 *   out[t] = sum_{j<k} topk_w[t, j] * y[src_to_sorted[t*k + j]]
 *
 * fp32 accumulation in slot order j = 0..k-1, rounded once to bf16.
 *   y bf16 [M, H], topk_w fp32 [T, k], src_to_sorted int32 [T*k],
 *   out bf16 [T, H].  Requires H % 8 == 0, 1 <= k <= 32.
 */
mxmoe_status moe_finalize_routing(const uint16_t* y, const float* topk_w,
                                  const int32_t* src_to_sorted, int T, int k, int H,
                                  uint16_t* out, void* stream);

/* Workspace bytes moe_forward_mxfp8 needs (all intermediates of the layer). */
size_t moe_forward_mxfp8_workspace_size(int T, int H, int E, int k, int I);

/*
 * The whole MXFP8 expert forward on one stream: route+quant, gmm1 (+SwiGLU
 * +requant), gmm2, finalize.  Weights are the MX-quantized w13 [E, 2I, H]
 * and w2 [E, H, I] with their [.., K/32] scales (from mx_quantize_3d, or an
 * offline checkpoint's float8_e4m3fn payload + uint8 e8m0 scales).
 *   out bf16 [T, H].  ws: moe_forward_mxfp8_workspace_size() bytes, 256-byte
 *   aligned; it holds every intermediate and may be reused between calls.
 *   Inside the call the activation scales and a copy of the weight scales
 *   live in the MMA layout (see mx_scales_to_mma_layout).
 */
mxmoe_status moe_forward_mxfp8(const uint16_t* x, const float* logits, const uint8_t* w13q,
                               const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                               int T, int H, int E, int k, int I, int renormalize,
                               uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Load-time re-layout of weight scales into the tensor-core ("MMA") layout
 * that moe_forward_mxfp8_mma_scales consumes.  Not an operation of the
 * pages (their FRACTAL_NZ re-tiling plays the same role for Ascend): the
 * GB300 tensor cores read each 128-row x 128-K block's 512 scale bytes as
 * one chunk, byte (r % 32) * 16 + (r / 32) * 4 + kb for row r of the block
 * and 32-element block kb, chunks ordered (row block, K slice).
 *   scale  e8m0 [E, N, ceil(K/32)]  ->  out  e8m0, E * ceil(N/128) *
 *          ceil(K/128) * 512 bytes (the same size when N, K % 128 == 0)
 * Requires K % 16 == 0; N % 128 == 0 when E > 1.  Slots past the data (the
 * last K slice when K % 128 != 0, the rows of a ragged last row block when
 * E == 1) are written as 127 (scale 1; the GEMMs read zero payload there).
 */
mxmoe_status mx_scales_to_mma_layout(const uint8_t* scale, int64_t E, int64_t N, int64_t K,
                                     uint8_t* out, void* stream);

/*
 * Router gate GEMM fused with softmax top-k (the step upstream of the
 * routing; "Quantization on Ascend", MoE MXFP8 notes: the router gate is a
 * ReplicatedLinear kept in bf16 on the online path and dequantized on the
 * offline path, see mx_dequantize_bf16_2d):
 *   logits[t, e] = sum_h x[t, h] * gate[e, h]      tensor cores, fp32 accumulate
 *   topk_ids[t, :], topk_w[t, :] = top-k softmax of logits[t, :], the rule of
 *   moe_route_quant_mxfp8 (ties to the lower id, descending; renormalize
 *   divides by the k weights' sum); on the same fp32 logits both give the same
 *   bytes.
 *   x bf16 [T, H], gate bf16 [E, H] (16-byte aligned); logits_out fp32 [T, E]
 *   (NULL: not written); topk_ids int32 [T, k], topk_w fp32 [T, k].
 * Requires H % 64 == 0, 1 <= E <= 256, 1 <= k <= min(32, E).
 */
mxmoe_status moe_router_gate_topk(const uint16_t* x, const uint16_t* gate, int T, int H, int E,
                                  int k, int renormalize, float* logits_out, int32_t* topk_ids,
                                  float* topk_w, void* stream);

/*
 * The MXFP8 layer from the hidden states and the bf16 router gate: the gate
 * GEMM and softmax top-k run fused (moe_router_gate_topk's kernel, which also
 * leaves the routing step's ranks and histograms), then the layer as
 * moe_forward_mxfp8_mma_scales.  Arguments as that call with `gate` bf16
 * [E, H] in place of the logits.
 */
mxmoe_status moe_forward_mxfp8_gated_mma_scales(const uint16_t* x, const uint16_t* gate,
                                                const uint8_t* w13q, const uint8_t* w13s_mma,
                                                const uint8_t* w2q, const uint8_t* w2s_mma, int T,
                                                int H, int E, int k, int I, int renormalize,
                                                uint16_t* out, void* ws, size_t ws_bytes,
                                                void* stream);

/*
 * Load-time dequant of an MXFP8 tensor to bf16 (the offline router gate: a
 * quantized gate used without its block scale scrambles the routing, PR
 * #32266 router-gate note): out[r, j] = bf16(dec(q[r, j]) * 2^(s[r, j/32] -
 * 127)), exact for every value in bf16's range.
 *   q e4m3 [rows, K], scale e8m0 [rows, K/32], out bf16 [rows, K]; K % 32 == 0.
 */
mxmoe_status mx_dequantize_bf16_2d(const uint8_t* q, const uint8_t* scale, int64_t rows,
                                   int64_t K, uint16_t* out, void* stream);

/*
 * Dense MXFP8 linear ("Quantization on Ascend", MXFP8 implementation notes,
 * online path: weights quantized once at load along K, activations
 * quantized per token at inference, then a block-scaled matmul with one
 * e8m0 scale per 32 elements of K; that is one group of the grouped GEMM):
 *
 *   out[m, n] = bf16( sum_k deq(xq)[m, k] * deq(wq)[n, k] )   fp32 accumulate
 *   xq, xs    = MX-quant(x) along K (the rule of mx_quantize_3d)
 *
 *   x      bf16 [M, K] row-major, 16-byte aligned
 *   wq     e4m3 [N, K] (K contiguous: the storage of the pages' pre-transposed
 *          [in, out] view), 16-byte aligned, from mx_quantize_3d(w, 1, N, K)
 *          or an offline checkpoint
 *   ws     e8m0 [N, ceil(K/32)] (mxfp8_linear) or its MMA layout from
 *          mx_scales_to_mma_layout(ws, 1, N, K) (mxfp8_linear_mma_scales,
 *          16-byte aligned)
 *   out    bf16 [M, N], 32-byte aligned
 *   workspace  mxfp8_linear_workspace_size(M, N, K) bytes, 256-byte aligned,
 *          sized for the current device; it holds xq, the activation scales,
 *          (mxfp8_linear only) the re-laid weight scales and, when M is too
 *          small to fill the GPU with tiles, the split-K partial sums (each
 *          tile's K slices split over idle SMs, fp32 partials added in a fixed
 *          order and rounded once to bf16).
 * Requires K % 16 == 0 (K % 32 == 16 gives each row a partial last block of
 * 16, PR #32266 summary, "Offline partial MXFP8 block-scale layout") and
 * N % 16 == 0; 0 <= M < 2^31.  M == 0 is a no-op.
 */
size_t mxfp8_linear_workspace_size(int64_t M, int64_t N, int64_t K);
mxmoe_status mxfp8_linear(const uint16_t* x, const uint8_t* wq, const uint8_t* ws, int64_t M,
                          int64_t N, int64_t K, uint16_t* out, void* workspace, size_t ws_bytes,
                          void* stream);
mxmoe_status mxfp8_linear_mma_scales(const uint16_t* x, const uint8_t* wq, const uint8_t* ws_mma,
                                     int64_t M, int64_t N, int64_t K, uint16_t* out,
                                     void* workspace, size_t ws_bytes, void* stream);

/*
 * W4A4 dense linear ("Quantization on Ascend", W4A4 notes, offline
 * single-level path: both matmul inputs packed float4_e2m1fn_x2 with one
 * UE8M0 scale per 32 elements of K, group sizes [1, 1, 32]): the activations
 * are MXFP4-quantized per token (the rule of mx_quantize_fp4_3d), then
 *   out[m, n] = bf16( sum_k deq(xp)[m, k] * deq(wp)[n, k] )   fp32 accumulate
 *   wp     packed e2m1 [N, K/2] from mx_quantize_fp4_3d(w, 1, N, K), 32-byte
 *          aligned; ws e8m0 [N, K/32] (mxfp4_linear) or its MMA layout
 *          (mxfp4_linear_mma_scales, 16-byte aligned)
 *   x, out, workspace as mxfp8_linear (mxfp8_linear_workspace_size bytes).
 * Requires K % 128 == 0 (each 256-element k-slice of the packed e2m1 x e2m1
 * GEMM holds one or two whole 128-element scale chunks) and N % 16 == 0.
 */
mxmoe_status mxfp4_linear(const uint16_t* x, const uint8_t* wp, const uint8_t* ws, int64_t M,
                          int64_t N, int64_t K, uint16_t* out, void* workspace, size_t ws_bytes,
                          void* stream);
mxmoe_status mxfp4_linear_mma_scales(const uint16_t* x, const uint8_t* wp, const uint8_t* ws_mma,
                                     int64_t M, int64_t N, int64_t K, uint16_t* out,
                                     void* workspace, size_t ws_bytes, void* stream);

/*
 * moe_forward_mxfp8 with the weight scales already in the MMA layout
 * (mx_scales_to_mma_layout, done once at load); saves re-laying them out on
 * every call.  All other arguments and results as moe_forward_mxfp8.
 */
mxmoe_status moe_forward_mxfp8_mma_scales(const uint16_t* x, const float* logits,
                                          const uint8_t* w13q, const uint8_t* w13s_mma,
                                          const uint8_t* w2q, const uint8_t* w2s_mma, int T,
                                          int H, int E, int k, int I, int renormalize,
                                          uint16_t* out, void* ws, size_t ws_bytes,
                                          void* stream);

/*
 * W4A8: the same layer with MXFP4 expert weights ("Quantization on Ascend",
 * W4A8 notes: packed FP4 float4_e2m1fn_x2, two nibbles per byte, UE8M0 scale
 * per 32-element block; activations per-token MXFP8; the path measured in
 * sglang PR #40519).  Routing, the fused activation quant, the SwiGLU +
 * requant epilogue and finalize are those of the MXFP8 layer; the grouped
 * GEMMs run tcgen05 block-scaled MMAs with e4m3 activations x e2m1 weights.
 *   w13p uint8 [E, 2I, H/2], w2p uint8 [E, H, I/2]: packed e2m1, element 2i
 *     in the low nibble of byte i (mx_quantize_fp4_3d); 32-byte aligned.
 *   w13s_mma, w2s_mma: their scales in the MMA layout (mx_scales_to_mma_layout).
 * Workspace: moe_forward_mxfp8_workspace_size(T, H, E, k, I).
 */
mxmoe_status moe_forward_w4a8_mma_scales(const uint16_t* x, const float* logits,
                                         const uint8_t* w13p, const uint8_t* w13s_mma,
                                         const uint8_t* w2p, const uint8_t* w2s_mma, int T, int H,
                                         int E, int k, int I, int renormalize, uint16_t* out,
                                         void* ws, size_t ws_bytes, void* stream);

/*
 * W4A4: MXFP4 expert weights and MXFP4 expert inputs ("Quantization on
 * Ascend", W4A4 MoE notes: packed MXFP4 w13 / w2 with UE8M0 block-32 scales;
 * each expert input is quantized to MXFP4 right before the grouped matmul).
 * The routing step quantizes the permuted hidden states to MXFP4 (scale byte
 * clamp(floor(log2 amax) - 2, -127, 127) + 127, e2m1 round-to-nearest-even
 * saturating at +-6, element 2i in the low nibble of byte i); gmm1's epilogue
 * requantizes the SwiGLU output (rounded to fp32) to MXFP4 by the same rule;
 * both grouped GEMMs run e2m1 x e2m1 block-scaled tcgen05 MMAs on packed
 * operands (kind::mxf4, K = 64 per instruction).  Arguments, weights and workspace as
 * moe_forward_w4a8_mma_scales.
 */
mxmoe_status moe_forward_w4a4_mma_scales(const uint16_t* x, const float* logits,
                                         const uint8_t* w13p, const uint8_t* w13s_mma,
                                         const uint8_t* w2p, const uint8_t* w2s_mma, int T, int H,
                                         int E, int k, int I, int renormalize, uint16_t* out,
                                         void* ws, size_t ws_bytes, void* stream);

/*
 * The layer on HOST buffers, with the host<->device copies overlapped with
 * compute: the tokens are processed in chunks through three library-owned
 * streams (copy in, compute, copy out) and two device staging slots in ws, so
 * chunk c's layer runs while chunk c+1's inputs arrive and chunk c-1's output
 * leaves.  n_chunks > 0: that many near-equal chunks.  n_chunks <= 0: the
 * default plan (one chunk up to 4096 tokens; else three chunks, the first and
 * last of 3/16 of the tokens each, which shortens the unoverlapped first
 * copy-in and last copy-out while every chunk re-reads the weights).  Weight scales in
 * the MMA layout (mx_scales_to_mma_layout); weights stay on the device.
 *   x_host bf16 [T, H], logits_host fp32 [T, E], out_host bf16 [T, H]: host
 *   memory (pinned, e.g. cudaHostAlloc, for the copies to overlap).
 *   ws: moe_forward_mxfp8_host_workspace_size(...) bytes of device memory.
 * The work is ordered after the caller's prior work on `stream`, and `stream`
 * waits for the whole call (out_host is complete once `stream` is).
 */
size_t moe_forward_mxfp8_host_workspace_size(int T, int H, int E, int k, int I, int n_chunks);
mxmoe_status moe_forward_mxfp8_host(const uint16_t* x_host, const float* logits_host,
                                    const uint8_t* w13q, const uint8_t* w13s_mma,
                                    const uint8_t* w2q, const uint8_t* w2s_mma, int T, int H,
                                    int E, int k, int I, int renormalize, uint16_t* out_host,
                                    int n_chunks, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward_mxfp8_host with an explicit chunk plan: chunk_tokens[0..n_chunks)
 * (host array, positive, summing to T; n_chunks <= 1024).  The workspace is
 * moe_forward_mxfp8_host_workspace_size(max chunk, H, E, k, I, 1) bytes.
 */
mxmoe_status moe_forward_mxfp8_host_plan(const uint16_t* x_host, const float* logits_host,
                                         const uint8_t* w13q, const uint8_t* w13s_mma,
                                         const uint8_t* w2q, const uint8_t* w2s_mma, int T, int H,
                                         int E, int k, int I, int renormalize, uint16_t* out_host,
                                         const int32_t* chunk_tokens, int n_chunks, void* ws,
                                         size_t ws_bytes, void* stream);

/*
 * Per-kernel timing of moe_forward_mxfp8 / moe_forward_mxfp8_mma_scales / mxfp8_linear*
 * (instrumentation, off by default; not part of the method).  enable = 1:
 * each layer call records CUDA events on its stream between its kernels;
 * mxmoe_layer_profile_read then returns, for the last such call on the
 * current device, n <= 5 segment times in milliseconds:
 *   [0] weight-scale re-layout (0 for the _mma_scales entry point),
 *   [1] route + fused quant, [2] gmm1, [3] gmm2, [4] finalize.
 * A dense-linear call (mxfp8_linear*) records [0] weight-scale re-layout,
 * [1] activation quant, [2] GEMM, and 0 for [3], [4].
 * enable = 2: events only around gmm1 (the dense linear's GEMM), so the other
 * kernel boundaries keep their overlapped (programmatic dependent) launches;
 * the read returns [2] and 0 elsewhere.  enable = 0: off.  Other values:
 * MXMOE_ERR_SHAPE.  The read synchronizes on the call's last event.  Not
 * thread-safe.
 */
mxmoe_status mxmoe_layer_profile_enable(int enable);
mxmoe_status mxmoe_layer_profile_read(float* ms, int n);

/*
 * Device status word of the current device: 0 or the first error a kernel
 * recorded (MXMOE_ERR_DEVICE_TIMEOUT / MXMOE_ERR_DEVICE_CHECK).  Synchronizes
 * the device.  clear != 0 resets the word to 0 afterwards.
 */
mxmoe_status mxmoe_get_device_status(int32_t* status_out, int clear);

/*
 * Time limit, in SM clock cycles, of every bounded device-side wait that a
 * kernel launched afterwards uses (default about 2^32 cycles, ~2 s).
 * Values < 1 restore the default.  Meant for tests of the timeout path.
 */
void mxmoe_set_wait_limit_cycles(long long cycles);

/*
 * Grouped-GEMM kernel selection (not part of the method; process-wide).
 * Both kernels give the same bytes.  mode 0: every grouped GEMM runs the 1-SM
 * kernel.  mode 1: 256-wide tiles with MMA-layout scales (the layer calls)
 * run the 2-SM kernel (tcgen05 cta_group::2 over CTA pairs) when the device
 * can co-schedule pairs.  mode 2 (the default): the 2-SM kernel for the
 * bf16-output GEMM (grouped GEMM2) when its rows average at least 512 per
 * expert (M >= 512 * E) and for the SwiGLU GEMM (grouped GEMM1) when they
 * average at least 1024 (M >= 1024 * E), the 1-SM kernel otherwise.  Other
 * values select mode 2.
 */
void mxmoe_set_gemm_2sm(int mode);

/*
 * Small-batch grouped GEMMs (not part of the method; process-wide).  enable
 * != 0 (the default): an MXFP8 layer call whose token count is at most 32
 * (so no expert has more than 32 rows), with H % 256 == 0 and logits given,
 * runs both grouped GEMMs in one persistent kernel, gmm2's work of an expert
 * starting once that expert's gmm1 output is stored; 0: one kernel per GEMM.
 * Both give the same bytes.  With the one-kernel form the layer profile
 * (mxmoe_layer_profile_read) reports the pair's time as gmm1's and 0 for
 * gmm2.
 */
void mxmoe_set_gemm_chain(int enable);

/* Library version string. */
const char* mxmoe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXMOE_H_ */
