// Internal launchers of the MXFP8 MoE library (host side, not exported).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mxmoe {

// Routing: tokens handled by one block of the top-k / rank kernel.
constexpr int kRouteTokensPerBlock = 64;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int num_sms();                       // of the current device (cached)
// Unique id of the calling thread's current CUDA context, 0 when none is
// current yet.  Per-device caches (device addresses of the library's
// globals, kernel attributes) record it: after cudaDeviceReset the device
// gets a new primary context whose module globals and kernel attributes are
// new, and no context ever reuses an id, so a changed id means "set up again".
uint64_t context_id();
int* device_status_ptr();            // library status word on the current device
long long wait_limit_cycles();
bool use_two_sm_gemm(bool swiglu, int64_t M, int E);  // 2-SM grouped GEMM kernel?

cudaError_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                               uint8_t* scale, cudaStream_t stream);
// Any K % 16 == 0 (ceil(K/32) scales, a partial last block of 16), scales
// written in the tiled layout (KT = ceil(K/128)); offsets (nullable) <- {0, rows}.
// fp4: MXFP4 rows, q [rows, K/2] packed e2m1, K % 32 == 0.
cudaError_t launch_mx_quantize_tiled(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                                     uint8_t* scale_tiled, int64_t* offsets, cudaStream_t stream,
                                     bool fp4 = false);
// MXFP4 (packed e2m1, W4A8 weights): q [rows, K/2], scale [rows, K/32].
cudaError_t launch_mx_quantize_fp4(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                                   uint8_t* scale, cudaStream_t stream);

// Routing + permutation.  quant 1: MXFP8 xq [M, H] / xs outputs; 2: MXFP4 xq
// [M, H/2] / xs (tiled scales only); 0: bf16 xp output.  zero_e (nullable): E
// ints the routing step sets to zero (the chained GEMMs' counters).
cudaError_t launch_route(const uint16_t* x, const float* logits, int T, int H, int E, int k,
                         bool renormalize, int quant, uint8_t* xq, uint8_t* xs, uint16_t* xp,
                         int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                         int32_t* src_to_sorted, int64_t* counts, int64_t* offsets,
                         int32_t* block_hist, cudaStream_t stream,
                         int32_t* tile_base = nullptr, bool topk_done = false,
                         int32_t* zero_e = nullptr);

// Router gate GEMM (bf16 x [T, H] . bf16 gate [E, H]^T, fp32 accumulate on the
// tensor cores) fused with softmax top-k.  logits (nullable) receives the fp32
// logits.  local_rank / block_hist (both nullable) receive the routing step's
// in-block ranks and per-block expert histograms (the state launch_route's
// first kernel leaves), so launch_route can continue with topk_done.
// Requires H % 64 == 0, 1 <= E <= 256, 1 <= k <= min(32, E).
cudaError_t launch_router_gate_topk(const uint16_t* x, const uint16_t* gate, int T, int H, int E,
                                    int k, bool renormalize, float* logits, int32_t* topk_ids,
                                    float* topk_w, int32_t* local_rank, int32_t* block_hist,
                                    cudaStream_t stream);
// e4m3 [rows, K] + e8m0 [rows, K/32] -> bf16 [rows, K] (value dec(q) * 2^(s - 127)
// rounded to bf16, exact for every value in bf16's range); K % 32 == 0.
cudaError_t launch_mx_dequantize_bf16(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K,
                                      uint16_t* out, cudaStream_t stream);

size_t route_workspace_bytes(int T, int E);
// Bytes of the routing scratch's histogram part [E][nb]; the scan's block
// bases (as many bytes) follow it.
size_t route_hist_bytes(int T, int E);

// Launch with programmatic stream serialization: the kernel may begin while
// its predecessor on the stream is still running and must call pdl_wait()
// (common.cuh) before it reads anything that predecessor writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_finalize(const uint16_t* y, const float* topk_w, const int32_t* src_to_sorted,
                            int T, int k, int H, uint16_t* out, cudaStream_t stream);

// Grouped GEMMs.  Return cudaErrorInvalidValue when a tensor map can't be built.
// tiled_scales: every scale array (inputs and gmm1's output scales) is in the
// tiled layout of tiled_scales.h instead of [rows, K/32].
// group_rows_max > 0: the caller guarantees that no group has more rows (the
// layer passes its token count: a token picks an expert at most once), which
// lets small batches load only the first rows of each m-tile.
// fmt: 0 = W8A8; 1 = W4A8 (w13q / w2q packed MXFP4, e2m1 [rows, K/2]); 2 =
// W4A4 (the activations packed MXFP4 too, and gmm1's output aq [M, I/2]); 1
// and 2 require tiled_scales.
cudaError_t launch_gemm_swiglu_quant(const uint8_t* xq, const uint8_t* xs, const uint8_t* w13q,
                                     const uint8_t* w13s, const int64_t* offsets, int64_t M,
                                     int E, int H, int I, uint8_t* aq, uint8_t* as,
                                     cudaStream_t stream, bool tiled_scales = false,
                                     int fmt = 0, int64_t group_rows_max = 0);
// ksplit > 1 (E == 1, tiled scales): split-K over ksplit K ranges whose fp32
// partial sums go to partial [ksplit][M][H], then one reduce kernel rounds
// their in-order sum to bf16.
cudaError_t launch_gemm_bf16(const uint8_t* aq, const uint8_t* as, const uint8_t* w2q,
                             const uint8_t* w2s, const int64_t* offsets, int64_t M, int E,
                             int I, int H, uint16_t* y, cudaStream_t stream,
                             bool tiled_scales = false, int fmt = 0, int ksplit = 1,
                             float* partial = nullptr, int64_t group_rows_max = 0);
// Both grouped GEMMs of an MXFP8 layer (MMA-layout scales) in one persistent
// kernel, for small batches: gemm_chain_supported(group_rows_max, H, I) says
// when it applies (every group at most 32 rows, H % 256 == 0).  done: E ints of
// scratch that are zero when the kernel starts (the layer's routing kernel
// zeroes them).  Same outputs, byte for byte, as launch_gemm_swiglu_quant then
// launch_gemm_bf16.
bool gemm_chain_supported(int64_t group_rows_max, int H, int I);
cudaError_t launch_gemm_chain(const uint8_t* xq, const uint8_t* xs, const uint8_t* w13q,
                              const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                              const int64_t* offsets, int64_t M, int E, int H, int I, uint8_t* aq,
                              uint8_t* as, uint16_t* y, int* done, cudaStream_t stream,
                              int64_t group_rows_max);
// Split count the dense linear uses for an [M, K] x [N, K]^T product on the
// current device (1 when the tiles alone fill the GPU).  packed_fp4: the W4A4
// kernel, whose k-slices hold 256 K elements instead of 128 (never more splits
// than the MXFP8 count for the same shape).
int gemm_bf16_ksplit(int64_t M, int N, int K, bool packed_fp4 = false);

// [rows, ceil(K/32)] scales -> tiled layout with KT = ceil(K/128); rows and
// slots past the data (a ragged row block or K slice) are written as 127.
cudaError_t launch_scales_to_tiled(const uint8_t* scale, int64_t rows, int64_t K, uint8_t* out,
                                   cudaStream_t stream);

}  // namespace mxmoe
