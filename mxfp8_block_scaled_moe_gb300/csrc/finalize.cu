// Finalize routing: weighted top-k combine of the expert outputs back to
// token order ("Quantization on Ascend": MoE layers use init_routing /
// finalize_routing; sglang PR #32266 fused experts note, last step).
//
//   out[t] = sum_{j<k} topk_w[t, j] * y[src_to_sorted[t*k + j]]
//
// fp32 accumulation in slot order, one bf16 rounding (RNE) at the end.
// One warp per token; each lane owns 8 consecutive columns (one 16 B load per
// source row).  Roofline: HBM-bound, k*H*2 B read + H*2 B written per token.
#include "common.cuh"
#include "internal.h"

namespace mxmoe {

constexpr int kFinThreads = 256;

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(
    const uint16_t* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ src_to_sorted, int T, int k, int H, uint16_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kFinThreads / 32) + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform
  int64_t my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_row = src_to_sorted[(int64_t)t * k + lane];
    my_w = topk_w[(int64_t)t * k + lane];
  }
  uint16_t* orow = out + (int64_t)t * H;
  for (int c0 = 0; c0 < H; c0 += 256) {  // warp-uniform trip count
    const int c = c0 + lane * 8;
    const bool ok = c < H;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      const float w = __shfl_sync(0xffffffffu, my_w, j);
      const uint4 v = ok ? ld_nc_v4(y + row * H + c) : make_uint4(0, 0, 0, 0);
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, bf16_bits_to_float(vv[i] & 0xFFFFu), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, bf16_bits_to_float(vv[i] >> 16), acc[2 * i + 1]);
      }
    }
    uint4 o;
    o.x = float_to_bf16_bits(acc[0]) | (float_to_bf16_bits(acc[1]) << 16);
    o.y = float_to_bf16_bits(acc[2]) | (float_to_bf16_bits(acc[3]) << 16);
    o.z = float_to_bf16_bits(acc[4]) | (float_to_bf16_bits(acc[5]) << 16);
    o.w = float_to_bf16_bits(acc[6]) | (float_to_bf16_bits(acc[7]) << 16);
    if (ok) st_cs_v4(orow + c, o);
  }
}

cudaError_t launch_finalize(const uint16_t* y, const float* topk_w, const int32_t* src_to_sorted,
                            int T, int k, int H, uint16_t* out, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int blocks = (int)ceil_div(T, kFinThreads / 32);
  finalize_kernel<<<blocks, kFinThreads, 0, stream>>>(y, topk_w, src_to_sorted, T, k, H, out);
  return cudaGetLastError();
}

}  // namespace mxmoe
