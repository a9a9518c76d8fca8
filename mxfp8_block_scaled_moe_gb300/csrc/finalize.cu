// Finalize routing: weighted top-k combine of the expert outputs back to
// token order ("Quantization on Ascend": MoE layers use init_routing /
// finalize_routing; sglang PR #32266 fused experts note, last step).
//
//   out[t] = sum_{j<k} topk_w[t, j] * y[src_to_sorted[t*k + j]]
//
// fp32 accumulation in slot order, one bf16 rounding (RNE) at the end.
// Every index is checked against [0, T*k) before it is used: an index
// outside records MXMOE_ERR_DEVICE_CHECK in the status word and its slot
// contributes nothing (row 0 is read with weight 0).
// One warp per token; each lane owns 16 consecutive columns (one 32 B load per
// source row), two 512-column chunks in flight.  Roofline: HBM-bound,
// k*H*2 B read + H*2 B written per token.
#include "common.cuh"
#include "internal.h"

namespace mxmoe {

constexpr int kFinThreads = 256;
constexpr int kErrDeviceCheck = 8;  // MXMOE_ERR_DEVICE_CHECK

// Lane owns 16 consecutive columns (one 32-byte load per source row) of a
// 512-column chunk; two chunks are in flight per iteration (2k loads).
template <bool kV8>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(
    const uint16_t* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ src_to_sorted, int T, int k, int H, uint16_t* __restrict__ out,
    int* status) {
  pdl_wait();  // y of the GEMM before (programmatic serialization)
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kFinThreads / 32) + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform
  int64_t my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_row = src_to_sorted[(int64_t)t * k + lane];
    my_w = topk_w[(int64_t)t * k + lane];
    if (my_row < 0 || my_row >= (int64_t)T * k) {
      report_error(status, kErrDeviceCheck);
      my_row = 0;
      my_w = 0.f;
    }
  }
  uint16_t* orow = out + (int64_t)t * H;
  for (int c0 = 0; c0 < H; c0 += 1024) {  // warp-uniform trip count
    const int ca = c0 + lane * 16, cb = ca + 512;
    const bool oka = ca < H, okb = cb < H;
    float acc_a[16], acc_b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) { acc_a[i] = 0.f; acc_b[i] = 0.f; }
    for (int j = 0; j < k; ++j) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, j);
      const float w = __shfl_sync(0xffffffffu, my_w, j);
      uint32_t va[8], vb[8];
      if (kV8) {
        if (oka) ld_nc_v8(y + row * H + ca, va);
        if (okb) ld_nc_v8(y + row * H + cb, vb);
      } else {
        if (oka) {
          const uint4 u0 = ld_nc_v4(y + row * H + ca), u1 = ld_nc_v4(y + row * H + ca + 8);
          va[0] = u0.x; va[1] = u0.y; va[2] = u0.z; va[3] = u0.w;
          va[4] = u1.x; va[5] = u1.y; va[6] = u1.z; va[7] = u1.w;
        }
        if (okb) {
          const uint4 u0 = ld_nc_v4(y + row * H + cb), u1 = ld_nc_v4(y + row * H + cb + 8);
          vb[0] = u0.x; vb[1] = u0.y; vb[2] = u0.z; vb[3] = u0.w;
          vb[4] = u1.x; vb[5] = u1.y; vb[6] = u1.z; vb[7] = u1.w;
        }
      }
      if (oka) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc_a[2 * i] = fmaf(w, bf16_bits_to_float(va[i] & 0xFFFFu), acc_a[2 * i]);
          acc_a[2 * i + 1] = fmaf(w, bf16_bits_to_float(va[i] >> 16), acc_a[2 * i + 1]);
        }
      }
      if (okb) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc_b[2 * i] = fmaf(w, bf16_bits_to_float(vb[i] & 0xFFFFu), acc_b[2 * i]);
          acc_b[2 * i + 1] = fmaf(w, bf16_bits_to_float(vb[i] >> 16), acc_b[2 * i + 1]);
        }
      }
    }
    uint32_t oa[8], ob[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      oa[i] = cvt_bf16x2(acc_a[2 * i], acc_a[2 * i + 1]);
      ob[i] = cvt_bf16x2(acc_b[2 * i], acc_b[2 * i + 1]);
    }
    if (kV8) {
      if (oka) st_cs_v8(orow + ca, oa);
      if (okb) st_cs_v8(orow + cb, ob);
    } else {
      if (oka) { st_cs_v4(orow + ca, make_uint4(oa[0], oa[1], oa[2], oa[3]));
                 st_cs_v4(orow + ca + 8, make_uint4(oa[4], oa[5], oa[6], oa[7])); }
      if (okb) { st_cs_v4(orow + cb, make_uint4(ob[0], ob[1], ob[2], ob[3]));
                 st_cs_v4(orow + cb + 8, make_uint4(ob[4], ob[5], ob[6], ob[7])); }
    }
  }
}

// H % 16 != 0 (H % 8 == 0): lane owns 8 columns, one 16-byte load per row.
__global__ void __launch_bounds__(kFinThreads) finalize_narrow_kernel(
    const uint16_t* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ src_to_sorted, int T, int k, int H, uint16_t* __restrict__ out,
    int* status) {
  pdl_wait();  // y of the GEMM before (programmatic serialization)
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kFinThreads / 32) + (threadIdx.x >> 5);
  if (t >= T) return;  // warp-uniform
  int64_t my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_row = src_to_sorted[(int64_t)t * k + lane];
    my_w = topk_w[(int64_t)t * k + lane];
    if (my_row < 0 || my_row >= (int64_t)T * k) {
      report_error(status, kErrDeviceCheck);
      my_row = 0;
      my_w = 0.f;
    }
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
    const uint4 o = make_uint4(cvt_bf16x2(acc[0], acc[1]), cvt_bf16x2(acc[2], acc[3]),
                               cvt_bf16x2(acc[4], acc[5]), cvt_bf16x2(acc[6], acc[7]));
    if (ok) st_cs_v4(orow + c, o);
  }
}

cudaError_t launch_finalize(const uint16_t* y, const float* topk_w, const int32_t* src_to_sorted,
                            int T, int k, int H, uint16_t* out, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int blocks = (int)ceil_div(T, kFinThreads / 32);
  int* st = device_status_ptr();
  // 16-column lanes need H % 16 == 0; 32-byte accesses need 32-byte aligned rows
  if (H % 16 == 0 && ((uintptr_t)y & 31u) == 0 && ((uintptr_t)out & 31u) == 0)
    return launch_pdl(finalize_kernel<true>, dim3(blocks), dim3(kFinThreads), 0, stream, y, topk_w,
                      src_to_sorted, T, k, H, out, st);
  else if (H % 16 == 0)
    return launch_pdl(finalize_kernel<false>, dim3(blocks), dim3(kFinThreads), 0, stream, y, topk_w,
                      src_to_sorted, T, k, H, out, st);
  else
    return launch_pdl(finalize_narrow_kernel, dim3(blocks), dim3(kFinThreads), 0, stream, y, topk_w,
                      src_to_sorted, T, k, H, out, st);
}

}  // namespace mxmoe
