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
// One warp per token and 512-column chunk; each lane owns 16 consecutive
// columns (one 32 B load per source row), eight source rows in flight.
// Roofline: HBM-bound, k*H*2 B read + H*2 B written per token.
#include "common.cuh"
#include "internal.h"

namespace mxmoe {

constexpr int kFinThreads = 256;
constexpr int kErrDeviceCheck = 8;  // MXMOE_ERR_DEVICE_CHECK

// One warp per (token, 512-column chunk); a lane owns 16 consecutive columns
// (one 32-byte load per source row).  The slots go G at a time: the G rows'
// loads are all in flight before the first multiply-add.  Small batches take
// G = 8, so a warp waits for memory once per eight slots (there are too few
// warps to hide a chain of k dependent loads); large batches take G = 4
// (measured on the 16K-token prefill: 96.2 us against 102.4 with G = 2 and
// 110.6 with G = 8, whose registers leave fewer warps per SM in flight).
// The multiply-adds run in slot order whatever G is: the same bytes.
constexpr int kFinChunk = 512;

// Read-only 32-byte / 16-byte loads the compiler may schedule freely (y does
// not change while the kernel runs).
__device__ __forceinline__ void ld_ro_v8(const void* p, uint32_t (&r)[8]) {
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "l"(p));
}
__device__ __forceinline__ void ld_ro_v4x2(const void* p, uint32_t (&r)[8]) {
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "l"(p));
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "l"(static_cast<const char*>(p) + 16));
}

template <bool kV8, int kFinGroup>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(
    const uint16_t* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ src_to_sorted, int T, int k, int H, uint16_t* __restrict__ out,
    int* status) {
  pdl_wait();  // y of the GEMM before (programmatic serialization)
  const int lane = threadIdx.x & 31;
  const int nch = (H + kFinChunk - 1) / kFinChunk;
  const int64_t wid = (int64_t)blockIdx.x * (kFinThreads / 32) + (threadIdx.x >> 5);
  const int t = (int)(wid / nch);
  const int c = (int)(wid - (int64_t)t * nch);
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
  const int col = c * kFinChunk + lane * 16;
  const bool ok = col < H;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < k; j0 += kFinGroup) {  // warp-uniform
    uint32_t v[kFinGroup][8];
#pragma unroll
    for (int u = 0; u < kFinGroup; ++u) {
      const int64_t row = __shfl_sync(0xffffffffu, my_row, (j0 + u) & 31);
      if (ok && j0 + u < k) {
        if (kV8) ld_ro_v8(y + row * H + col, v[u]);
        else ld_ro_v4x2(y + row * H + col, v[u]);
      }
    }
    // fp32 multiply-adds in slot order j = 0, 1, ..., k - 1
#pragma unroll
    for (int u = 0; u < kFinGroup; ++u) {
      const float w = __shfl_sync(0xffffffffu, my_w, (j0 + u) & 31);
      if (ok && j0 + u < k) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[2 * i] = fmaf(w, bf16_bits_to_float(v[u][i] & 0xFFFFu), acc[2 * i]);
          acc[2 * i + 1] = fmaf(w, bf16_bits_to_float(v[u][i] >> 16), acc[2 * i + 1]);
        }
      }
    }
  }
  if (!ok) return;
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = cvt_bf16x2(acc[2 * i], acc[2 * i + 1]);
  uint16_t* dst = out + (int64_t)t * H + col;
  if (kV8) {
    st_cs_v8(dst, o);
  } else {
    st_cs_v4(dst, make_uint4(o[0], o[1], o[2], o[3]));
    st_cs_v4(dst + 8, make_uint4(o[4], o[5], o[6], o[7]));
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
  const int64_t chunk_blocks = ceil_div((int64_t)T * ceil_div(H, kFinChunk), kFinThreads / 32);
  int* st = device_status_ptr();
  // 16-column lanes need H % 16 == 0; 32-byte accesses need 32-byte aligned
  // rows; a few warps per SM take deep per-warp load groups, many take shallow ones
  const bool deep = chunk_blocks <= 4 * (int64_t)num_sms();
  const bool v8 = ((uintptr_t)y & 31u) == 0 && ((uintptr_t)out & 31u) == 0;
  if (H % 16 == 0) {
    auto kern = v8 ? (deep ? finalize_kernel<true, 8> : finalize_kernel<true, 4>)
                   : (deep ? finalize_kernel<false, 8> : finalize_kernel<false, 4>);
    return launch_pdl(kern, dim3((unsigned)chunk_blocks), dim3(kFinThreads), 0, stream, y,
                      topk_w, src_to_sorted, T, k, H, out, st);
  }
  return launch_pdl(finalize_narrow_kernel, dim3(blocks), dim3(kFinThreads), 0, stream, y, topk_w,
                    src_to_sorted, T, k, H, out, st);
}

}  // namespace mxmoe
