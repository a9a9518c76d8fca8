// MX quantization of bf16 rows along K (load-time weight quant and the
// standalone activation quant of the two-step comparator).
//
// "Quantization on Ascend", MoE MXFP8 online path: bf16 expert weights are
// quantized once at load, a 3D [E, N, K] input accepted directly.  With
// K % 32 == 0 no block straddles a row, so [E, N, K] is a flat run of
// E*N*K/32 blocks and the [E, N, K/32] scale array is indexed by the flat
// block number.
//
// Roofline: HBM-bound, 2 B read + 1 B + 1/32 B written per element.  Each
// thread owns half a block (16 elements = two 16 B loads, one 16 B store);
// the partner lane holds the other half, so the block amax is one shuffle.
#include "common.cuh"
#include "internal.h"
#include "tiled_scales.h"

namespace mxmoe {

__global__ void __launch_bounds__(256) mx_quantize_kernel(const uint16_t* __restrict__ x,
                                                          int64_t n_units,
                                                          uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = warp * 32; base < n_units; base += nwarps * 32) {
    const int64_t u = base + lane;  // half-block index: elements [16u, 16u+16)
    const bool ok = u < n_units;
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (ok) {
      a = ld_nc_v4(x + u * 16);
      b = ld_nc_v4(x + u * 16 + 8);
    }
    uint32_t m = umax(umax(bf16x2_absmax_bits(a.x), bf16x2_absmax_bits(a.y)),
                      umax(bf16x2_absmax_bits(a.z), bf16x2_absmax_bits(a.w)));
    m = umax(m, umax(umax(bf16x2_absmax_bits(b.x), bf16x2_absmax_bits(b.y)),
                     umax(bf16x2_absmax_bits(b.z), bf16x2_absmax_bits(b.w))));
    m = umax(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const uint32_t sb = e8m0_from_amax_bits(m);
    const float inv = inv_scale_from_e8m0(sb);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
      o[i] = cvt_e4m3x4(bf16_bits_to_float(w0 & 0xFFFFu) * inv, bf16_bits_to_float(w0 >> 16) * inv,
                        bf16_bits_to_float(w1 & 0xFFFFu) * inv, bf16_bits_to_float(w1 >> 16) * inv);
    }
    if (ok) {
      st_cs_v4(q + u * 16, make_uint4(o[0], o[1], o[2], o[3]));
      if ((lane & 1) == 0) scale[u >> 1] = (uint8_t)sb;
    }
  }
}

cudaError_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                               uint8_t* scale, cudaStream_t stream) {
  const int64_t n_units = rows * K / 16;
  if (n_units == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = ceil_div(n_units, threads);
  const int64_t cap = (int64_t)num_sms() * 8;  // 2048 resident threads per SM
  if (blocks > cap) blocks = cap;
  mx_quantize_kernel<<<(unsigned)blocks, threads, 0, stream>>>(x, n_units, q, scale);
  return cudaGetLastError();
}

// [rows, K/32] e8m0 scales -> the tiled layout of tiled_scales.h.  One thread
// moves one row's 4 scale bytes of one 128-element K slice (a 4-byte word:
// K/32 is a multiple of 4, so every word is aligned).
__global__ void __launch_bounds__(256) scales_to_tiled_kernel(const uint32_t* __restrict__ in,
                                                              int64_t rows, int KT,
                                                              uint32_t* __restrict__ out) {
  const int64_t n = rows * KT;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / KT;
    const int kt = (int)(i - row * KT);
    out[tiled_scale_offset(row, kt * 4, KT) >> 2] = in[i];
  }
}

cudaError_t launch_scales_to_tiled(const uint8_t* scale, int64_t rows, int64_t K, uint8_t* out,
                                   cudaStream_t stream) {
  const int KT = (int)(K / 128);
  const int64_t n = rows * KT;
  if (n == 0) return cudaSuccess;
  int64_t blocks = ceil_div(n, 256);
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  scales_to_tiled_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const uint32_t*>(scale), rows, KT, reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

}  // namespace mxmoe
