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
// thread owns one block (two 32-byte loads, one 32-byte store, one scale
// byte; a warp's scale bytes are 32 contiguous bytes).
#include "common.cuh"
#include "internal.h"
#include "tiled_scales.h"

namespace mxmoe {

template <bool kV8>
__global__ void __launch_bounds__(256) mx_quantize_kernel(const uint16_t* __restrict__ x,
                                                          int64_t n_blocks,
                                                          uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ scale) {
  // one lane = one 32-element block: 64 B in, 32 B + 1 scale byte out
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks;
       b += (int64_t)gridDim.x * blockDim.x) {
    uint32_t w[16], o[8];
    load_block32_bf16<kV8>(x + b * 32, w);
    const uint32_t sb = quant_block32_bf16(w, o);
    store_block32_e4m3<kV8>(q + b * 32, o);
    scale[b] = (uint8_t)sb;
  }
}

cudaError_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                               uint8_t* scale, cudaStream_t stream) {
  const int64_t n_blocks = rows * K / 32;
  if (n_blocks == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = ceil_div(n_blocks, threads);
  const int64_t cap = (int64_t)num_sms() * 8;  // 2048 resident threads per SM
  if (blocks > cap) blocks = cap;
  const bool v8 = ((uintptr_t)x & 31u) == 0 && ((uintptr_t)q & 31u) == 0;
  if (v8)
    mx_quantize_kernel<true><<<(unsigned)blocks, threads, 0, stream>>>(x, n_blocks, q, scale);
  else
    mx_quantize_kernel<false><<<(unsigned)blocks, threads, 0, stream>>>(x, n_blocks, q, scale);
  return cudaGetLastError();
}

// MXFP4 (W4A8 weights): one lane per block, 64 B in, 16 B + 1 scale byte out.
template <bool kV8>
__global__ void __launch_bounds__(256) mx_quantize_fp4_kernel(const uint16_t* __restrict__ x,
                                                              int64_t n_blocks,
                                                              uint8_t* __restrict__ q,
                                                              uint8_t* __restrict__ scale) {
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks;
       b += (int64_t)gridDim.x * blockDim.x) {
    uint32_t w[16], o[4];
    load_block32_bf16<kV8>(x + b * 32, w);
    const uint32_t sb = quant_block32_bf16_fp4(w, o);
    st_cs_v4(q + b * 16, make_uint4(o[0], o[1], o[2], o[3]));
    scale[b] = (uint8_t)sb;
  }
}

cudaError_t launch_mx_quantize_fp4(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                                   uint8_t* scale, cudaStream_t stream) {
  const int64_t n_blocks = rows * K / 32;
  if (n_blocks == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = ceil_div(n_blocks, threads);
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (((uintptr_t)x & 31u) == 0)
    mx_quantize_fp4_kernel<true><<<(unsigned)blocks, threads, 0, stream>>>(x, n_blocks, q, scale);
  else
    mx_quantize_fp4_kernel<false><<<(unsigned)blocks, threads, 0, stream>>>(x, n_blocks, q, scale);
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
