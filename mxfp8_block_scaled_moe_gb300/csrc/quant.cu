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

// Row-wise MX quantization for any K % 16 == 0 (the dense linear's
// activations and weights).  With K % 32 == 16 every row ends in a partial
// block of 16 elements ("offline partial MXFP8 block-scale layout", sglang
// PR #32266): ceil(K/32) scales per row, the last over the elements that
// exist.  One thread per block; block b = row * nbr + j (nbr = ceil(K/32)).
// Rows are 32-byte aligned in bf16 and 16-byte aligned in e4m3.
// kTiled: scales go straight to the tiled layout with KT = ceil(K/128)
// slices; the slots of the last slice past nbr get 127 (scale 1 over an
// all-zero payload, so they add exactly 0 in the GEMM).  `offsets` (optional)
// receives the one-group offsets {0, rows} the grouped GEMM reads.
// kFp4: MXFP4 rows (W4A4 activations; K % 32 == 0): q is [rows, K/2] packed
// e2m1, 16 bytes per block.
template <bool kV8, bool kTiled, bool kFp4 = false>
__global__ void __launch_bounds__(256) mx_quantize_rows_kernel(const uint16_t* __restrict__ x,
                                                               int64_t rows, int64_t K,
                                                               uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ scale,
                                                               int64_t* __restrict__ offsets) {
  if (offsets && blockIdx.x == 0 && threadIdx.x == 0) {
    offsets[0] = 0;
    offsets[1] = rows;
  }
  const int64_t nbr = (K + 31) / 32;
  const int KT = (int)((K + 127) / 128);
  const int64_t n = rows * nbr;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = b / nbr;
    const int j = (int)(b - r * nbr);
    const uint16_t* xb = x + r * K + 32 * j;
    uint8_t* qb = q + r * K + 32 * j;
    uint32_t sb;
    if (kFp4) {
      uint32_t w[16], o[4];
      load_block32_bf16<kV8>(xb, w);
      sb = quant_block32_bf16_fp4(w, o);
      st_cs_v4(q + (r * K + 32 * j) / 2, make_uint4(o[0], o[1], o[2], o[3]));
    } else if (j != nbr - 1 || (K & 31) == 0) {
      uint32_t w[16], o[8];
      load_block32_bf16<kV8>(xb, w);
      sb = quant_block32_bf16(w, o);
      store_block32_e4m3<false>(qb, o);
    } else {
      uint32_t w[8], o[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 v = ld_nc_v4(xb + 8 * i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = umax(m, bf16x2_absmax_bits(w[i]));
      sb = e8m0_from_amax_bits(m);
      const float inv = inv_scale_from_e8m0(sb);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
        o[i] = cvt_e4m3x4(bf16_bits_to_float(w0 & 0xFFFFu) * inv, bf16_bits_to_float(w0 >> 16) * inv,
                          bf16_bits_to_float(w1 & 0xFFFFu) * inv, bf16_bits_to_float(w1 >> 16) * inv);
      }
      st_cs_v4(qb, make_uint4(o[0], o[1], o[2], o[3]));
    }
    if (kTiled) {
      scale[tiled_scale_offset(r, j, KT)] = (uint8_t)sb;
      if (j == nbr - 1)
        for (int jj = j + 1; jj < 4 * KT; ++jj) scale[tiled_scale_offset(r, jj, KT)] = 127;
    } else {
      scale[b] = (uint8_t)sb;
    }
  }
}

template <bool kTiled, bool kFp4 = false>
static cudaError_t launch_rows(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                               uint8_t* scale, cudaStream_t stream, int64_t* offsets = nullptr) {
  const int64_t n = rows * ((K + 31) / 32);
  if (n == 0) return cudaSuccess;
  int64_t blocks = ceil_div(n, 256);
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (((uintptr_t)x & 31u) == 0)
    mx_quantize_rows_kernel<true, kTiled, kFp4>
        <<<(unsigned)blocks, 256, 0, stream>>>(x, rows, K, q, scale, offsets);
  else
    mx_quantize_rows_kernel<false, kTiled, kFp4>
        <<<(unsigned)blocks, 256, 0, stream>>>(x, rows, K, q, scale, offsets);
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_tiled(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                                     uint8_t* scale_tiled, int64_t* offsets, cudaStream_t stream,
                                     bool fp4) {
  if (fp4) {
    if (K % 32 != 0) return cudaErrorInvalidValue;
    return launch_rows<true, true>(x, rows, K, q, scale_tiled, stream, offsets);
  }
  return launch_rows<true>(x, rows, K, q, scale_tiled, stream, offsets);
}

cudaError_t launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t K, uint8_t* q,
                               uint8_t* scale, cudaStream_t stream) {
  if (K % 32 != 0) return launch_rows<false>(x, rows, K, q, scale, stream);
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

// K % 128 != 0 or rows % 128 != 0 (the dense linear's weights): byte-wise
// over the rows padded to whole 128-row blocks; every slot past the ceil(K/32)
// scales of a row, and every slot of a padding row, gets 127 (scale 1 over a
// payload that the GEMM's loads zero-fill).
__global__ void __launch_bounds__(256) scales_to_tiled_partial_kernel(const uint8_t* __restrict__ in,
                                                                      int64_t rows, int K32, int KT,
                                                                      uint8_t* __restrict__ out) {
  const int64_t n = (rows + 127) / 128 * 128 * KT * 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / (KT * 4);
    const int j = (int)(i - row * KT * 4);
    out[tiled_scale_offset(row, j, KT)] =
        row < rows && j < K32 ? in[row * K32 + j] : (uint8_t)127;
  }
}

cudaError_t launch_scales_to_tiled(const uint8_t* scale, int64_t rows, int64_t K, uint8_t* out,
                                   cudaStream_t stream) {
  if (K % 128 != 0 || rows % 128 != 0) {
    const int KT = (int)((K + 127) / 128), K32 = (int)((K + 31) / 32);
    const int64_t n = ceil_div(rows, 128) * 128 * KT * 4;
    if (n == 0) return cudaSuccess;
    int64_t blocks = ceil_div(n, 256);
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    scales_to_tiled_partial_kernel<<<(unsigned)blocks, 256, 0, stream>>>(scale, rows, K32, KT, out);
    return cudaGetLastError();
  }
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
