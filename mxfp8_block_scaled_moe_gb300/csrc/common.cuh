// Device helpers shared by the MXFP8 MoE kernels (sm_103a).
//
// MX element/scale arithmetic (OCP MX v1.0, the format named on
// "Quantization on Ascend", MoE MXFP8 notes):
//   block scale byte  b = clamp(floor(log2(amax)) - 8, -127, 127) + 127
//   element           q = e4m3_rn_satfinite(x * 2^(127 - b))
// For a finite fp32/bf16 amax with biased exponent field ef (0 for zero and
// subnormals), floor(log2(amax)) - 8 + 127 = ef - 8 for normal values, and
// every subnormal or zero amax clamps to -127, so b = max(ef - 8, 0).  The
// largest b any bf16/fp32 input reaches is 254 - 8 = 246, so 2^(127 - b) is
// always a normal fp32 and the product x * 2^(127 - b) is exact (|x|/2^s <
// 512; values below 2^-126 after scaling round to zero in e4m3 anyway).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxmoe {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// fp32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t float_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

// Scale byte from the bit pattern of |amax| as fp32 (sign cleared).
__device__ __forceinline__ uint32_t e8m0_from_amax_bits(uint32_t amax_bits) {
  int ef = (int)(amax_bits >> 23);
  int b = ef - 8;
  return (uint32_t)(b < 0 ? 0 : b);
}

// 2^(127 - b) as an fp32 multiplier.
__device__ __forceinline__ float inv_scale_from_e8m0(uint32_t b) {
  return __uint_as_float((254u - b) << 23);
}

// Two fp32 -> two e4m3 bytes (lo -> bits 0..7, hi -> bits 8..15), RNE, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Four fp32 -> packed 4 e4m3 bytes (v0 in the lowest byte).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float v0, float v1, float v2, float v3) {
  return cvt_e4m3x2(v0, v1) | (cvt_e4m3x2(v2, v3) << 16);
}

// Two fp32 -> packed bf16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t umax(uint32_t a, uint32_t b) { return a > b ? a : b; }

// |x| bit pattern of a bf16 pair packed in a 32-bit word, as two fp32 patterns' max.
__device__ __forceinline__ uint32_t bf16x2_absmax_bits(uint32_t w) {
  uint32_t lo = (w & 0x7FFFu) << 16;
  uint32_t hi = (w & 0x7FFF0000u);
  return umax(lo, hi);
}

// Streaming 16-byte global accesses.
// Ask the L2 to fetch [p, p + bytes) (16-byte aligned, a multiple of 16
// bytes); the issuing thread does not wait for the data, but the SM's bulk
// copy unit moves the bytes one request after another.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_cs_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" :: "l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w) : "memory");
}

// 32-byte (one full sector) global store; the address must be 32-byte aligned.
__device__ __forceinline__ void st_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 32-byte global load (read-only, not kept in L1) / streaming store; the
// address must be 32-byte aligned.
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st_cs_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Load the 32 bf16 of one MX block (64 bytes) as 16 words; 32-byte loads
// when kV8 (64-byte aligned block), else 16-byte loads.
template <bool kV8>
__device__ __forceinline__ void load_block32_bf16(const uint16_t* p, uint32_t (&w)[16]) {
  if (kV8) {
    ld_nc_v8(p, *reinterpret_cast<uint32_t(*)[8]>(&w[0]));
    ld_nc_v8(p + 16, *reinterpret_cast<uint32_t(*)[8]>(&w[8]));
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = ld_nc_v4(p + 8 * i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

// MX-quantize one block of 32 bf16 (16 words) into 32 e4m3 bytes (8 words);
// returns the e8m0 scale byte.
__device__ __forceinline__ uint32_t quant_block32_bf16(const uint32_t (&w)[16], uint32_t (&o)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = umax(m, bf16x2_absmax_bits(w[i]));
  const uint32_t sb = e8m0_from_amax_bits(m);
  const float inv = inv_scale_from_e8m0(sb);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w0 = w[2 * i], w1 = w[2 * i + 1];
    o[i] = cvt_e4m3x4(bf16_bits_to_float(w0 & 0xFFFFu) * inv, bf16_bits_to_float(w0 >> 16) * inv,
                      bf16_bits_to_float(w1 & 0xFFFFu) * inv, bf16_bits_to_float(w1 >> 16) * inv);
  }
  return sb;
}

template <bool kV8>
__device__ __forceinline__ void store_block32_e4m3(uint8_t* p, const uint32_t (&o)[8]) {
  if (kV8) {
    st_cs_v8(p, o);
  } else {
    st_cs_v4(p, make_uint4(o[0], o[1], o[2], o[3]));
    st_cs_v4(p + 16, make_uint4(o[4], o[5], o[6], o[7]));
  }
}

// ---- MXFP4 (e2m1 elements, W4A8 weights).  Same rule with the e2m1 element's
// largest power-of-two exponent 2: b = max(ef - 2, 0), elements
// e2m1_rn_satfinite(x * 2^(127 - b)); 2^(127 - b) stays a normal fp32 for
// every b a bf16 input reaches (b <= 252).

// MXFP4 scale byte from the bit pattern of |amax| as fp32 (sign cleared).
__device__ __forceinline__ uint32_t e8m0_fp4_from_amax_bits(uint32_t amax_bits) {
  const int ef = (int)(amax_bits >> 23);
  return (uint32_t)(ef - 2 < 0 ? 0 : ef - 2);
}

// Two fp32 -> one byte of two e2m1 codes (lo -> bits 0..3, hi -> bits 4..7),
// round to nearest even, saturating to +-6.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// MXFP4-quantize one block of 32 bf16 (16 words) into 16 packed bytes (4
// words; element 2i in the low nibble of byte i); returns the e8m0 scale byte.
__device__ __forceinline__ uint32_t quant_block32_bf16_fp4(const uint32_t (&w)[16],
                                                           uint32_t (&o)[4]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = umax(m, bf16x2_absmax_bits(w[i]));
  const uint32_t sb = e8m0_fp4_from_amax_bits(m);
  const float inv = inv_scale_from_e8m0(sb);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t wj = w[4 * i + j];
      word |= cvt_e2m1x2(bf16_bits_to_float(wj & 0xFFFFu) * inv,
                         bf16_bits_to_float(wj >> 16) * inv) << (8 * j);
    }
    o[i] = word;
  }
  return sb;
}

// Total order of finite fp32 values as unsigned keys (top-k selection) (-0 is ordered with +0).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ bool aligned32(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 31u) == 0;
}

// Programmatic dependent launch: a kernel launched with the
// programmatic-serialization attribute may start before its predecessor on
// the stream has finished; pdl_wait() blocks until that predecessor grid has
// completed and its memory is visible (a no-op for an ordinary launch), and
// pdl_launch_dependents() lets the next such kernel be scheduled.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Record the first device-side error in the library's status word.
__device__ __forceinline__ void report_error(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace mxmoe
