// Shared device code of the grouped MXFP8 GEMM kernels (1-SM and 2-SM).
//
// PTX wrappers (mbarrier, TMA, bulk copies, tcgen05), descriptor builders,
// bounded barrier waits, the per-expert tile schedule, the fused epilogues
// (SwiGLU + MX requant for gmm1, bf16 for gmm2) and the host-side tensor-map
// helpers.  See gemm.cu for the design of the kernels.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tiled_scales.h"

namespace mxmoe {
namespace gemm {

constexpr int BM = 128;         // rows of A per CTA tile (tokens)
constexpr int BK = 128;         // K elements (= bytes) per stage
constexpr int EPI_WARPS = 16;   // epilogue warps (a multiple of 4)
constexpr int EPI_GROUPS = EPI_WARPS / 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;  // 2-SM kernel: producer, MMA, epilogue
constexpr int SF_WARPS = 4;     // 1-SM kernel: one scale-factor writer per TMEM lane quarter
constexpr int EPI_WARP0 = 2 + SF_WARPS;       // 1-SM kernel: first epilogue warp
constexpr int THREADS1 = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr int MAX_E = 256;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256;    // scale factors after the accumulator
constexpr int SF_COLS_PER_STAGE = 16;
constexpr int ERR_TIMEOUT = 7;  // MXMOE_ERR_DEVICE_TIMEOUT
constexpr int ERR_CHECK = 8;    // MXMOE_ERR_DEVICE_CHECK

struct Params {
  const uint8_t* sfa;        // [M, K/32], or tiled (tiled_scales.h)
  const uint8_t* sfb;        // [E * Nw, K/32], or tiled
  const int64_t* offsets;    // [E+1]
  void* out;                 // aq [M, n_out] e4m3 or y [M, n_out] bf16
  uint8_t* out_scale;        // as [M, n_out/32] (gmm1), or tiled
  int64_t M;
  int E, K, Nw, n_out, n_tiles_n;
  int* status;
  long long wait_limit;
  // split-K (1-SM kernel, bf16-out GEMM with one group): tile = base * ksplit
  // + ks covers K slices [ks * kper, min(KT, (ks + 1) * kper)) and writes its
  // fp32 partial sums to partial [ksplit][M][n_out]; ksplit = 1 otherwise
  int ksplit;
  float* partial;
  // small batches (1-SM kernel, gmm1): the raw weight array [E * Nw, row
  // bytes], whose rows the CTA's first unit would read if every expert had
  // one m-tile, prefetched into L2 before the wait for the previous kernel (a
  // guess, made while the routing runs); null: no prefetch
  const uint8_t* pf_b;
  int64_t pf_row_bytes;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
// kind::mxf4: packed e2m1 x e2m1 operands (two elements per byte in shared
// memory), K = 64 per instruction, two UE8M0 scales per row (scale_vec::2X:
// bytes id and id + 1 of the row's scale word, id = 0 or 2).
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 TMEM lanes (this warp's quarter) x 4 columns from registers.
__device__ __forceinline__ void tmem_st_4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), descriptor version 1 at bits 46-48, and
// the swizzle mode at bits 61-63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swizzle) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A e4m3
// (format 0 at bits 7-9), B e4m3 or, for the MXFP4 weights of W4A8, e2m1
// (format 5 at bits 10-12), both K-major, N >> 3 at bits 17-22, UE8M0 scale
// type (bit 23), M >> 4 at bits 24-28; the scale-factor byte selectors (bits
// 29-30 for A, 4-5 for B) are or-ed in per K step.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_fp4 = false) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
         (b_fp4 ? 5u << 10 : 0u);
}

// Instruction descriptor of kind::mxf4 (both operands packed e2m1, format 1
// at bits 7-9 / 10-12), K-major, same N / M / UE8M0 fields as above; with
// scale_vec::2X the byte selectors are 0 or 2.
__host__ __device__ constexpr uint32_t make_idesc_mxf4(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) | (1u << 10) |
         (1u << 7);
}

// Operand formats of a GEMM instantiation: W8A8 (e4m3 x e4m3), W4A8 (e4m3
// activations x e2m1 weights; kind::mxf8f6f4, the weights unpacked to one
// element per byte by the tensor map), W4A4 (e2m1 x e2m1, kind::mxf4 on
// packed operands; gmm1 then requantizes its output to MXFP4 as well).
enum : int { FMT_W8A8 = 0, FMT_W4A8 = 1, FMT_W4A4 = 2 };

// Bounded mbarrier wait.  Returns false when the CTA is aborting (another
// role timed out) or this wait ran out of time (then it starts the abort).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, long long limit,
                                         int* status, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      report_error(status, ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// Map a flat tile index to (expert, m tile, n tile).
__device__ __forceinline__ void decode_tile(int tile, const int* ts, int E, int n_tiles_n,
                                            int& e, int& mt, int& nt) {
  int lo = 0, hi = E - 1;  // last e with ts[e] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ts[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  e = lo;
  const int local = tile - ts[e];
  mt = local / n_tiles_n;
  nt = local - mt * n_tiles_n;
}

// silu(g) * u = g * u / (1 + e^-g), with e^-g = 2^(-g * log2 e) on the
// hardware ex2 unit and the reciprocal on rcp.approx (relative error of a few
// fp32 ulp; e^-g -> inf gives 0, e^-g -> 0 gives g * u).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float swiglu(float g, float u) {
  const float e = ex2_approx(-1.4426950408889634f * g);
  return (g * u) * rcp_approx(1.0f + e);
}


// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_cluster(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster (cluster address), with
// the default release at CTA scope: a cluster-scope release fences every prior
// memory operation of the thread and costs on the order of a thousand cycles
// per arrive.  The signals sent this way order tcgen05 work (TMEM stores and
// loads, bracketed by tcgen05 thread-sync fences), not generic memory traffic.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// ---------------------------------------------------------------- schedule

// Per-expert schedule in shared memory, built by one warp: s_off[0..E] the
// row offsets, s_ts[e] the first work unit of expert e (a unit is CL
// consecutive 128-row m-tiles x one n-tile), s_ts[E] the unit count, s_mtb[e]
// the first 128-row block of expert e (tiled scale layout), s_mtb[E] total.
//
// The offsets are checked on the way: offsets[0] == 0, non-decreasing, and
// offsets[E] == M.  Any other array would send tiles to rows outside
// [0, M); instead the kernel records MXMOE_ERR_DEVICE_CHECK and schedules no
// work (every CTA sees the same offsets, so every CTA stops).
template <int CL>
__device__ __forceinline__ void build_schedule(const Params& p, int lane, int64_t* s_off,
                                               int* s_ts, int* s_mtb) {
  constexpr int PER = MAX_E / 32;
  const int E = p.E;
  int cnt[PER], mcnt[PER];
  int run = 0, mrun = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    int c = 0;
    if (e < E) {
      const int64_t o0 = p.offsets[e], o1 = p.offsets[e + 1];
      s_off[e] = o0;
      if (e == E - 1) s_off[E] = o1;
      bad |= o1 < o0 || (e == 0 && o0 != 0) || (e == E - 1 && o1 != p.M);
      c = o1 < o0 ? 0 : (int)((o1 - o0 + BM - 1) / BM);
    }
    cnt[i] = run;
    mcnt[i] = mrun;
    run += (c + CL - 1) / CL * p.n_tiles_n;
    mrun += c;
  }
  bad = __any_sync(0xffffffffu, bad);
  int incl = run, mincl = mrun;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    const int mo = __shfl_up_sync(0xffffffffu, mincl, off);
    if (lane >= off) { incl += o; mincl += mo; }
  }
  const int excl = incl - run, mexcl = mincl - mrun;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    if (e < E) { s_ts[e] = bad ? 0 : excl + cnt[i]; s_mtb[e] = bad ? 0 : mexcl + mcnt[i]; }
  }
  if (lane == 31) { s_ts[E] = bad ? 0 : incl; s_mtb[E] = bad ? 0 : mincl; }
  if (bad && lane == 0) report_error(p.status, ERR_CHECK);
}

// ---------------------------------------------------------------- epilogue

// One epilogue thread's work on one tile: drain its slice of the TMEM
// accumulator row into registers, signal `release` (the accumulator may be
// overwritten), then SwiGLU + MX requant (gmm1) or bf16 rounding (gmm2) and
// the stores.  BN = accumulator columns, grp = column slice of this warp.
// `release` is called by every thread; it arrives once per warp.
template <int BN, bool kSwiglu, bool kTiledSF, bool kFp4Out, bool kPartial, typename Release>
__device__ __forceinline__ void epilogue_tile(const Params& p, uint32_t t_row, int grp, int row,
                                              int lane, int64_t grow, bool valid, int nt,
                                              int64_t tiled_row, Release release, int ks = 0) {
  constexpr int GC = BN / 2 / EPI_GROUPS;
  constexpr int PC = BN / EPI_GROUPS;
  constexpr int CH = kSwiglu ? 2 * (GC / 32) : PC / 32;  // 32-column chunks
  static_assert(kSwiglu ? GC % 32 == 0 : PC % 32 == 0, "epilogue slices are whole 32-column chunks");
  uint32_t v[CH][32];
  if (kSwiglu) {
    // gate columns [grp*GC, +GC), up columns BN/2 + the same
#pragma unroll
    for (int c = 0; c < CH / 2; ++c) {
      tmem_ld_32(t_row + grp * GC + c * 32, v[c]);
      tmem_ld_32(t_row + BN / 2 + grp * GC + c * 32, v[CH / 2 + c]);
    }
  } else {
#pragma unroll
    for (int c = 0; c < CH; ++c) tmem_ld_32(t_row + grp * PC + c * 32, v[c]);
  }
  tmem_ld_wait();
  tc_fence_before();
  __syncwarp();
  release();
  if (kSwiglu) {
    uint8_t* aq = reinterpret_cast<uint8_t*>(p.out);
#pragma unroll
    for (int c = 0; c < CH / 2; ++c) {
      float a[32];
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        a[i] = swiglu(__uint_as_float(v[c][i]), __uint_as_float(v[CH / 2 + c][i]));
        m = umax(m, __float_as_uint(a[i]) & 0x7FFFFFFFu);
      }
      const uint32_t sb = kFp4Out ? e8m0_fp4_from_amax_bits(m) : e8m0_from_amax_bits(m);
      const float inv = inv_scale_from_e8m0(sb);
      uint32_t o[8];
      if (kFp4Out) {
        // MXFP4: 16 packed bytes, element 2i in the low nibble of byte i
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t word = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            word |= cvt_e2m1x2(a[8 * i + 2 * j] * inv, a[8 * i + 2 * j + 1] * inv) << (8 * j);
          o[i] = word;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          o[i] = cvt_e4m3x4(a[4 * i] * inv, a[4 * i + 1] * inv, a[4 * i + 2] * inv,
                            a[4 * i + 3] * inv);
      }
      if (valid) {
        const int64_t col = (int64_t)nt * (BN / 2) + grp * GC + c * 32;
        if (kFp4Out)
          st_v4(aq + grow * (p.n_out / 2) + col / 2, make_uint4(o[0], o[1], o[2], o[3]));
        else
          st_v8(aq + grow * p.n_out + col, o);
        if (kTiledSF)
          p.out_scale[tiled_scale_offset(tiled_row, (int)(col >> 5), p.n_out / 128)] = (uint8_t)sb;
        else
          p.out_scale[grow * (p.n_out / 32) + (col >> 5)] = (uint8_t)sb;
      }
    }
  } else if (kPartial) {
    // split-K: this K range's fp32 partial sums (the ranges are added in a
    // fixed order and rounded to bf16 by splitk_reduce_kernel)
    if (valid) {
      float* dst = p.partial + ((int64_t)ks * p.M + grow) * p.n_out;
#pragma unroll
      for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int64_t col = (int64_t)nt * BN + grp * PC + c * 32 + 4 * i;
          if (col < p.n_out)
            *reinterpret_cast<float4*>(dst + col) =
                make_float4(__uint_as_float(v[c][4 * i]), __uint_as_float(v[c][4 * i + 1]),
                            __uint_as_float(v[c][4 * i + 2]), __uint_as_float(v[c][4 * i + 3]));
        }
    }
  } else {
    uint16_t* y = reinterpret_cast<uint16_t*>(p.out);
    if constexpr (CH == 2) {
      // x[s]: 32-byte sector s (16 columns) of this thread's 64-column row slice
      uint32_t x[4][8];
#pragma unroll
      for (int c = 0; c < CH; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          x[2 * c + i / 8][i % 8] =
              cvt_bf16x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1]));
      // 4 x 4 transpose of sectors inside each quad of lanes (two xor-shuffle
      // rounds): afterwards lane q of a quad holds sector q of the quad's four
      // rows, so one warp store writes 8 whole 128-byte lines instead of 32
      // sectors of 32 different lines.
      const int qi = lane & 3;
      const bool odd = (qi & 1) != 0, hi = (qi & 2) != 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        uint32_t r = __shfl_xor_sync(0xffffffffu, odd ? x[0][w] : x[1][w], 1);
        if (odd) x[0][w] = r; else x[1][w] = r;
        r = __shfl_xor_sync(0xffffffffu, odd ? x[2][w] : x[3][w], 1);
        if (odd) x[2][w] = r; else x[3][w] = r;
        r = __shfl_xor_sync(0xffffffffu, hi ? x[0][w] : x[2][w], 2);
        if (hi) x[0][w] = r; else x[2][w] = r;
        r = __shfl_xor_sync(0xffffffffu, hi ? x[1][w] : x[3][w], 2);
        if (hi) x[1][w] = r; else x[3][w] = r;
      }
      // the quad's rows are consecutive: row j of the quad is grow - qi + j
      // (a ragged last n-tile, n_out % 16 == 0, masks whole sectors)
      const int64_t col = (int64_t)nt * BN + grp * PC + qi * 16;
      const bool col_ok = col < p.n_out;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool ok = __shfl_sync(0xffffffffu, valid ? 1 : 0, (lane & ~3) + j) != 0;
        if (ok && col_ok) st_v8(y + (grow - qi + j) * p.n_out + col, x[j]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = cvt_bf16x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1]));
        const int64_t col = (int64_t)nt * BN + grp * PC + c * 32;
        if (valid) {
          uint16_t* dst = y + grow * p.n_out + col;
          if (col < p.n_out) st_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(&o[0]));
          if (col + 16 < p.n_out) st_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(&o[8]));
        }
      }
    }
  }
}

// ---------------------------------------------------------------- host

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2D tensor [outer, inner] (inner contiguous), 128-byte swizzled box.  fp4
// (W4A8's weights, read by kind::mxf8f6f4): packed e2m1 (two per byte, inner
// counted in elements) landing in shared memory as 16-element groups of 8
// packed bytes in 16-byte slots, so a 128-element row of the box takes 128
// bytes there, as an e4m3 row does.  W4A4's packed operands (kind::mxf4) are
// plain bytes: inner = K / 2.
inline bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer, bool fp4 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {fp4 ? inner / 2 : inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// 2-SM launch (gemm2sm.cu): returns cudaErrorNotSupported when the device
// cannot co-schedule CTA pairs, so the caller falls back to the 1-SM kernel.
template <bool kSwiglu, bool kTiledSF, int kFmt>
cudaError_t launch_pair(const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                        const uint8_t* sfb, const int64_t* offsets, int64_t M, int E, int K,
                        int Nw, int n_out, void* out, uint8_t* out_scale, cudaStream_t stream);

}  // namespace gemm
}  // namespace mxmoe
