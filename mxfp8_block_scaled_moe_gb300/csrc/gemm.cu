// Grouped MXFP8 GEMMs of the MoE expert forward on 5th-generation tensor
// cores (tcgen05, sm_103a).
//
//   gmm1 (grouped_gemm_swiglu_quant_mxfp8): per expert e, rows r of
//        [off_e, off_{e+1}): h = xq[r] . w13[e]^T, a = silu(h_gate) * h_up,
//        requantized to MXFP8 along I (PR #30768 report,
//        GroupedMatmulSwigluQuant; "Quantization on Ascend", MoE "Forward").
//   gmm2 (grouped_gemm_mxfp8): y[r] = aq[r] . w2[e]^T, bf16 out.
//
// Design (one persistent CTA per SM, 576 threads, warp-specialized):
//   warp 0      producer: TMA (128B swizzle) loads of the A tile [128 x 128]
//               and the B tile [BN x 128] e4m3, plus cp.async of the e8m0
//               scales into the tensor-core scale-factor staging layout;
//               all land on one mbarrier per pipeline stage.
//   warp 1      MMA issuer (one thread): tcgen05.cp moves each stage's scale
//               factors from shared memory into tensor memory, then four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (M=128, N=BN, K=32,
//               UE8M0 scales, one scale per 32 K-elements) accumulate the
//               fp32 tile in tensor memory; tcgen05.commit frees the stage.
//   warps 2-17  epilogue: tcgen05.ld the accumulator into registers (one
//               thread per row and a quarter of the columns), release it to the
//               MMA warp, then SwiGLU + MX requant (gmm1) or bf16 rounding
//               (gmm2) and the stores, overlapping the next tile's mainloop.
// Tiles are scheduled per expert from the device-side offsets: the CTA reads
// offsets[0..E], builds the prefix of per-expert tile counts in shared
// memory and walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...  A tile that
// runs past its expert's last row computes rows of the next expert (or
// TMA zero fill past M) and masks them at the store.
//
// gmm1 stacks the gate and up rows of the same output columns into one
// B tile: rows [0, BN/2) = gate rows n0.., rows [BN/2, BN) = up rows I+n0..,
// so one N=256 MMA produces both halves and the epilogue pairs column c
// with column BN/2 + c.
//
// Every mbarrier wait has a clock-based limit; when it runs out the kernel
// records a timeout in the library status word, every role stops, in-flight
// copies and MMAs are drained with bounded waits, and tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tiled_scales.h"

namespace mxmoe {
namespace gemm {

constexpr int BM = 128;         // rows of A per tile (tokens)
constexpr int BK = 128;         // K elements (= bytes) per stage
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 16;  // epilogue warps (a multiple of 4)
constexpr int EPI_GROUPS = EPI_WARPS / 4;
constexpr int THREADS = 64 + 32 * EPI_WARPS;  // producer, MMA, epilogue
constexpr int MAX_E = 256;
constexpr int TMEM_COLS = 512;
constexpr int SF_COL0 = 256;    // scale factors after the accumulator
constexpr int SF_COLS_PER_STAGE = 16;
constexpr int ERR_TIMEOUT = 7;  // MXMOE_ERR_DEVICE_TIMEOUT

template <int BN_>
struct Layout {
  static constexpr int BN = BN_;
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFA_BYTES = 512;
  static constexpr int SFB_BYTES = (BN / 128) * 512;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
  // full[S], empty[S], acc_full, acc_empty, drain
  static constexpr int NUM_BARS = 2 * STAGES + 3;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem addr, abort flag
  static constexpr int OFF_OFFS = OFF_MISC + 16;            // int64 offsets [E+1]
  static constexpr int OFF_TS = OFF_OFFS + (MAX_E + 1) * 8; // int tile_start [E+1]
  static constexpr int OFF_MTB = OFF_TS + (MAX_E + 1) * 4;  // int m-tile base [E+1]
  static constexpr int BYTES = OFF_MTB + (MAX_E + 1) * 4;
  static constexpr int ALLOC = BYTES + 1024;                // 1 KB alignment slack
};

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
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
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

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), descriptor version 1 at bits 46-48, and
// the swizzle mode at bits 61-63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swizzle) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A and B e4m3
// (format 0 at bits 7-9 / 10-12), both K-major, N >> 3 at bits 17-22, UE8M0
// scale type (bit 23), M >> 4 at bits 24-28; the scale-factor byte selectors
// (bits 29-30 for A, 4-5 for B) are or-ed in per K step.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
  return ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}

// Bounded mbarrier wait.  Returns false when the CTA is aborting (another
// role timed out) or this wait ran out of time (then it starts the abort).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, long long limit,
                                         int* status, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) {
        report_error(status, ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
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

// kTiledSF: all scales (A, B and gmm1's output scales) use the tiled layout
// of tiled_scales.h and each stage's scale chunks arrive by bulk copy;
// otherwise they are the row-major [rows, K/32] arrays, staged by cp.async.
template <int BN, bool kSwiglu, bool kTiledSF>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const Params p) {
  using L = Layout<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  int64_t* s_off = reinterpret_cast<int64_t*>(smem + L::OFF_OFFS);
  int* s_ts = reinterpret_cast<int*>(smem + L::OFF_TS);
  int* s_mtb = reinterpret_cast<int*>(smem + L::OFF_MTB);
  auto bar_full = [&](int s) { return sbase + L::OFF_BAR + 8u * s; };
  auto bar_empty = [&](int s) { return sbase + L::OFF_BAR + 8u * (STAGES + s); };
  const uint32_t bar_acc_full = sbase + L::OFF_BAR + 8u * (2 * STAGES);
  const uint32_t bar_acc_empty = bar_acc_full + 8;
  const uint32_t bar_drain = bar_acc_full + 16;

  const int E = p.E;
  // ---- set-up: barriers, TMEM, tile schedule
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // producer expect_tx (+ 32 cp.async arrivals when scales come by cp.async)
      mbar_init(bar_full(s), kTiledSF ? 1 : 1 + 32);
      mbar_init(bar_empty(s), 1);      // tcgen05.commit
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, EPI_WARPS);  // one arrive per epilogue warp
    mbar_init(bar_drain, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {
    // per-expert tile counts -> exclusive prefix (E <= 256: 8 experts per lane)
    // and of m-tile counts (the tiled scale layout's per-expert block base)
    constexpr int PER = MAX_E / 32;
    int cnt[PER], mcnt[PER];
    int run = 0, mrun = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      int c = 0;
      if (e < E) {
        const int64_t o0 = p.offsets[e], o1 = p.offsets[e + 1];
        s_off[e] = o0;
        if (e == E - 1) s_off[E] = o1;
        c = (int)((o1 - o0 + BM - 1) / BM);
      }
      cnt[i] = run;
      mcnt[i] = mrun;
      run += c * p.n_tiles_n;
      mrun += c;
    }
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
      if (e < E) { s_ts[e] = excl + cnt[i]; s_mtb[e] = mexcl + mcnt[i]; }
    }
    if (lane == 31) { s_ts[E] = incl; s_mtb[E] = mincl; }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int total_tiles = s_ts[E];
  const int KT = p.K / BK;
  const int K32 = p.K / 32;

  if (warp == 0) {
    // ================= producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;  // per-stage bit masks, for the abort drain
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt;
      decode_tile(tile, s_ts, E, p.n_tiles_n, e, mt, nt);
      const int64_t row0 = s_off[e] + (int64_t)mt * BM;
      const int64_t brow = (int64_t)e * p.Nw;
      for (int kt = 0; kt < KT; ++kt) {
        const bool got = wait_bar(bar_empty(stage), phase ^ 1, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {  // keep the warp converged
          ok = false;
          break;
        }
        const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
        const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
        const uint32_t sSFA = sbase + L::OFF_SFA + stage * L::SFA_BYTES;
        const uint32_t sSFB = sbase + L::OFF_SFB + stage * L::SFB_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_full(stage), L::A_BYTES + L::B_BYTES +
                                                     (kTiledSF ? L::SFA_BYTES + L::SFB_BYTES : 0));
          tma_load_2d(sA, &tmA, kt * BK, (int)row0, bar_full(stage));
          if (kSwiglu) {
            tma_load_2d(sB, &tmB, kt * BK, (int)(brow + (int64_t)nt * (BN / 2)), bar_full(stage));
            tma_load_2d(sB + (BN / 2) * BK, &tmB, kt * BK,
                        (int)(brow + p.n_out + (int64_t)nt * (BN / 2)), bar_full(stage));
          } else {
            tma_load_2d(sB, &tmB, kt * BK, (int)(brow + (int64_t)nt * BN), bar_full(stage));
          }
          if (kTiledSF) {
            // one 512-byte chunk per 128 rows: A's m-tile block, B's row blocks
            bulk_copy_g2s(sSFA, p.sfa + ((int64_t)(s_mtb[e] + mt) * KT + kt) * 512, 512,
                          bar_full(stage));
#pragma unroll
            for (int c = 0; c < BN / 128; ++c) {
              int64_t wrow;
              if (kSwiglu)
                wrow = c == 0 ? brow + (int64_t)nt * (BN / 2) : brow + p.n_out + (int64_t)nt * (BN / 2);
              else
                wrow = brow + (int64_t)nt * BN + 128 * c;
              bulk_copy_g2s(sSFB + 512 * c, p.sfb + ((wrow >> 7) * KT + kt) * 512, 512,
                            bar_full(stage));
            }
          }
        }
        // scale factors: 4 bytes (4 K-blocks) per row, staged as
        // byte(r, kb) = (r % 32) * 16 + (r / 32) * 4 + kb per 128-row chunk
        if (!kTiledSF) {
#pragma unroll
        for (int i = 0; i < BM / 32; ++i) {
          const int r = lane + 32 * i;
          const int64_t grow = row0 + r;
          const bool valid = grow < p.M;
          const uint8_t* src = valid ? p.sfa + grow * K32 + kt * 4 : p.sfa;
          cp_async_4(sSFA + (r & 31) * 16 + (r >> 5) * 4, src, valid ? 4u : 0u);
        }
#pragma unroll
        for (int i = 0; i < BN / 32; ++i) {
          const int r = lane + 32 * i;
          int64_t wrow;
          if (kSwiglu)
            wrow = r < BN / 2 ? brow + (int64_t)nt * (BN / 2) + r
                              : brow + p.n_out + (int64_t)nt * (BN / 2) + (r - BN / 2);
          else
            wrow = brow + (int64_t)nt * BN + r;
          const int rr = r & 127;
          cp_async_4(sSFB + (r >> 7) * 512 + (rr & 31) * 16 + (rr >> 5) * 4,
                     p.sfb + wrow * K32 + kt * 4, 4u);
        }
        cp_async_mbar_arrive_noinc(bar_full(stage));
        }
        armed |= 1u << stage;
        if (phase) armed_parity |= 1u << stage; else armed_parity &= ~(1u << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok) {
      // drain: wait for this thread's cp.async and every armed stage's copies
      cp_async_wait_all();
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) {
          volatile int no_abort = 0;
          wait_bar(bar_full(s), (armed_parity >> s) & 1u, 1ll << 32, nullptr, &no_abort);
        }
    }
  } else if (warp == 1) {
    // ================= MMA issuer (one thread)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      constexpr uint32_t IDESC = make_idesc(BM, BN);
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!wait_bar(bar_acc_empty, acc_phase ^ 1, p.wait_limit, p.status, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt) {
          if (!wait_bar(bar_full(stage), phase, p.wait_limit, p.status, s_abort)) {
            ok = false;
            break;
          }
          if (!kTiledSF) fence_proxy_async_smem();  // cp.async-written scales -> async proxy
          tc_fence_after();
          const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
          const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
          const uint32_t sSFA = sbase + L::OFF_SFA + stage * L::SFA_BYTES;
          const uint32_t sSFB = sbase + L::OFF_SFB + stage * L::SFB_BYTES;
          const uint32_t t_sfa = tmem + SF_COL0 + stage * SF_COLS_PER_STAGE;
          const uint32_t t_sfb = t_sfa + 4;
          tc_cp_sf(t_sfa, make_sdesc(sSFA, 128, 128, 0));
#pragma unroll
          for (int c = 0; c < BN / 128; ++c) tc_cp_sf(t_sfb + 4 * c, make_sdesc(sSFB + 512 * c, 128, 128, 0));
          const uint64_t adesc = make_sdesc(sA, 16, 1024, 2);
          const uint64_t bdesc = make_sdesc(sB, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t idesc = IDESC | ((uint32_t)kk << 29) | ((uint32_t)kk << 4);
            tc_mma_mxf8(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, t_sfa, t_sfb,
                        (kt | kk) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(bar_empty(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(bar_acc_full);
        acc_phase ^= 1;
      }
      if (!ok && issued) {
        // drain: every MMA and copy issued so far completes before TMEM is freed
        tc_commit(bar_drain);
        volatile int no_abort = 0;
        wait_bar(bar_drain, 0, 1ll << 32, nullptr, &no_abort);
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue: EPI_WARPS warps, EPI_GROUPS per TMEM lane
    // quarter (warp & 3 = quarter; group g takes the g-th slice of the
    // columns).  Each thread drains its row's slice of the accumulator into
    // registers, releases the accumulator to the MMA warp at once, and only
    // then does the math and the stores, so the epilogue of tile i overlaps
    // the mainloop of tile i+1.
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    // columns per thread: SwiGLU -> GC gate + GC up columns; plain -> PC
    constexpr int GC = BN / 2 / EPI_GROUPS;
    constexpr int PC = BN / EPI_GROUPS;
    constexpr int CH = kSwiglu ? 2 * (GC / 32) : PC / 32;  // 32-column chunks
    static_assert(kSwiglu ? GC % 32 == 0 : PC % 32 == 0, "epilogue slices are whole 32-column chunks");
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt;
      decode_tile(tile, s_ts, E, p.n_tiles_n, e, mt, nt);
      const int64_t grow = s_off[e] + (int64_t)mt * BM + row;
      const bool valid = grow < s_off[e + 1];
      const bool got = wait_bar(bar_acc_full, acc_phase, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) break;  // keep the warp converged
      tc_fence_after();
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
      if (lane == 0) mbar_arrive(bar_acc_empty);
      acc_phase ^= 1;
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
          const uint32_t sb = e8m0_from_amax_bits(m);
          const float inv = inv_scale_from_e8m0(sb);
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o[i] = cvt_e4m3x4(a[4 * i] * inv, a[4 * i + 1] * inv, a[4 * i + 2] * inv,
                              a[4 * i + 3] * inv);
          if (valid) {
            const int64_t col = (int64_t)nt * (BN / 2) + grp * GC + c * 32;
            st_v8(aq + grow * p.n_out + col, o);
            if (kTiledSF)
              p.out_scale[tiled_scale_offset((int64_t)(s_mtb[e] + mt) * BM + row, (int)(col >> 5),
                                             p.n_out / 128)] = (uint8_t)sb;
            else
              p.out_scale[grow * (p.n_out / 32) + (col >> 5)] = (uint8_t)sb;
          }
        }
      } else {
        uint16_t* y = reinterpret_cast<uint16_t*>(p.out);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            o[i] = cvt_bf16x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1]));
          if (valid) {
            uint16_t* dst = y + grow * p.n_out + (int64_t)nt * BN + grp * PC + c * 32;
            st_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(&o[0]));
            st_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(&o[8]));
          }
        }
      }
    }
  }

  // ---- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2D uint8 tensor [outer, inner] (inner contiguous), 128-byte swizzled box.
static bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                     uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, bool kSwiglu, bool kTiledSF>
static cudaError_t launch(const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                          const uint8_t* sfb, const int64_t* offsets, int64_t M, int E, int K,
                          int Nw, int n_out, void* out, uint8_t* out_scale, cudaStream_t stream) {
  using L = Layout<BN>;
  if (M == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  const uint32_t b_box_rows = kSwiglu ? BN / 2 : BN;
  if (!make_map(&tmA, a, (uint64_t)K, (uint64_t)M, BK, BM)) return cudaErrorInvalidValue;
  if (!make_map(&tmB, b, (uint64_t)K, (uint64_t)E * Nw, BK, b_box_rows))
    return cudaErrorInvalidValue;
  Params p;
  p.sfa = sfa;
  p.sfb = sfb;
  p.offsets = offsets;
  p.out = out;
  p.out_scale = out_scale;
  p.M = M;
  p.E = E;
  p.K = K;
  p.Nw = Nw;
  p.n_out = n_out;
  p.n_tiles_n = kSwiglu ? n_out / (BN / 2) : n_out / BN;
  p.status = device_status_ptr();
  p.wait_limit = wait_limit_cycles();
  auto kern = grouped_gemm_kernel<BN, kSwiglu, kTiledSF>;
  static int configured_dev = -1;  // smem attribute is per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (err != cudaSuccess) return err;
    configured_dev = dev;
  }
  const int64_t tiles_bound = (ceil_div(M, BM) + E) * (int64_t)p.n_tiles_n;
  const int grid = (int)std::min<int64_t>(tiles_bound, num_sms());
  kern<<<grid, THREADS, L::ALLOC, stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

}  // namespace gemm

cudaError_t launch_gemm_swiglu_quant(const uint8_t* xq, const uint8_t* xs, const uint8_t* w13q,
                                     const uint8_t* w13s, const int64_t* offsets, int64_t M,
                                     int E, int H, int I, uint8_t* aq, uint8_t* as,
                                     cudaStream_t stream, bool tiled_scales) {
  if (tiled_scales)
    return gemm::launch<256, true, true>(xq, xs, w13q, w13s, offsets, M, E, H, 2 * I, I, aq, as,
                                         stream);
  return gemm::launch<256, true, false>(xq, xs, w13q, w13s, offsets, M, E, H, 2 * I, I, aq, as,
                                        stream);
}

cudaError_t launch_gemm_bf16(const uint8_t* aq, const uint8_t* as, const uint8_t* w2q,
                             const uint8_t* w2s, const int64_t* offsets, int64_t M, int E,
                             int I, int H, uint16_t* y, cudaStream_t stream, bool tiled_scales) {
  if (H % 256 == 0) {
    if (tiled_scales)
      return gemm::launch<256, false, true>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y, nullptr,
                                            stream);
    return gemm::launch<256, false, false>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y, nullptr,
                                           stream);
  }
  if (tiled_scales)
    return gemm::launch<128, false, true>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y, nullptr,
                                          stream);
  return gemm::launch<128, false, false>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y, nullptr,
                                         stream);
}

}  // namespace mxmoe
