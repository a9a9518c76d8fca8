// 2-SM grouped MXFP8 GEMM (tcgen05 cta_group::2) for 256-wide tiles with
// scales in the tiled layout of tiled_scales.h; same contract as the 1-SM
// kernel of gemm.cu, and bit-identical results.
//
// A cluster of two CTAs (on two SMs) computes a 256 x 256 tile: CTA r holds
// m-tile 2u + r of the work unit's expert (128 token rows) and half r of the
// 256 weight rows, in its own shared memory; one tcgen05.mma.cta_group::2
// (M = 256, N = 256, K = 32) issued by the even CTA reads both CTAs' operands
// and accumulates each CTA's 128 rows x 256 columns in that CTA's TMEM.  Per
// 128-K stage each SM stages 32 KB (A 16 KB + half of B 16 KB) instead of the
// 1-SM tile's 48 KB, so the pair pulls a third less from L2 per FLOP and six
// stages fit where the 1-SM ring holds four.
//
// Roles (704 threads per CTA, as in the 1-SM kernel): warp 0 producer, warp 1
// MMA issuer (even CTA only), warps 2-5 scale-factor writers (tcgen05.st, one
// per TMEM lane quarter), warps 6-21 epilogue.
//
// Synchronization (every wait bounded, as in the 1-SM kernel):
//   full[s]     in the leader, count 1: the leader's producer arms it with
//               both CTAs' operand bytes; every operand TMA load of both
//               CTAs (.cta_group::2 form) completes on it.  A peer load may
//               land before the leader arms the phase; the pending arrival
//               keeps the phase open until then.
//   sf_full[s]  in each CTA, count 1: that CTA's scale chunks (bulk copies).
//   sf_ready[s] in the leader, count 2 x SF_WARPS: the scale writers of both
//               CTAs, once their TMEM stores of stage s are complete.
//   empty[s]    in each CTA; the leader's tcgen05.commit is multicast to both.
//   acc_full    in each CTA; likewise.
//   acc_empty   in the leader, count 2 x EPI_WARPS: every epilogue warp of
//               both CTAs, once it has drained its accumulator slice.
// Each CTA's TMEM holds the scales of its own 128 A rows and of all 256 B
// rows (both CTAs stage the B rows' scale chunks).
#include "gemm_common.cuh"

namespace mxmoe {
namespace gemm {

constexpr int STAGES2 = 6;
constexpr int SEG2 = 8;           // k-slices per scale segment
constexpr int SEG2_COLS = 128;    // TMEM columns per segment buffer (16 per k-slice)

struct Layout2 {
  static constexpr int S = STAGES2;
  static constexpr int A_BYTES = BM * BK;          // own 128 rows
  static constexpr int B_BYTES = 128 * BK;         // own half of the 256 weight rows
  static constexpr int SFA_SEG = SEG2 * 512;       // own A rows: one chunk per k-slice
  static constexpr int SFB_SEG = 2 * SEG2 * 512;   // both 128-row blocks of B
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + S * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + S * B_BYTES;     // [2] segments
  static constexpr int OFF_SFB = OFF_SFA + 2 * SFA_SEG;   // [2] segments
  static constexpr int OFF_BAR = OFF_SFB + 2 * SFB_SEG;
  // full[S], empty[S], acc_full, acc_empty, drain,
  // sfs_full[2], sfs_free[2], sft_ready[2], sft_free[2]
  static constexpr int NUM_BARS = 2 * S + 3 + 8;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem addr, abort flag
  static constexpr int OFF_OFFS = OFF_MISC + 16;
  static constexpr int OFF_TS = OFF_OFFS + (MAX_E + 1) * 8;
  static constexpr int OFF_MTB = OFF_TS + (MAX_E + 1) * 4;
  static constexpr int BYTES = OFF_MTB + (MAX_E + 1) * 4;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ALLOC <= 232448, "shared memory");
  static_assert(SF_COL0 + 2 * SEG2_COLS <= TMEM_COLS, "tensor memory");
};

// ---------------------------------------------------------------- cta_group::2 PTX

// TMA tile load into this CTA's shared memory that completes on an mbarrier
// of either CTA of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals come from both CTAs).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, long long limit,
                                                 int* status, volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      report_error(status, ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void tc2_mma_mxf4(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tc2_mma_mxf8(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
// Arrive on the barrier at `bar`'s offset in both CTAs once all prior
// tcgen05 operations of this thread have completed.
__device__ __forceinline__ void tc2_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)0x3)
      : "memory");
}

template <bool kSwiglu, int kFmt>
__global__ void __launch_bounds__(THREADS1, 1)
    gemm2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const Params p) {
  using L = Layout2;
  constexpr int STAGES = L::S;
  constexpr int BN = 256;
  constexpr bool kFp4B = kFmt != FMT_W8A8, kFp4A = kFmt == FMT_W4A4;
  // W4A4: kind::mxf4 on packed operands (as in the 1-SM kernel): 256 K
  // elements and two scale chunks per k-slice, four K = 64 MMAs
  constexpr bool kPacked = kFmt == FMT_W4A4;
  constexpr int CH = kPacked ? 2 : 1;
  constexpr int SEGK = SEG2 / CH;
  constexpr int SLICE_COLS = SF_COLS_PER_STAGE * CH;
  constexpr int MPC = (BK / 32) / CH;
  static_assert(SEGK * SLICE_COLS == SEG2_COLS, "segment columns");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

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
  // scale segments: this CTA's smem buffer landed / copied out (local), TMEM
  // buffers of both CTAs written (leader) / consumed (multicast commit)
  auto bar_sfs_full = [&](int b) { return bar_acc_full + 24 + 8u * b; };
  auto bar_sfs_free = [&](int b) { return bar_acc_full + 40 + 8u * b; };
  auto bar_sft_ready = [&](int b) { return bar_acc_full + 56 + 8u * b; };
  auto bar_sft_free = [&](int b) { return bar_acc_full + 72 + 8u * b; };

  const int E = p.E;
  const int unit0 = blockIdx.x >> 1;  // cluster index
  const int unit_step = gridDim.x >> 1;
  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);              // leader: its producer's expect_tx
      mbar_init(bar_empty(s), 1);             // the leader's multicast commit
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, 2 * EPI_WARPS);  // leader: every epilogue warp of both CTAs
    mbar_init(bar_drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_sfs_full(b), 1);          // this CTA's producer's expect_tx
      mbar_init(bar_sfs_free(b), SF_WARPS);   // this CTA's scale writers
      mbar_init(bar_sft_ready(b), 2 * SF_WARPS);  // leader: scale writers of both CTAs
      mbar_init(bar_sft_free(b), 1);          // the leader's multicast commit
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    // both CTAs' warps allocate together (same columns in each TMEM)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // programmatic serialization: the set-up above overlaps the previous
  // kernel's tail; its outputs are read only after this wait
  pdl_launch_dependents();
  pdl_wait();
  if (warp == 2) build_schedule<2>(p, lane, s_off, s_ts, s_mtb);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialized before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int total_units = s_ts[E];
  // k-slices; a partial last slice is zero-filled by TMA
  const int KT = (p.K + BK * CH - 1) / (BK * CH);
  const int KTC = (p.K + BK - 1) / BK;  // 128-element scale chunks per row block
  const int nseg = (KT + SEGK - 1) / SEGK;  // scale segments per unit
  // the leader's barriers as seen from this CTA
  const uint32_t lead_full0 = mapa_cluster(bar_full(0), 0);
  const uint32_t lead_sftr0 = mapa_cluster(bar_sft_ready(0), 0);
  const uint32_t lead_acc_empty = mapa_cluster(bar_acc_empty, 0);

  // B row blocks of a unit: gmm1 = gate rows | up rows, gmm2 = 256 rows
  auto unit_rows = [&](int unit, int& e, int& mt, int& nt, int64_t& bh0, int64_t& bh1) {
    decode_tile(unit, s_ts, E, p.n_tiles_n, e, mt, nt);
    mt = 2 * mt + (int)rank;  // this CTA's m-tile of the unit's pair
    const int64_t brow = (int64_t)e * p.Nw;
    bh0 = kSwiglu ? brow + (int64_t)nt * (BN / 2) : brow + (int64_t)nt * BN;
    bh1 = kSwiglu ? brow + p.n_out + (int64_t)nt * (BN / 2) : bh0 + BN / 2;
  };

  if (warp == 0) {
    // ================= producer (both CTAs): operand stages, and each unit
    // segment's scales (this CTA's A rows, all 256 B rows) one segment ahead
    int stage = 0;
    uint32_t phase = 0;
    int g = 0;
    bool ok = true;
    int req_hi = -1;  // the last scale segment requested
    auto load_scales = [&](int gseg, int unit, int sg) -> bool {
      const int b = gseg & 1;
      const uint32_t par = ((uint32_t)(gseg >> 1) & 1u) ^ 1u;
      const bool got = wait_bar(bar_sfs_free(b), par, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) return false;
      req_hi = gseg;
      if (lane == 0) {
        int e, mt, nt;
        int64_t bh0, bh1;
        unit_rows(unit, e, mt, nt, bh0, bh1);
        // tiled A scales: the m-tile's block (a CTA without rows reads its expert's last block)
        const int64_t a_blk = min(s_mtb[e] + mt, s_mtb[e + 1] - 1);
        const int kt0 = sg * SEGK, len = min(SEGK, KT - kt0);
        // the segment's scale chunks (a packed last k-slice may hold only one)
        const int c0 = kt0 * CH, nch = min(len * CH, KTC - c0);
        const uint32_t sA = sbase + L::OFF_SFA + b * L::SFA_SEG;
        const uint32_t sB = sbase + L::OFF_SFB + b * L::SFB_SEG;
        mbar_arrive_expect_tx(bar_sfs_full(b), (uint32_t)(3 * nch * 512));
        bulk_copy_g2s(sA, p.sfa + (a_blk * KTC + c0) * 512, (uint32_t)(nch * 512),
                      bar_sfs_full(b));
        bulk_copy_g2s(sB, p.sfb + ((bh0 >> 7) * KTC + c0) * 512, (uint32_t)(nch * 512),
                      bar_sfs_full(b));
        bulk_copy_g2s(sB + SEG2 * 512, p.sfb + ((bh1 >> 7) * KTC + c0) * 512,
                      (uint32_t)(nch * 512), bar_sfs_full(b));
      }
      __syncwarp();
      return true;
    };
    if (unit0 < total_units) ok = load_scales(0, unit0, 0);
    for (int unit = unit0; ok && unit < total_units; unit += unit_step) {
      int e, mt, nt;
      int64_t bh0, bh1;
      unit_rows(unit, e, mt, nt, bh0, bh1);
      const int64_t row0 = s_off[e] + (int64_t)mt * BM;
      for (int kt = 0; kt < KT; ++kt) {
        if (kt % SEGK == 0) {
          const int sg = kt / SEGK;
          const int nunit = sg + 1 < nseg ? unit : unit + unit_step;
          if (nunit < total_units && !load_scales(g + 1, nunit, sg + 1 < nseg ? sg + 1 : 0)) {
            ok = false;
            break;
          }
          ++g;
        }
        const bool got = wait_bar(bar_empty(stage), phase ^ 1, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          // W4A8's unpacked FP4 B counts its global (packed) bytes: half its
          // smem footprint; packed W4A4 operands land byte for byte
          if (leader)
            mbar_arrive_expect_tx(bar_full(stage),
                                  2 * (L::A_BYTES +
                                       (kFp4B && !kPacked ? L::B_BYTES / 2 : L::B_BYTES)));
          const uint32_t fb = lead_full0 + 8u * stage;  // leader's full[stage]
          const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
          const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
          tma_load_2d_pair(sA, &tmA, kt * BK, (int)row0, fb);
          tma_load_2d_pair(sB, &tmB, kt * BK, (int)(rank ? bh1 : bh0), fb);
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (ok) {
      // tail: wait until the leader's MMAs have released every stage this CTA
      // loaded, so no commit of the pair is still on its way to this CTA
      for (int i = 0; i < STAGES; ++i) {
        wait_bar(bar_empty(stage), phase ^ 1, p.wait_limit, p.status, s_abort);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    } else {
      // abort: this CTA's scale copies land on its own barriers (wait for the
      // last two segments requested); its operand loads complete on the
      // leader's barriers, so give them a bounded moment to land before the
      // CTA pair tears down
      volatile int no_abort = 0;
      for (int sg = req_hi - 1; sg <= req_hi; ++sg)
        if (sg >= 0)
          wait_bar(bar_sfs_full(sg & 1), (uint32_t)(sg >> 1) & 1u, 1ll << 32, nullptr,
                   &no_abort);
      const long long t0 = clock64();
      while (clock64() - t0 < 200000) __nanosleep(1000);
    }
  } else if (warp == 1) {
    // ================= MMA issuer: one thread of the leader CTA
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      int g = 0;
      bool ok = true;
      bool issued = false;
      constexpr uint32_t IDESC =
          kPacked ? make_idesc_mxf4(2 * BM, BN) : make_idesc(2 * BM, BN, kFp4B);
      for (int unit = unit0; ok && unit < total_units; unit += unit_step) {
        if (!wait_bar_cluster(bar_acc_empty, acc_phase ^ 1, p.wait_limit, p.status, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt) {
          const int i = kt % SEGK;
          const int b = g & 1;
          // both CTAs' scales of this segment are in TMEM buffer b
          if (i == 0 && !wait_bar_cluster(bar_sft_ready(b), (uint32_t)(g >> 1) & 1u,
                                          p.wait_limit, p.status, s_abort)) {
            ok = false;
            break;
          }
          // both CTAs' operands landed
          if (!wait_bar(bar_full(stage), phase, p.wait_limit, p.status, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
          const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
          // scale columns of k-slice i as in the 1-SM kernel (B chunk j:
          // 8 columns, both 128-row blocks)
          const uint32_t t_sf = tmem + SF_COL0 + b * SEG2_COLS + i * SLICE_COLS;
          const uint64_t adesc = make_sdesc(sA, 16, 1024, 2);
          const uint64_t bdesc = make_sdesc(sB, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            if (kPacked && (kt * (BK / 32) + kk) * 64 >= p.K) break;  // packed K tail
            const int j = kk / MPC;
            const uint32_t sfid = (uint32_t)((kk % MPC) * CH);
            const uint32_t idesc = IDESC | (sfid << 29) | (sfid << 4);
            const uint32_t t_sfa = t_sf + 4 * j, t_sfb = t_sf + 4 * CH + 8 * j;
            const uint32_t acc = (kt | kk) != 0 ? 1u : 0u;
            if constexpr (kPacked)
              tc2_mma_mxf4(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, t_sfa, t_sfb, acc);
            else
              tc2_mma_mxf8(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, t_sfa, t_sfb, acc);
          }
          issued = true;
          tc2_commit_both(bar_empty(stage));
          if (i == SEGK - 1 || kt == KT - 1) {
            tc2_commit_both(bar_sft_free(b));  // the segment's scales may be overwritten
            ++g;
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc2_commit_both(bar_acc_full);
        acc_phase ^= 1;
      }
      if (ok) {
        // the last tile's releases (some from the peer CTA) land before exit
        wait_bar_cluster(bar_acc_empty, acc_phase ^ 1, p.wait_limit, p.status, s_abort);
      } else if (issued) {
        tc2_commit_both(bar_drain);
        volatile int no_abort = 0;
        wait_bar(bar_drain, 0, 1ll << 32, nullptr, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp < EPI_WARP0) {
    // ================= scale-factor writers (both CTAs), one per TMEM lane
    // quarter: a segment's staged chunks (this CTA's A rows, all 256 B rows)
    // go into this CTA's TMEM (tcgen05.st, the layout of the 1-SM kernel)
    // once the pair's MMAs are done with the buffer; the leader's MMA waits
    // for the writers of both CTAs.
    const uint32_t t_q = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int g = 0;
    bool ok = true;
    for (int unit = unit0; ok && unit < total_units; unit += unit_step) {
      for (int sg = 0; sg < nseg; ++sg, ++g) {
        const int b = g & 1;
        const uint32_t par = (uint32_t)(g >> 1) & 1u;
        const bool got = wait_bar(bar_sfs_full(b), par, p.wait_limit, p.status, s_abort) &&
                         wait_bar(bar_sft_free(b), par ^ 1u, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const int len = min(SEGK, KT - sg * SEGK);
        const uint8_t* sfa_s = smem + L::OFF_SFA + b * L::SFA_SEG;
        const uint8_t* sfb_s = smem + L::OFF_SFB + b * L::SFB_SEG;
        // (a chunk past K is never copied in; its columns are never read)
        for (int i = 0; i < len; ++i) {
          const uint32_t col = SF_COL0 + b * SEG2_COLS + i * SLICE_COLS;
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            const int ch = i * CH + j;
            tmem_st_4(t_q + col + 4 * j,
                      *reinterpret_cast<const uint4*>(sfa_s + ch * 512 + lane * 16));
            tmem_st_4(t_q + col + 4 * CH + 8 * j,
                      *reinterpret_cast<const uint4*>(sfb_s + ch * 512 + lane * 16));
            tmem_st_4(t_q + col + 4 * CH + 8 * j + 4,
                      *reinterpret_cast<const uint4*>(sfb_s + SEG2 * 512 + ch * 512 + lane * 16));
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(bar_sft_ready(b));
          else mbar_arrive_cluster(lead_sftr0 + 8u * b);
          mbar_arrive(bar_sfs_free(b));
        }
      }
    }
  } else {
    // ================= epilogue (both CTAs): EPI_GROUPS warps per TMEM lane quarter
    const int q = warp & 3;
    const int grp = (warp - EPI_WARP0) >> 2;
    const int row = q * 32 + lane;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t acc_phase = 0;
    for (int unit = unit0; unit < total_units; unit += unit_step) {
      int e, mt, nt;
      decode_tile(unit, s_ts, E, p.n_tiles_n, e, mt, nt);
      mt = 2 * mt + (int)rank;
      const int64_t grow = s_off[e] + (int64_t)mt * BM + row;
      const bool valid = grow < s_off[e + 1];
      const bool got = wait_bar(bar_acc_full, acc_phase, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      epilogue_tile<BN, kSwiglu, true, kFp4A, false>(
          p, t_row, grp, row, lane, grow, valid, nt, (int64_t)(s_mtb[e] + mt) * BM + row,
          [&] {
            if (lane == 0) {
              if (leader) mbar_arrive(bar_acc_empty);
              else mbar_arrive_cluster(lead_acc_empty);
            }
          });
      acc_phase ^= 1;
    }
  }

  // ---- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side

template <bool kSwiglu, int kFmt>
cudaError_t launch_pair_impl(const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                             const uint8_t* sfb, const int64_t* offsets, int64_t M, int E, int K,
                             int Nw, int n_out, void* out, uint8_t* out_scale,
                             cudaStream_t stream) {
  using L = Layout2;
  if (M == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static int max_clusters[64];
  static uint64_t configured[64] = {0};  // context id the attribute was set in
  auto kern = gemm2sm_kernel<kSwiglu, kFmt>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(THREADS1, 1, 1);
  cfg.dynamicSmemBytes = L::ALLOC;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint64_t ctx = context_id();
  if (ctx == 0 || configured[dev] != ctx) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (err != cudaSuccess) return err;
    cfg.gridDim = dim3(2 * 64, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    max_clusters[dev] = n;
    configured[dev] = context_id();
  }
  if (max_clusters[dev] <= 0) return cudaErrorNotSupported;
  CUtensorMap tmA, tmB;
  const uint64_t inner = kFmt == FMT_W4A4 ? (uint64_t)K / 2 : (uint64_t)K;  // packed W4A4 bytes
  if (!make_map(&tmA, a, inner, (uint64_t)M, BK, BM))
    return cudaErrorInvalidValue;
  if (!make_map(&tmB, b, inner, (uint64_t)E * Nw, BK, 128, kFmt == FMT_W4A8))
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
  p.n_tiles_n = kSwiglu ? n_out / 128 : (int)ceil_div(n_out, 256);
  p.ksplit = 1;
  p.partial = nullptr;
  p.pf_b = nullptr;
  p.pf_row_bytes = 0;
  p.status = device_status_ptr();
  p.wait_limit = wait_limit_cycles();
  const int64_t units_bound = (ceil_div(M, BM) / 2 + E) * (int64_t)p.n_tiles_n;
  const int clusters = (int)std::min<int64_t>(
      {units_bound, (int64_t)max_clusters[dev], (int64_t)num_sms() / 2});
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.numAttrs = 2;  // the cluster shape (as queried above) + programmatic serialization
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
}

template <bool kSwiglu, bool kTiledSF, int kFmt>
cudaError_t launch_pair(const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                        const uint8_t* sfb, const int64_t* offsets, int64_t M, int E, int K,
                        int Nw, int n_out, void* out, uint8_t* out_scale, cudaStream_t stream) {
  if (!kTiledSF) return cudaErrorNotSupported;  // scale chunks arrive by bulk copy
  return launch_pair_impl<kSwiglu, kFmt>(a, sfa, b, sfb, offsets, M, E, K, Nw, n_out, out,
                                          out_scale, stream);
}

#define MXMOE_PAIR_INSTANCE(SW, TL, F4)                                                           \
  template cudaError_t launch_pair<SW, TL, F4>(const uint8_t*, const uint8_t*, const uint8_t*,  \
                                               const uint8_t*, const int64_t*, int64_t, int, int, \
                                               int, int, void*, uint8_t*, cudaStream_t);
MXMOE_PAIR_INSTANCE(true, true, FMT_W8A8)
MXMOE_PAIR_INSTANCE(false, true, FMT_W8A8)
MXMOE_PAIR_INSTANCE(true, false, FMT_W8A8)
MXMOE_PAIR_INSTANCE(false, false, FMT_W8A8)
MXMOE_PAIR_INSTANCE(true, true, FMT_W4A8)
MXMOE_PAIR_INSTANCE(false, true, FMT_W4A8)
MXMOE_PAIR_INSTANCE(true, true, FMT_W4A4)
MXMOE_PAIR_INSTANCE(false, true, FMT_W4A4)
#undef MXMOE_PAIR_INSTANCE

}  // namespace gemm
}  // namespace mxmoe
