// Grouped MXFP8 GEMMs of the MoE expert forward on 5th-generation tensor
// cores (tcgen05, sm_103a).
//
//   gmm1 (grouped_gemm_swiglu_quant_mxfp8): per expert e, rows r of
//        [off_e, off_{e+1}): h = xq[r] . w13[e]^T, a = silu(h_gate) * h_up,
//        requantized to MXFP8 along I (PR #30768 report,
//        GroupedMatmulSwigluQuant; "Quantization on Ascend", MoE "Forward").
//   gmm2 (grouped_gemm_mxfp8): y[r] = aq[r] . w2[e]^T, bf16 out.
//
// Two kernels share this pipeline: the 1-SM kernel here (the default) and
// an opt-in 2-SM kernel in gemm2sm.cu (tcgen05 cta_group::2, M = 256 over a
// CTA pair).
//
// Design of the 1-SM kernel (one persistent CTA per SM, 704 threads, warp-specialized):
//   warp 0      producer: TMA (128B swizzle) loads of the A tile [128 x 128]
//               and the B tile [BN x 128] e4m3, plus the e8m0 scale chunks
//               (bulk copies of the tiled layout, or cp.async of [rows, K/32]
//               scales into the same staging layout); all land on one mbarrier
//               per pipeline stage.
//   warps 2-5   scale-factor writers, one per TMEM lane quarter: tcgen05.st
//               moves each stage's staged scales into tensor memory.
//   warp 1      MMA issuer (one thread): four
//               tcgen05.mma.kind::mxf8f6f4.block_scale (M=128, N=BN, K=32,
//               UE8M0 scales, one scale per 32 K-elements) accumulate the
//               fp32 tile in tensor memory; tcgen05.commit frees the stage.
//               W4A4 takes kind::mxf4 on packed e2m1 operands instead: a
//               128-byte stage then holds 256 K elements, four K=64 MMAs
//               with two scales per row each (scale_vec::2X).
//   warps 6-21  epilogue: tcgen05.ld the accumulator into registers (one
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
#include <cmath>

#include "gemm_common.cuh"

namespace mxmoe {
namespace gemm {

constexpr int STAGES1 = 4;
constexpr int SEG = 8;           // k-slices per scale segment
constexpr int SEG_COLS = 128;    // TMEM columns per segment buffer (16 per k-slice)

// BMA: A rows staged per stage (the TMA box).  128 = the whole m-tile.  When
// every group has at most BMA_SMALL rows (small batches: an expert's rows
// are at most the token count), only the first BMA_SMALL rows of each tile
// are loaded; the MMA still reads 128 rows from the stage's address on, the
// rows past BMA_SMALL are whatever shared memory holds there and only ever
// reach accumulator rows past the group's end, which the epilogue masks.
// The 12 KB saved per stage buy a fifth stage: more weight bytes in flight.
constexpr int BMA_SMALL = 32;

template <int BN_, int BMA = BM>
struct Layout1 {
  static constexpr int BN = BN_;
  static constexpr int S = BMA == BM ? STAGES1 : STAGES1 + 1;
  static constexpr int A_BYTES = BMA * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int SFA_SEG = SEG * 512;               // one 512-byte chunk per k-slice
  static constexpr int SFB_SEG = (BN / 128) * SEG * 512;  // per 128-row block of B
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + S * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + S * B_BYTES;     // [2] segments
  static constexpr int OFF_SFB = OFF_SFA + 2 * SFA_SEG;   // [2] segments
  static constexpr int OFF_BAR = OFF_SFB + 2 * SFB_SEG;
  // full[S], empty[S], acc_full, acc_empty, drain,
  // sfs_full[2], sfs_free[2], sft_ready[2], sft_free[2]
  static constexpr int NUM_BARS = 2 * S + 3 + 8;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem addr, abort flag
  static constexpr int OFF_OFFS = OFF_MISC + 16;            // int64 offsets [E+1]
  static constexpr int OFF_TS = OFF_OFFS + (MAX_E + 1) * 8; // int unit start [E+1]
  static constexpr int OFF_MTB = OFF_TS + (MAX_E + 1) * 4;  // int m-tile base [E+1]
  static constexpr int BYTES = OFF_MTB + (MAX_E + 1) * 4;
  static constexpr int ALLOC = BYTES + 1024;                // 1 KB alignment slack
  static_assert(ALLOC <= 232448, "shared memory");
  static_assert(SF_COL0 + 2 * SEG_COLS <= TMEM_COLS, "tensor memory");
};

// Small batches: before the routing results exist, guess this CTA's first
// unit (unit blockIdx.x with one m-tile per expert: expert u / n-tiles,
// n-tile u % n-tiles) and start its weight rows (gmm1: the gate and the up
// block) and their tiled scales into L2, one 64 KB piece per lane of the
// calling warp.  The weights are inputs of the layer call, written before
// its first kernel started; rows outside [0, E * Nw) are never touched.
template <int BN, bool kSwiglu>
__device__ __forceinline__ void prefetch_first_unit(const Params& p, int lane) {
  const int e = (int)blockIdx.x / p.n_tiles_n, nt = (int)blockIdx.x % p.n_tiles_n;
  const int64_t brow = (int64_t)e * p.Nw;
  const int64_t r0 = kSwiglu ? brow + (int64_t)nt * (BN / 2) : brow + (int64_t)nt * BN;
  const int64_t r1 = brow + p.n_out + (int64_t)nt * (BN / 2);
  const int64_t nrows = kSwiglu ? BN / 2 : BN;  // per block
  const int64_t rows_all = (int64_t)p.E * p.Nw;
  const int KTC = (p.K + BK - 1) / BK;
  if (e >= p.E || r0 + nrows > rows_all || (kSwiglu && r1 + nrows > rows_all)) return;
  constexpr int64_t kPiece = 64 << 10;
  const int64_t blk_bytes = nrows * p.pf_row_bytes;
  const int64_t per_blk = (blk_bytes + kPiece - 1) / kPiece;
  const int nblk = kSwiglu ? 2 : 1;
  for (int64_t i = lane; i < nblk * per_blk; i += 32) {
    const int64_t bi = i / per_blk, o = (i - bi * per_blk) * kPiece;
    prefetch_l2_bulk(p.pf_b + (bi == 0 ? r0 : r1) * p.pf_row_bytes + o,
                     (uint32_t)min(kPiece, blk_bytes - o));
  }
  // the tiled scales of the 128-row blocks (KTC chunks of 512 bytes each)
  if (lane == 31)
    prefetch_l2_bulk(p.sfb + (r0 >> 7) * KTC * 512, (uint32_t)((nrows / 128) * KTC * 512));
  if (kSwiglu && lane == 30) prefetch_l2_bulk(p.sfb + (r1 >> 7) * KTC * 512, (uint32_t)(KTC * 512));
}

// kTiledSF: all scales (A, B and gmm1's output scales) use the tiled layout
// of tiled_scales.h (a segment's chunks are contiguous: one bulk copy per 128
// rows); otherwise they are the row-major [rows, K/32] arrays, gathered into
// the same staging layout by cp.async.
// kSplit: split-K tiles (Params::ksplit); the other instantiations fold the
// split arithmetic away.
template <int BN, bool kSwiglu, bool kTiledSF, int kFmt, bool kSplit, int BMA = BM>
__global__ void __launch_bounds__(THREADS1, 1)
    gemm1sm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const Params p) {
  using L = Layout1<BN, BMA>;
  static_assert(BMA == BM || kTiledSF, "short A boxes take tiled scales");
  constexpr int STAGES = L::S;
  constexpr bool kFp4B = kFmt != FMT_W8A8, kFp4A = kFmt == FMT_W4A4;
  // W4A4: kind::mxf4 on packed operands, so a 128-byte k-slice holds 256
  // K elements (two 128-element scale chunks) and takes four K = 64 MMAs
  constexpr bool kPacked = kFmt == FMT_W4A4;
  constexpr int CH = kPacked ? 2 : 1;          // scale chunks per k-slice
  constexpr int SEGK = SEG / CH;               // k-slices per scale segment
  constexpr int SLICE_COLS = SF_COLS_PER_STAGE * CH;  // TMEM scale columns per k-slice
  constexpr int MPC = (BK / 32) / CH;          // MMAs per scale chunk
  static_assert(!kPacked || kTiledSF, "packed operands take tiled scales");
  static_assert(SEGK * SLICE_COLS == SEG_COLS, "segment columns");
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
  // scale segments: smem buffer landed / copied out, TMEM buffer written / consumed
  auto bar_sfs_full = [&](int b) { return bar_acc_full + 24 + 8u * b; };
  auto bar_sfs_free = [&](int b) { return bar_acc_full + 40 + 8u * b; };
  auto bar_sft_ready = [&](int b) { return bar_acc_full + 56 + 8u * b; };
  auto bar_sft_free = [&](int b) { return bar_acc_full + 72 + 8u * b; };

  const int E = p.E;
  // ---- set-up: barriers, TMEM, tile schedule
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);          // producer expect_tx
      mbar_init(bar_empty(s), 1);         // tcgen05.commit
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, EPI_WARPS);  // one arrive per epilogue warp
    mbar_init(bar_drain, 1);
    for (int b = 0; b < 2; ++b) {
      // expect_tx of the bulk copies, or the 32 producer lanes' cp.async arrivals
      mbar_init(bar_sfs_full(b), kTiledSF ? 1 : 32);
      mbar_init(bar_sfs_free(b), SF_WARPS);
      mbar_init(bar_sft_ready(b), SF_WARPS);
      mbar_init(bar_sft_free(b), 1);      // tcgen05.commit
    }
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
  if (p.pf_b != nullptr && kTiledSF && warp == 0) prefetch_first_unit<BN, kSwiglu>(p, lane);
  // launched with programmatic serialization: everything above overlaps the
  // previous kernel's tail; the offsets, operands and scales it (or an
  // earlier kernel) wrote are read only after this wait
  pdl_launch_dependents();
  pdl_wait();
  if (warp == 2) build_schedule<1>(p, lane, s_off, s_ts, s_mtb);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // k-slices; a partial last slice is zero-filled by TMA
  const int KT = (p.K + BK * CH - 1) / (BK * CH);
  const int KTC = (p.K + BK - 1) / BK;  // 128-element scale chunks per row block
  const int K32 = p.K / 32;
  const int KSPL = kSplit ? p.ksplit : 1;
  const int kper = (KT + KSPL - 1) / KSPL;  // K slices per split (every split non-empty)
  const int total_tiles = s_ts[E] * KSPL;
  // tile -> (expert, m tile, n tile, split) and the split's K slices [k0, k1)
  auto tile_at = [&](int tile, int& e, int& mt, int& nt, int& ks, int& k0, int& k1) {
    const int base = tile / KSPL;
    ks = tile - base * KSPL;
    decode_tile(base, s_ts, E, p.n_tiles_n, e, mt, nt);
    k0 = ks * kper;
    k1 = min(KT, k0 + kper);
  };

  if (warp == 0) {
    // ================= producer: operand stages, and each tile segment's
    // scales one segment ahead of the operands (segment g+1 is requested
    // when segment g's first stage is)
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;  // per-stage bit masks, for the abort drain
    int g = 0;                             // global segment index of the operand loads
    bool ok = true;
    int req_hi = -1;                       // the last scale segment requested
    // request the scales of segment (tile, sg) into buffer gseg & 1
    auto load_scales = [&](int gseg, int tile, int sg) -> bool {
      const int b = gseg & 1;
      const uint32_t par = ((uint32_t)(gseg >> 1) & 1u) ^ 1u;
      const bool got = wait_bar(bar_sfs_free(b), par, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) return false;
      req_hi = gseg;
      int e, mt, nt, ks, k0, k1;
      tile_at(tile, e, mt, nt, ks, k0, k1);
      const int64_t row0 = s_off[e] + (int64_t)mt * BM;
      const int64_t brow = (int64_t)e * p.Nw;
      const int64_t bh0 = kSwiglu ? brow + (int64_t)nt * (BN / 2) : brow + (int64_t)nt * BN;
      const int64_t bh1 = brow + p.n_out + (int64_t)nt * (BN / 2);
      const int kt0 = k0 + sg * SEGK, len = min(SEGK, k1 - kt0);
      // the segment's scale chunks (a packed last k-slice may hold only one)
      const int c0 = kt0 * CH, nch = min(len * CH, KTC - c0);
      const uint32_t sA = sbase + L::OFF_SFA + b * L::SFA_SEG;
      const uint32_t sB = sbase + L::OFF_SFB + b * L::SFB_SEG;
      if (kTiledSF) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_sfs_full(b), (uint32_t)((1 + BN / 128) * nch * 512));
          bulk_copy_g2s(sA, p.sfa + ((int64_t)(s_mtb[e] + mt) * KTC + c0) * 512,
                        (uint32_t)(nch * 512), bar_sfs_full(b));
#pragma unroll
          for (int c = 0; c < BN / 128; ++c) {
            const int64_t wrow = kSwiglu ? (c == 0 ? bh0 : bh1) : bh0 + 128 * c;
            bulk_copy_g2s(sB + c * SEG * 512, p.sfb + ((wrow >> 7) * KTC + c0) * 512,
                          (uint32_t)(nch * 512), bar_sfs_full(b));
          }
        }
      } else {
        // 4 bytes (4 K-blocks) per row and k-slice into the staging layout
        // byte (r % 32) * 16 + (r / 32) * 4 + kb of each 512-byte chunk
        for (int i = 0; i < len; ++i) {
          const int kt = kt0 + i;
#pragma unroll
          for (int q = 0; q < BM / 32; ++q) {
            const int r = lane + 32 * q;
            const int64_t grow = row0 + r;
            const bool valid = grow < p.M;
            const uint8_t* src = valid ? p.sfa + grow * K32 + kt * 4 : p.sfa;
            cp_async_4(sA + i * 512 + (r & 31) * 16 + (r >> 5) * 4, src, valid ? 4u : 0u);
          }
#pragma unroll
          for (int q = 0; q < BN / 32; ++q) {
            const int r = lane + 32 * q;
            const int64_t wrow = kSwiglu ? (r < BN / 2 ? bh0 + r : bh1 + (r - BN / 2)) : bh0 + r;
            const int rr = r & 127;
            cp_async_4(sB + (r >> 7) * SEG * 512 + i * 512 + (rr & 31) * 16 + (rr >> 5) * 4,
                       p.sfb + wrow * K32 + kt * 4, 4u);
          }
        }
        cp_async_mbar_arrive_noinc(bar_sfs_full(b));
      }
      return true;
    };
    if (blockIdx.x < total_tiles) ok = load_scales(0, blockIdx.x, 0);
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt, ks, k0, k1;
      tile_at(tile, e, mt, nt, ks, k0, k1);
      const int nseg = (k1 - k0 + SEGK - 1) / SEGK;  // scale segments of this tile
      const int64_t row0 = s_off[e] + (int64_t)mt * BM;
      const int64_t brow = (int64_t)e * p.Nw;
      // B tile halves: gmm1 = gate rows | up rows; gmm2 = one BN-row box
      const int64_t bh0 = kSwiglu ? brow + (int64_t)nt * (BN / 2) : brow + (int64_t)nt * BN;
      const int64_t bh1 = brow + p.n_out + (int64_t)nt * (BN / 2);
      for (int kt = k0; kt < k1; ++kt) {
        if ((kt - k0) % SEGK == 0) {
          // the next segment's scales: later in this tile, or the next tile's first
          const int sg = (kt - k0) / SEGK;
          const int ntile = sg + 1 < nseg ? tile : tile + (int)gridDim.x;
          if (ntile < total_tiles && !load_scales(g + 1, ntile, sg + 1 < nseg ? sg + 1 : 0)) {
            ok = false;
            break;
          }
          ++g;
        }
        const bool got = wait_bar(bar_empty(stage), phase ^ 1, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {  // keep the warp converged
          ok = false;
          break;
        }
        const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
        const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
        if (lane == 0) {
          // W4A8's unpacked FP4 B counts its global (packed) bytes: half its
          // smem footprint; packed W4A4 operands land byte for byte
          mbar_arrive_expect_tx(bar_full(stage),
                                L::A_BYTES + (kFp4B && !kPacked ? L::B_BYTES / 2 : L::B_BYTES));
          tma_load_2d(sA, &tmA, kt * BK, (int)row0, bar_full(stage));
          if (kSwiglu) {
            tma_load_2d(sB, &tmB, kt * BK, (int)bh0, bar_full(stage));
            tma_load_2d(sB + (BN / 2) * BK, &tmB, kt * BK, (int)bh1, bar_full(stage));
          } else {
            tma_load_2d(sB, &tmB, kt * BK, (int)bh0, bar_full(stage));
          }
        }
        armed |= 1u << stage;
        if (phase) armed_parity |= 1u << stage; else armed_parity &= ~(1u << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok) {
      // drain: wait for this thread's cp.async, every armed stage's copies and
      // the last two scale segments requested (bulk copies into this CTA)
      cp_async_wait_all();
      volatile int no_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u)
          wait_bar(bar_full(s), (armed_parity >> s) & 1u, 1ll << 32, nullptr, &no_abort);
      if (kTiledSF)
        for (int sg = req_hi - 1; sg <= req_hi; ++sg)
          if (sg >= 0)
            wait_bar(bar_sfs_full(sg & 1), (uint32_t)(sg >> 1) & 1u, 1ll << 32, nullptr,
                     &no_abort);
    }
    // every requested scale segment is consumed by the scale writers, which
    // wait for its copies; this thread's own cp.async complete here
    cp_async_wait_all();
  } else if (warp == 1) {
    // ================= MMA issuer (one thread)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      int g = 0;
      bool ok = true;
      bool issued = false;
      constexpr uint32_t IDESC =
          kPacked ? make_idesc_mxf4(BM, BN) : make_idesc(BM, BN, kFp4B);
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, mt, nt, ks, k0, k1;
        tile_at(tile, e, mt, nt, ks, k0, k1);
        if (!wait_bar(bar_acc_empty, acc_phase ^ 1, p.wait_limit, p.status, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = k0; kt < k1; ++kt) {
          const int i = (kt - k0) % SEGK;
          const int b = g & 1;
          if (i == 0) {
            // this segment's scales are in TMEM buffer b
            if (!wait_bar(bar_sft_ready(b), (uint32_t)(g >> 1) & 1u, p.wait_limit, p.status,
                          s_abort)) {
              ok = false;
              break;
            }
          }
          if (!wait_bar(bar_full(stage), phase, p.wait_limit, p.status, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
          const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
          // k-slice i's scale columns: A chunk j at 4j, B chunk j (BN / 32
          // columns, 128-row blocks side by side) at 4 CH + (BN / 32) j
          const uint32_t t_sf = tmem + SF_COL0 + b * SEG_COLS + i * SLICE_COLS;
          const uint64_t adesc = make_sdesc(sA, 16, 1024, 2);
          const uint64_t bdesc = make_sdesc(sB, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            // 32 bytes of each row per MMA; a packed K tail of 128 elements
            // takes the first two only (the slice's second chunk has no scales)
            if (kPacked && (kt * (BK / 32) + kk) * 64 >= p.K) break;
            const int j = kk / MPC;
            const uint32_t sfid = (uint32_t)((kk % MPC) * CH);
            const uint32_t idesc = IDESC | (sfid << 29) | (sfid << 4);
            const uint32_t t_sfa = t_sf + 4 * j, t_sfb = t_sf + 4 * CH + (BN / 32) * j;
            const uint32_t acc = ((kt - k0) | kk) != 0 ? 1u : 0u;
            if constexpr (kPacked)
              tc_mma_mxf4(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, t_sfa, t_sfb, acc);
            else
              tc_mma_mxf8(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, t_sfa, t_sfb, acc);
          }
          issued = true;
          tc_commit(bar_empty(stage));
          if (i == SEGK - 1 || kt == k1 - 1) {
            tc_commit(bar_sft_free(b));  // the segment's scales may be overwritten
            ++g;
          }
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
  } else if (warp < EPI_WARP0) {
    // ================= scale-factor writers, one per TMEM lane quarter
    // (warp & 3): a segment's staged chunks (byte (r % 32) * 16 + (r / 32) *
    // 4 + kb of 128 rows, per k-slice) go from shared memory into this
    // quarter's lanes, 16 bytes (4 columns) per lane and chunk.  Every quarter
    // holds the whole chunk, the layout the block-scaled MMA reads for
    // M = 128.  Register stores keep these copies out of the tensor pipe,
    // where tcgen05.cp would serialize with the MMAs.
    const uint32_t t_q = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt, ks, k0, k1;
      tile_at(tile, e, mt, nt, ks, k0, k1);
      const int nseg = (k1 - k0 + SEGK - 1) / SEGK;
      for (int sg = 0; sg < nseg; ++sg, ++g) {
        const int b = g & 1;
        const uint32_t par = (uint32_t)(g >> 1) & 1u;
        // staged in shared memory, and the MMAs that last read TMEM buffer b are done
        const bool got = wait_bar(bar_sfs_full(b), par, p.wait_limit, p.status, s_abort) &&
                         wait_bar(bar_sft_free(b), par ^ 1u, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {  // keep the warp converged
          ok = false;
          break;
        }
        const int len = min(SEGK, k1 - (k0 + sg * SEGK));
        const uint8_t* sfa_s = smem + L::OFF_SFA + b * L::SFA_SEG;
        const uint8_t* sfb_s = smem + L::OFF_SFB + b * L::SFB_SEG;
        // (a chunk past K is never copied in; its columns are never read)
        for (int i = 0; i < len; ++i) {
          const uint32_t col = SF_COL0 + b * SEG_COLS + i * SLICE_COLS;
#pragma unroll
          for (int j = 0; j < CH; ++j) {
            const int ch = i * CH + j;
            tmem_st_4(t_q + col + 4 * j,
                      *reinterpret_cast<const uint4*>(sfa_s + ch * 512 + lane * 16));
#pragma unroll
            for (int c = 0; c < BN / 128; ++c)
              tmem_st_4(t_q + col + 4 * CH + (BN / 32) * j + 4 * c,
                        *reinterpret_cast<const uint4*>(sfb_s + c * SEG * 512 + ch * 512 +
                                                        lane * 16));
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_sft_ready(b));
          mbar_arrive(bar_sfs_free(b));
        }
      }
    }
  } else {
    // ================= epilogue: EPI_GROUPS warps per TMEM lane quarter
    // (warp & 3 = quarter; group g takes the g-th slice of the columns)
    const int q = warp & 3;
    const int grp = (warp - EPI_WARP0) >> 2;
    const int row = q * 32 + lane;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt, ks, k0, k1;
      tile_at(tile, e, mt, nt, ks, k0, k1);
      const int64_t grow = s_off[e] + (int64_t)mt * BM + row;
      const bool valid = grow < s_off[e + 1];
      const bool got = wait_bar(bar_acc_full, acc_phase, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) break;  // keep the warp converged
      tc_fence_after();
      epilogue_tile<BN, kSwiglu, kTiledSF, kFp4A, kSplit>(
          p, t_row, grp, row, lane, grow, valid, nt, (int64_t)(s_mtb[e] + mt) * BM + row,
          [&] { if (lane == 0) mbar_arrive(bar_acc_empty); }, ks);
      acc_phase ^= 1;
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

// ---------------------------------------------------------------- both GEMMs in one kernel
//
// Small batches (every group at most BMA_SMALL rows, MXFP8, MMA-layout
// scales): the layer's two grouped GEMMs run as one persistent kernel.  CTA b
// takes units b, b + grid, ... of one list holding gmm1's U1 units (expert by
// expert, n-tile fastest) and then gmm2's U2 units, so gmm2 fills the SMs
// that gmm1's last partial round leaves idle and needs no launch of its own.
// A gmm2 unit of expert e reads gmm1's output rows of e (payload by TMA, tiled
// scales by bulk copy): every epilogue warp of a gmm1 unit, once its stores
// are done, fences them for the async proxy and adds one to done[e] (after a
// gpu-scope fence); the producer of a gmm2 unit reads done[e] with acquire
// until it holds EPI_WARPS x the expert's gmm1 units, then fences for the
// async proxy before its loads.  That wait is bounded and happens only at the
// unit's first load, where every earlier unit of the CTA can finish without
// the producer; the scale request made one segment ahead only polls, and a
// gmm2 unit whose expert is not done yet gets its first scale segment
// requested at its start instead.  gmm1 units wait for nothing, and the grid
// (at most one CTA per SM) is co-resident, so every wait ends.  done[] is
// zeroed by the layer's routing kernel before this kernel's wait returns.
struct ChainParams {
  Params g[2];  // [0] gmm1 (SwiGLU + requant), [1] gmm2 (bf16 out)
  int* done;    // [E]
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__global__ void __launch_bounds__(THREADS1, 1)
    gemm_chain_kernel(const __grid_constant__ CUtensorMap tmA1,
                      const __grid_constant__ CUtensorMap tmB1,
                      const __grid_constant__ CUtensorMap tmA2,
                      const __grid_constant__ CUtensorMap tmB2, const ChainParams cp) {
  constexpr int BN = 256;
  using L = Layout1<BN, BMA_SMALL>;
  constexpr int STAGES = L::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Params& p = cp.g[0];  // the fields both GEMMs share: E, M, offsets, status, limit

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
  auto bar_sfs_full = [&](int b) { return bar_acc_full + 24 + 8u * b; };
  auto bar_sfs_free = [&](int b) { return bar_acc_full + 40 + 8u * b; };
  auto bar_sft_ready = [&](int b) { return bar_acc_full + 56 + 8u * b; };
  auto bar_sft_free = [&](int b) { return bar_acc_full + 72 + 8u * b; };

  const int E = p.E;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_empty, EPI_WARPS);
    mbar_init(bar_drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_sfs_full(b), 1);
      mbar_init(bar_sfs_free(b), SF_WARPS);
      mbar_init(bar_sft_ready(b), SF_WARPS);
      mbar_init(bar_sft_free(b), 1);
    }
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
  if (p.pf_b != nullptr && warp == 0) prefetch_first_unit<BN, true>(p, lane);
  pdl_launch_dependents();
  pdl_wait();
  if (warp == 2) build_schedule<1>(p, lane, s_off, s_ts, s_mtb);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int U1 = s_ts[E];                          // gmm1 units (n_tiles_n of gmm1)
  const int total = U1 + s_mtb[E] * cp.g[1].n_tiles_n;
  const int KT[2] = {(cp.g[0].K + BK - 1) / BK, (cp.g[1].K + BK - 1) / BK};
  // unit -> (GEMM gi, expert, m-tile, n-tile)
  auto unit_at = [&](int u, int& gi, int& e, int& mt, int& nt) {
    gi = u >= U1 ? 1 : 0;
    const int lu = gi ? u - U1 : u;
    const int ntn = cp.g[gi].n_tiles_n;
    const int m = lu / ntn;
    nt = lu - m * ntn;
    int unused;
    decode_tile(m, s_mtb, E, 1, e, mt, unused);
  };
  // gmm1 epilogue-warp completions that make expert e's gmm2 inputs whole
  auto done_need = [&](int e) { return EPI_WARPS * (s_mtb[e + 1] - s_mtb[e]) * cp.g[0].n_tiles_n; };

  if (warp == 0) {
    // ================= producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;
    int g = 0;
    bool ok = true;
    int deferred = -1;  // a gmm2 unit whose first scale segment waits for its start
    int req_hi = -1;    // the last scale segment requested
    auto load_scales = [&](int gseg, int u, int sg) -> bool {
      const int b = gseg & 1;
      const uint32_t par = ((uint32_t)(gseg >> 1) & 1u) ^ 1u;
      const bool got = wait_bar(bar_sfs_free(b), par, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) return false;
      req_hi = gseg;
      int gi, e, mt, nt;
      unit_at(u, gi, e, mt, nt);
      const Params& q = cp.g[gi];
      const int64_t brow = (int64_t)e * q.Nw;
      const int64_t bh0 = gi == 0 ? brow + (int64_t)nt * (BN / 2) : brow + (int64_t)nt * BN;
      const int64_t bh1 = gi == 0 ? brow + q.n_out + (int64_t)nt * (BN / 2) : bh0 + 128;
      const int kt0 = sg * SEG, len = min(SEG, KT[gi] - kt0);
      const uint32_t sA = sbase + L::OFF_SFA + b * L::SFA_SEG;
      const uint32_t sB = sbase + L::OFF_SFB + b * L::SFB_SEG;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_sfs_full(b), (uint32_t)(3 * len * 512));
        bulk_copy_g2s(sA, q.sfa + ((int64_t)(s_mtb[e] + mt) * KT[gi] + kt0) * 512,
                      (uint32_t)(len * 512), bar_sfs_full(b));
        bulk_copy_g2s(sB, q.sfb + ((bh0 >> 7) * KT[gi] + kt0) * 512, (uint32_t)(len * 512),
                      bar_sfs_full(b));
        bulk_copy_g2s(sB + SEG * 512, q.sfb + ((bh1 >> 7) * KT[gi] + kt0) * 512,
                      (uint32_t)(len * 512), bar_sfs_full(b));
      }
      __syncwarp();
      return true;
    };
    // expert e's gmm1 outputs all stored (lane 0 reads; the whole warp agrees)
    auto expert_done = [&](int e) -> bool {
      int ready = 0;
      if (lane == 0) ready = ld_acquire_gpu(cp.done + e) >= done_need(e);
      return __shfl_sync(0xffffffffu, ready, 0) != 0;
    };
    auto wait_expert = [&](int e) -> bool {
      bool ready = expert_done(e);
      const long long t0 = clock64();
      while (!ready) {
        if (*s_abort) return false;
        if (clock64() - t0 > p.wait_limit) {
          if (lane == 0) report_error(p.status, ERR_TIMEOUT);
          *s_abort = 1;
          return false;
        }
        __nanosleep(200);
        ready = expert_done(e);
      }
      fence_proxy_async_global();
      return true;
    };
    // request segment 0 (the first unit's first), or defer it
    if ((int)blockIdx.x < total) {
      int gi, e, mt, nt;
      unit_at(blockIdx.x, gi, e, mt, nt);
      if (gi == 1 && !expert_done(e)) deferred = blockIdx.x;
      else ok = load_scales(0, blockIdx.x, 0);
    }
    for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
      int gi, e, mt, nt;
      unit_at(u, gi, e, mt, nt);
      if (gi == 1) {
        // gmm1's rows of this expert (and their scales) are stored
        if (!wait_expert(e)) { ok = false; break; }
        if (deferred == u) {
          deferred = -1;
          if (!load_scales(g, u, 0)) { ok = false; break; }
        }
      }
      const Params& q = cp.g[gi];
      const CUtensorMap* mA = gi ? &tmA2 : &tmA1;
      const CUtensorMap* mB = gi ? &tmB2 : &tmB1;
      const int kt_n = KT[gi];
      const int nseg = (kt_n + SEG - 1) / SEG;
      const int64_t row0 = s_off[e] + (int64_t)mt * BM;
      const int64_t brow = (int64_t)e * q.Nw;
      const int64_t bh0 = gi == 0 ? brow + (int64_t)nt * (BN / 2) : brow + (int64_t)nt * BN;
      const int64_t bh1 = brow + q.n_out + (int64_t)nt * (BN / 2);
      for (int kt = 0; kt < kt_n; ++kt) {
        if (kt % SEG == 0) {
          // the next segment: later in this unit, or the next unit's first
          const int sg = kt / SEG;
          const int nu = sg + 1 < nseg ? u : u + (int)gridDim.x;
          if (nu < total) {
            int ngi, ne, nmt, nnt;
            unit_at(nu, ngi, ne, nmt, nnt);
            if (nu != u && ngi == 1 && !expert_done(ne)) {
              deferred = nu;
            } else if (!load_scales(g + 1, nu, sg + 1 < nseg ? sg + 1 : 0)) {
              ok = false;
              break;
            }
          }
          ++g;
        }
        const bool got = wait_bar(bar_empty(stage), phase ^ 1, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
        const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_full(stage), L::A_BYTES + L::B_BYTES);
          tma_load_2d(sA, mA, kt * BK, (int)row0, bar_full(stage));
          if (gi == 0) {
            tma_load_2d(sB, mB, kt * BK, (int)bh0, bar_full(stage));
            tma_load_2d(sB + (BN / 2) * BK, mB, kt * BK, (int)bh1, bar_full(stage));
          } else {
            tma_load_2d(sB, mB, kt * BK, (int)bh0, bar_full(stage));
          }
        }
        armed |= 1u << stage;
        if (phase) armed_parity |= 1u << stage; else armed_parity &= ~(1u << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok) {
      // abort: every copy into this CTA's shared memory lands before it exits
      // (the armed operand stages and the last two scale segments requested)
      volatile int no_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u)
          wait_bar(bar_full(s), (armed_parity >> s) & 1u, 1ll << 32, nullptr, &no_abort);
      for (int sg = req_hi - 1; sg <= req_hi; ++sg)
        if (sg >= 0)
          wait_bar(bar_sfs_full(sg & 1), (uint32_t)(sg >> 1) & 1u, 1ll << 32, nullptr, &no_abort);
    }
  } else if (warp == 1) {
    // ================= MMA issuer (one thread)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      int g = 0;
      bool ok = true;
      bool issued = false;
      constexpr uint32_t IDESC = make_idesc(BM, BN, false);
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        int gi, e, mt, nt;
        unit_at(u, gi, e, mt, nt);
        const int kt_n = KT[gi];
        if (!wait_bar(bar_acc_empty, acc_phase ^ 1, p.wait_limit, p.status, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < kt_n; ++kt) {
          const int i = kt % SEG;
          const int b = g & 1;
          if (i == 0 && !wait_bar(bar_sft_ready(b), (uint32_t)(g >> 1) & 1u, p.wait_limit,
                                  p.status, s_abort)) {
            ok = false;
            break;
          }
          if (!wait_bar(bar_full(stage), phase, p.wait_limit, p.status, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = sbase + L::OFF_A + stage * L::A_BYTES;
          const uint32_t sB = sbase + L::OFF_B + stage * L::B_BYTES;
          const uint32_t t_sf = tmem + SF_COL0 + b * SEG_COLS + i * SF_COLS_PER_STAGE;
          const uint64_t adesc = make_sdesc(sA, 16, 1024, 2);
          const uint64_t bdesc = make_sdesc(sB, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t sfid = (uint32_t)kk;
            const uint32_t idesc = IDESC | (sfid << 29) | (sfid << 4);
            const uint32_t acc = (kt | kk) != 0 ? 1u : 0u;
            tc_mma_mxf8(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, t_sf, t_sf + 4, acc);
          }
          issued = true;
          tc_commit(bar_empty(stage));
          if (i == SEG - 1 || kt == kt_n - 1) {
            tc_commit(bar_sft_free(b));
            ++g;
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(bar_acc_full);
        acc_phase ^= 1;
      }
      if (!ok && issued) {
        tc_commit(bar_drain);
        volatile int no_abort = 0;
        wait_bar(bar_drain, 0, 1ll << 32, nullptr, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp < EPI_WARP0) {
    // ================= scale-factor writers (as in the single-GEMM kernel)
    const uint32_t t_q = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int g = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
      int gi, e, mt, nt;
      unit_at(u, gi, e, mt, nt);
      const int nseg = (KT[gi] + SEG - 1) / SEG;
      for (int sg = 0; sg < nseg; ++sg, ++g) {
        const int b = g & 1;
        const uint32_t par = (uint32_t)(g >> 1) & 1u;
        const bool got = wait_bar(bar_sfs_full(b), par, p.wait_limit, p.status, s_abort) &&
                         wait_bar(bar_sft_free(b), par ^ 1u, p.wait_limit, p.status, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const int len = min(SEG, KT[gi] - sg * SEG);
        const uint8_t* sfa_s = smem + L::OFF_SFA + b * L::SFA_SEG;
        const uint8_t* sfb_s = smem + L::OFF_SFB + b * L::SFB_SEG;
        for (int i = 0; i < len; ++i) {
          const uint32_t col = SF_COL0 + b * SEG_COLS + i * SF_COLS_PER_STAGE;
          tmem_st_4(t_q + col, *reinterpret_cast<const uint4*>(sfa_s + i * 512 + lane * 16));
          tmem_st_4(t_q + col + 4, *reinterpret_cast<const uint4*>(sfb_s + i * 512 + lane * 16));
          tmem_st_4(t_q + col + 8,
                    *reinterpret_cast<const uint4*>(sfb_s + SEG * 512 + i * 512 + lane * 16));
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_sft_ready(b));
          mbar_arrive(bar_sfs_free(b));
        }
      }
    }
  } else {
    // ================= epilogue
    const int q = warp & 3;
    const int grp = (warp - EPI_WARP0) >> 2;
    const int row = q * 32 + lane;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      int gi, e, mt, nt;
      unit_at(u, gi, e, mt, nt);
      const int64_t grow = s_off[e] + (int64_t)mt * BM + row;
      const bool valid = grow < s_off[e + 1];
      const bool got = wait_bar(bar_acc_full, acc_phase, p.wait_limit, p.status, s_abort);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      auto release = [&] { if (lane == 0) mbar_arrive(bar_acc_empty); };
      const int64_t tiled_row = (int64_t)(s_mtb[e] + mt) * BM + row;
      if (gi == 0) {
        epilogue_tile<BN, true, true, false, false>(cp.g[0], t_row, grp, row, lane, grow, valid,
                                                    nt, tiled_row, release);
        // this warp's rows of expert e are stored: visible to the async
        // proxy, then counted (gpu-scope fence before the count)
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(cp.done + e, 1);
      } else {
        epilogue_tile<BN, false, true, false, false>(cp.g[1], t_row, grp, row, lane, grow, valid,
                                                     nt, tiled_row, release);
      }
      acc_phase ^= 1;
    }
  }

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

template <int BN, bool kSwiglu, bool kTiledSF, int kFmt, bool kSplit = false, int BMA = BM>
static cudaError_t launch_single(const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                                 const uint8_t* sfb, const int64_t* offsets, int64_t M, int E,
                                 int K, int Nw, int n_out, void* out, uint8_t* out_scale,
                                 cudaStream_t stream, int ksplit = 1, float* partial = nullptr,
                                 bool prefetch_first = false) {
  using L = Layout1<BN, BMA>;
  if (M == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static uint64_t configured[64] = {0};  // context id the attribute was set in
  auto kern = gemm1sm_kernel<BN, kSwiglu, kTiledSF, kFmt, kSplit, BMA>;
  const uint64_t ctx = context_id();
  if (ctx == 0 || configured[dev] != ctx) {
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (err != cudaSuccess) return err;
    configured[dev] = context_id();
  }
  CUtensorMap tmA, tmB;
  const uint32_t b_box_rows = kSwiglu ? BN / 2 : BN;
  // W4A4: packed bytes as they are (K / 2 per row); W4A8: B unpacked
  const uint64_t inner = kFmt == FMT_W4A4 ? (uint64_t)K / 2 : (uint64_t)K;
  if (!make_map(&tmA, a, inner, (uint64_t)M, BK, BMA))
    return cudaErrorInvalidValue;
  if (!make_map(&tmB, b, inner, (uint64_t)E * Nw, BK, b_box_rows, kFmt == FMT_W4A8))
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
  p.n_tiles_n = kSwiglu ? n_out / (BN / 2) : (int)ceil_div(n_out, BN);  // ragged last n-tile: E == 1
  p.status = device_status_ptr();
  p.wait_limit = wait_limit_cycles();
  p.ksplit = kSplit ? ksplit : 1;
  p.partial = kSplit ? partial : nullptr;
  // 16-byte aligned rows and pieces for the bulk prefetch
  const bool pf_ok = prefetch_first && kTiledSF && ((uintptr_t)b & 15u) == 0 &&
                     ((uintptr_t)sfb & 15u) == 0 && inner % 16 == 0;
  p.pf_b = pf_ok ? b : nullptr;
  p.pf_row_bytes = (int64_t)(kFmt == FMT_W8A8 ? K : K / 2);  // global bytes per weight row
  const int64_t tiles_bound = (ceil_div(M, BM) + E) * (int64_t)p.n_tiles_n * ksplit;
  const int grid = (int)std::min<int64_t>(tiles_bound, num_sms());
  return launch_pdl(kern, dim3(grid), dim3(THREADS1), L::ALLOC, stream, tmA, tmB, p);
}

// Kernel choice (mxmoe_set_gemm_2sm): 256-wide tiles with MMA-layout scales go
// to the 2-SM kernel when selected for this GEMM and the device can
// co-schedule CTA pairs; both kernels give the same bytes.  By default gmm2
// (bf16 out) takes the 2-SM kernel when experts average at least 4 m-tiles,
// everything else the 1-SM kernel.  group_rows_max > 0 bounds every group's
// row count (the caller's guarantee); at most BMA_SMALL rows select the 1-SM
// kernel's short A boxes (MMA-layout scales, 256-wide tiles, every format).
template <int BN, bool kSwiglu, bool kTiledSF, int kFmt>
static cudaError_t launch(const uint8_t* a, const uint8_t* sfa, const uint8_t* b,
                          const uint8_t* sfb, const int64_t* offsets, int64_t M, int E, int K,
                          int Nw, int n_out, void* out, uint8_t* out_scale, cudaStream_t stream,
                          int ksplit = 1, float* partial = nullptr, int64_t group_rows_max = 0) {
  if (ksplit > 1) {
    if constexpr (kSwiglu) {
      return cudaErrorNotSupported;
    } else {
      return launch_single<BN, false, kTiledSF, kFmt, true>(a, sfa, b, sfb, offsets, M, E, K, Nw,
                                                            n_out, out, out_scale, stream, ksplit,
                                                            partial);
    }
  }
  if (BN == 256 && use_two_sm_gemm(kSwiglu, M, E)) {
    const cudaError_t err = launch_pair<kSwiglu, kTiledSF, kFmt>(a, sfa, b, sfb, offsets, M, E, K, Nw,
                                                           n_out, out, out_scale, stream);
    if (err != cudaErrorNotSupported) return err;
  }
  if constexpr (BN == 256 && kTiledSF) {
    if (group_rows_max > 0 && group_rows_max <= BMA_SMALL) {
      // gmm1 (which follows the routing) prefetches its guessed first unit;
      // the guess assumes every expert has rows, so only when uniform routing
      // of T = group_rows_max tokens to k = M / T of the E experts would leave
      // at most a fifth of them empty.  (gmm2's weights gain nothing from it.)
      const double T = (double)group_rows_max, k = (double)M / T;
      const bool guess = kSwiglu && k < E && 1.0 - std::pow(1.0 - k / E, T) >= 0.8;
      return launch_single<BN, kSwiglu, kTiledSF, kFmt, false, BMA_SMALL>(
          a, sfa, b, sfb, offsets, M, E, K, Nw, n_out, out, out_scale, stream, 1, nullptr,
          guess);
    }
  }
  return launch_single<BN, kSwiglu, kTiledSF, kFmt>(a, sfa, b, sfb, offsets, M, E, K, Nw, n_out, out,
                                              out_scale, stream);
}

}  // namespace gemm

bool gemm_chain_supported(int64_t group_rows_max, int H, int I) {
  return group_rows_max > 0 && group_rows_max <= gemm::BMA_SMALL && H % 256 == 0 && I % 128 == 0;
}

cudaError_t launch_gemm_chain(const uint8_t* xq, const uint8_t* xs, const uint8_t* w13q,
                              const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                              const int64_t* offsets, int64_t M, int E, int H, int I, uint8_t* aq,
                              uint8_t* as, uint16_t* y, int* done, cudaStream_t stream,
                              int64_t group_rows_max) {
  using namespace gemm;
  using L = Layout1<256, BMA_SMALL>;
  if (!gemm_chain_supported(group_rows_max, H, I) || !done || E > MAX_E)
    return cudaErrorNotSupported;
  if (M == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static uint64_t configured[64] = {0};
  const uint64_t ctx = context_id();
  if (ctx == 0 || configured[dev] != ctx) {
    cudaError_t err = cudaFuncSetAttribute(gemm_chain_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (err != cudaSuccess) return err;
    configured[dev] = context_id();
  }
  CUtensorMap tmA1, tmB1, tmA2, tmB2;
  if (!make_map(&tmA1, xq, (uint64_t)H, (uint64_t)M, BK, BMA_SMALL) ||
      !make_map(&tmB1, w13q, (uint64_t)H, (uint64_t)E * 2 * I, BK, 128) ||
      !make_map(&tmA2, aq, (uint64_t)I, (uint64_t)M, BK, BMA_SMALL) ||
      !make_map(&tmB2, w2q, (uint64_t)I, (uint64_t)E * H, BK, 256))
    return cudaErrorInvalidValue;
  ChainParams cp;
  for (int gi = 0; gi < 2; ++gi) {
    Params& p = cp.g[gi];
    p.offsets = offsets;
    p.M = M;
    p.E = E;
    p.status = device_status_ptr();
    p.wait_limit = wait_limit_cycles();
    p.ksplit = 1;
    p.partial = nullptr;
    p.pf_b = nullptr;
    p.pf_row_bytes = 0;
  }
  cp.g[0].sfa = xs;
  cp.g[0].sfb = w13s;
  cp.g[0].out = aq;
  cp.g[0].out_scale = as;
  cp.g[0].K = H;
  cp.g[0].Nw = 2 * I;
  cp.g[0].n_out = I;
  cp.g[0].n_tiles_n = I / 128;
  cp.g[1].sfa = as;
  cp.g[1].sfb = w2s;
  cp.g[1].out = y;
  cp.g[1].out_scale = nullptr;
  cp.g[1].K = I;
  cp.g[1].Nw = H;
  cp.g[1].n_out = H;
  cp.g[1].n_tiles_n = H / 256;
  cp.done = done;
  // gmm1's first-unit guess, under the same condition as the single-GEMM launch
  const double T = (double)group_rows_max, k = (double)M / T;
  if (k < E && 1.0 - std::pow(1.0 - k / E, T) >= 0.8 && ((uintptr_t)w13q & 15u) == 0 &&
      ((uintptr_t)w13s & 15u) == 0) {
    cp.g[0].pf_b = w13q;
    cp.g[0].pf_row_bytes = H;
  }
  const int64_t units_bound = (ceil_div(M, BM) + E) * (int64_t)(I / 128 + H / 256);
  const int grid = (int)std::min<int64_t>(units_bound, num_sms());
  return launch_pdl(gemm_chain_kernel, dim3(grid), dim3(THREADS1), L::ALLOC, stream, tmA1, tmB1,
                    tmA2, tmB2, cp);
}

cudaError_t launch_gemm_swiglu_quant(const uint8_t* xq, const uint8_t* xs, const uint8_t* w13q,
                                     const uint8_t* w13s, const int64_t* offsets, int64_t M,
                                     int E, int H, int I, uint8_t* aq, uint8_t* as,
                                     cudaStream_t stream, bool tiled_scales, int fmt,
                                     int64_t group_rows_max) {
  if (fmt == gemm::FMT_W4A8 || fmt == gemm::FMT_W4A4) {
    if (!tiled_scales) return cudaErrorNotSupported;
    if (fmt == gemm::FMT_W4A8)
      return gemm::launch<256, true, true, gemm::FMT_W4A8>(xq, xs, w13q, w13s, offsets, M, E, H, 2 * I,
                                                     I, aq, as, stream, 1, nullptr, group_rows_max);
    return gemm::launch<256, true, true, gemm::FMT_W4A4>(xq, xs, w13q, w13s, offsets, M, E, H, 2 * I, I,
                                                   aq, as, stream, 1, nullptr, group_rows_max);
  }
  if (fmt != gemm::FMT_W8A8) return cudaErrorNotSupported;
  if (tiled_scales)
    return gemm::launch<256, true, true, gemm::FMT_W8A8>(xq, xs, w13q, w13s, offsets, M, E, H, 2 * I,
                                                   I, aq, as, stream, 1, nullptr, group_rows_max);
  return gemm::launch<256, true, false, gemm::FMT_W8A8>(xq, xs, w13q, w13s, offsets, M, E, H, 2 * I,
                                                  I, aq, as, stream);
}

// Split-K sums: out[m, n] = bf16(sum over s in order of partial[s][m][n]);
// one thread per 8 columns (N % 8 == 0, 16-byte aligned rows).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ partial,
                                                            int S, int64_t M, int N,
                                                            uint16_t* __restrict__ out) {
  const int64_t n8 = M * N / 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      const float4* src = reinterpret_cast<const float4*>(partial + (int64_t)s * M * N + i * 8);
      const float4 u = src[0], w = src[1];
      a[0] += u.x; a[1] += u.y; a[2] += u.z; a[3] += u.w;
      a[4] += w.x; a[5] += w.y; a[6] += w.z; a[7] += w.w;
    }
    st_v4(out + i * 8, make_uint4(cvt_bf16x2(a[0], a[1]), cvt_bf16x2(a[2], a[3]),
                                  cvt_bf16x2(a[4], a[5]), cvt_bf16x2(a[6], a[7])));
  }
}

// 256-wide tiles when the 128-row weight blocks pair up (a ragged last block,
// H % 128 != 0, only with E == 1 and MMA-layout scales), 128-wide otherwise.
template <int kFmt>
static cudaError_t launch_bf16_fmt(const uint8_t* aq, const uint8_t* as, const uint8_t* w2q,
                                   const uint8_t* w2s, const int64_t* offsets, int64_t M, int E,
                                   int I, int H, uint16_t* y, cudaStream_t stream, int ksplit,
                                   float* partial, int64_t group_rows_max) {
  cudaError_t err;
  if (ceil_div(H, 128) % 2 == 0)
    err = gemm::launch<256, false, true, kFmt>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y,
                                               nullptr, stream, ksplit, partial, group_rows_max);
  else
    err = gemm::launch<128, false, true, kFmt>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y,
                                               nullptr, stream, ksplit, partial);
  if (err != cudaSuccess || ksplit <= 1 || M == 0) return err;
  const int64_t n8 = M * H / 8;
  int64_t blocks = ceil_div(n8, 256);
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(partial, ksplit, M, H, y);
  return cudaGetLastError();
}

int gemm_bf16_ksplit(int64_t M, int N, int K, bool packed_fp4) {
  const int64_t n_tiles = ceil_div(N, ceil_div(N, 128) % 2 == 0 ? 256 : 128);
  const int64_t tiles = ceil_div(M, gemm::BM) * n_tiles;
  const int KT = (int)ceil_div(K, packed_fp4 ? 256 : 128);  // the kernel's k-slices
  const int sms = num_sms();
  if (tiles * 2 > sms) return 1;  // enough tiles to fill the GPU
  int S = (int)std::min<int64_t>({(int64_t)sms / tiles, (int64_t)KT / 4, 32});
  if (S <= 1) return 1;
  const int kper = (int)ceil_div(KT, S);
  return (int)ceil_div(KT, kper);  // every split non-empty
}

cudaError_t launch_gemm_bf16(const uint8_t* aq, const uint8_t* as, const uint8_t* w2q,
                             const uint8_t* w2s, const int64_t* offsets, int64_t M, int E,
                             int I, int H, uint16_t* y, cudaStream_t stream, bool tiled_scales,
                             int fmt, int ksplit, float* partial, int64_t group_rows_max) {
  if (ksplit > 1 && (E != 1 || !tiled_scales || !partial)) return cudaErrorNotSupported;
  if (fmt == gemm::FMT_W4A8 || fmt == gemm::FMT_W4A4) {
    if (!tiled_scales) return cudaErrorNotSupported;
    return fmt == gemm::FMT_W4A8
               ? launch_bf16_fmt<gemm::FMT_W4A8>(aq, as, w2q, w2s, offsets, M, E, I, H, y, stream,
                                                 ksplit, partial, group_rows_max)
               : launch_bf16_fmt<gemm::FMT_W4A4>(aq, as, w2q, w2s, offsets, M, E, I, H, y, stream,
                                                 ksplit, partial, group_rows_max);
  }
  if (fmt != gemm::FMT_W8A8) return cudaErrorNotSupported;
  if (tiled_scales)
    return launch_bf16_fmt<gemm::FMT_W8A8>(aq, as, w2q, w2s, offsets, M, E, I, H, y, stream,
                                           ksplit, partial, group_rows_max);
  if (ceil_div(H, 128) % 2 == 0)
    return gemm::launch<256, false, false, gemm::FMT_W8A8>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y,
                                                     nullptr, stream);
  return gemm::launch<128, false, false, gemm::FMT_W8A8>(aq, as, w2q, w2s, offsets, M, E, I, H, H, y,
                                                   nullptr, stream);
}

}  // namespace mxmoe
