// Top-k routing, expert permutation and the fused per-token MX activation
// quant (init_routing with quant_mode=3).
//
// "Quantization on Ascend", MoE MXFP8 "Forward": the dispatcher runs
// init_routing with quant_mode=3, which fuses the per-token MX activation
// quant into routing and emits the e4m3 payload, the e8m0 block scale and the
// per-expert token counts.  sglang PR #32266 (commit note on quant_mode=3):
// the fused output is byte-identical to routing followed by a separate quant.
//
// Three kernels, one stream:
//   1. route_topk_rank: one warp per token picks the top-k experts (descending
//      logit, ties -> lower id; k rounds of two warp reductions over
//      order-preserving integer keys) and their softmax weights; each 64-token block
//      marks its tokens in a per-expert 64-bit mask, from which every
//      assignment's rank inside the block (flat order) and the block's
//      per-expert histogram are popcounts.
//   2. route_scan: per-expert exclusive prefix of the block histograms (the
//      block's base row inside each expert, into a second array) and, in one
//      more CTA beside them, of the expert totals (offsets).
//   3. route_permute_quant: one warp per token computes its k destination rows
//      (offset + block base + rank); each lane quantizes one 32-element block
//      of the hidden row once and writes its 32 payload bytes and scale byte
//      to all k rows (or copies the bf16 block, two-step mode).
// The permutation is deterministic: rows of one expert are in flat-index
// (token) order.
//
// Roofline (kernel 3 dominates): x read once (2 B/elem) + k copies of the
// payload (1 B) and scales (1/32 B) written; ids/weights/indices are small.
#include "common.cuh"
#include "topk.cuh"
#include "internal.h"
#include "tiled_scales.h"

namespace mxmoe {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;


// TPW tokens per warp (kRouteTokensPerBlock / TPW warps per block): two, so a
// 64-token block runs 32 warps.  The selection is a chain of dependent warp
// reductions per token; the two tokens of a warp interleave, and the block's
// 32 warps keep the SM's schedulers busy (with four tokens per warp and 16
// warps, each warp's ~1800-instruction chain set the kernel's length).
template <int EPL>
constexpr int topk_tokens_per_warp() { return 2; }

// KC > 0: k == KC (the selection rounds unrolled)
template <int EPL, int TPW = topk_tokens_per_warp<EPL>(), int KC = 0>  // logits per lane: E <= 32 * EPL
__global__ void __launch_bounds__(32 * (kRouteTokensPerBlock / TPW)) route_topk_rank_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renormalize,
    int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
    int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist) {
  constexpr int WARPS = kRouteTokensPerBlock / TPW;
  // s_mask[e] bit tl: token tl of this block chose expert e.  A token's k
  // experts are distinct, so its rank among the block's rows of expert e in
  // flat (token) order is the number of earlier tokens with that bit set.
  extern __shared__ unsigned long long s_mask[];  // [E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kRouteTokensPerBlock;
  const int nt = min(kRouteTokensPerBlock, T - t0);
  // the scan and permute kernels may be scheduled now (they wait for this
  // grid's results before reading them)
  pdl_launch_dependents();

  for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0ull;
  __syncthreads();

  // the warp's tokens warp, warp + WARPS, ... go through the top-k NT at a
  // time (all together for narrow rows)
  constexpr int NT = EPL <= 4 ? TPW : 1;
  int chosen[TPW];
  float ws[TPW];
#pragma unroll
  for (int g = 0; g < TPW / NT; ++g) {
    const float* rows[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int tl = warp + WARPS * (g * NT + n);
      rows[n] = tl < nt ? logits + (int64_t)(t0 + tl) * E : nullptr;
    }
    int c[NT];
    float v[NT], w[NT];
    warp_topk_softmax<EPL, NT, KC>(rows, E, k, renormalize != 0, lane, c, v, w);
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      chosen[g * NT + n] = c[n];
      ws[g * NT + n] = w[n];
    }
  }
#pragma unroll
  for (int it = 0; it < TPW; ++it) {
    const int tl = warp + WARPS * it;
    if (tl < nt && lane < k) {
      const int64_t f = (int64_t)(t0 + tl) * k + lane;
      topk_ids[f] = chosen[it];
      topk_w[f] = ws[it];
      atomicOr(&s_mask[chosen[it]], 1ull << tl);
    }
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < TPW; ++it) {
    const int tl = warp + WARPS * it;
    if (tl < nt && lane < k)
      local_rank[(int64_t)(t0 + tl) * k + lane] =
          __popcll(s_mask[chosen[it]] & ((1ull << tl) - 1ull));
  }
  // expert-major histogram: row e holds expert e's count in every block
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    block_hist[(int64_t)e * gridDim.x + blockIdx.x] = __popcll(s_mask[e]);
}

// The scan, over the expert-major histogram hist[e][b] (nb blocks per row),
// by ceil(E / kScanWarps) row CTAs and one totals CTA that all start
// together; no CTA waits for another.  A row CTA's warp takes one expert row:
// it loads the row 256 blocks at a time (lane l holds blocks l, l + 32, ...,
// l + 224: coalesced, all in flight together), scans the eight 32-block
// chunks independently (their shuffle chains interleave), joins them by the
// prefix of the chunk totals, and writes the row's exclusive prefix (each
// block's base row inside expert e) to base[e][b].  The totals CTA (the last)
// sums every row itself, eight rows per warp with all their loads in flight,
// and scans the E totals into counts, offsets and the experts' first 128-row
// blocks of the tiled scale layout.  (Before, the row CTAs wrote the totals
// and the last of them to take a ticket scanned them: two more dependent
// round trips to memory.)
constexpr int kScanWarps = 16;
constexpr int kScanThreads = 32 * kScanWarps;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Exclusive scan of one value per thread over the block (blockDim.x a
// multiple of 32, at most 1024); *total receives the sum.  s_warp: 33 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int incl = warp_incl_scan(v, lane);
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
    const int xi = warp_incl_scan(x, lane);
    s_warp[lane] = xi - x;
    if (lane == 31) s_warp[32] = xi;
  }
  __syncthreads();
  const int r = incl - v + s_warp[w];
  *total = s_warp[32];
  return r;
}

__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(
    const int32_t* __restrict__ hist, int nb, int E, int32_t* __restrict__ base,
    int64_t* __restrict__ counts, int64_t* __restrict__ offsets,
    int32_t* __restrict__ tile_base) {
  pdl_launch_dependents();
  pdl_wait();  // the top-k kernel's histograms
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int U = 8;
  if (blockIdx.x + 1 < gridDim.x) {
    // ----- a row CTA
    const int e = blockIdx.x * kScanWarps + warp;
    if (e >= E) return;  // warp-uniform; no block-wide barrier follows
    const int32_t* row = hist + (int64_t)e * nb;
    int32_t* out = base + (int64_t)e * nb;
    int run = 0;
    for (int c0 = 0; c0 < nb; c0 += 32 * U) {
      int v[U], incl[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int b = c0 + 32 * u + lane;
        v[u] = b < nb ? row[b] : 0;
        incl[u] = v[u];
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int o = __shfl_up_sync(0xffffffffu, incl[u], off);
          if (lane >= off) incl[u] += o;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int b = c0 + 32 * u + lane;
        if (b < nb) out[b] = run + incl[u] - v[u];
        run += __shfl_sync(0xffffffffu, incl[u], 31);
      }
    }
    return;
  }
  // ----- the totals CTA: every row's sum, R rows per warp at a time
  __shared__ int s_tot[1024];
  __shared__ int s_warp[33];
  constexpr int R = 8;
  for (int e0 = warp; e0 < E; e0 += kScanWarps * R) {
    int sum[R];
#pragma unroll
    for (int r = 0; r < R; ++r) sum[r] = 0;
    for (int c0 = 0; c0 < nb; c0 += 32 * U) {
      int v[R][U];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = e0 + kScanWarps * r;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int b = c0 + 32 * u + lane;
          v[r][u] = e < E && b < nb ? hist[(int64_t)e * nb + b] : 0;
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int u = 0; u < U; ++u) sum[r] += v[r][u];
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = e0 + kScanWarps * r;
      const int t = __reduce_add_sync(0xffffffffu, sum[r]);
      if (lane == 0 && e < E) s_tot[e] = t;
    }
  }
  __syncthreads();
  // E <= 1024 totals, PER per thread in expert order
  constexpr int PER = 1024 / kScanThreads;
  int c[PER], tsum = 0, tl = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int x = tid * PER + i;
    c[i] = x < E ? s_tot[x] : 0;
    tsum += c[i];
    tl += (c[i] + 127) / 128;
  }
  int sum = 0, tiles = 0;
  int run = block_excl_scan(tsum, s_warp, &sum);
  __syncthreads();
  int trun = block_excl_scan(tl, s_warp, &tiles);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int x = tid * PER + i;
    if (x < E) {
      counts[x] = c[i];
      offsets[x] = run;
      if (tile_base) tile_base[x] = trun;
    }
    run += c[i];
    trun += (c[i] + 127) / 128;
  }
  if (tid == 0) {
    offsets[E] = sum;
    if (tile_base) tile_base[E] = tiles;
  }
}

// One token's row, by one warp, in chunks of 32 MX blocks: lane l of chunk c
// takes the row's 32-element block 32 c + l, quantizes it once and writes its
// payload and scale byte to the k destination rows dest[0..k) (sfrow: their
// tiled-layout rows), or copies the bf16 block there (two-step mode).
// kQ: 0 = bf16 rows to xp; 1 = MXFP8 (xq [M, H] e4m3); 2 = MXFP4 (xq [M, H/2]
// packed e2m1, the W4A4 path).  kTiled: xs goes to the MMA-ready tiled scale
// layout (tiled_scales.h) instead of [M, H/32]; requires H % 128 == 0 and the
// experts' tile bases.
//
// A quantized chunk: the lane's payload words (4 for MXFP4), its scale byte,
// and on lanes 4i the scale word of blocks 4i .. 4i + 3 (the scale bytes of
// four consecutive blocks are four consecutive bytes of a destination row:
// tiled layout always, [M, H/32] when H/32 is a multiple of 4, so one lane
// stores the four as one word).
struct QuantChunk {
  uint32_t o[8];
  uint32_t sb, sw;
};

template <int kQ, bool kV8>
__device__ __forceinline__ void quant_chunk(const uint16_t* __restrict__ xr, int H32, int j0,
                                            int lane, QuantChunk& q) {
  const int blk = j0 + lane;
  q.sb = 0;
  if (blk < H32) {
    uint32_t w[16];
    load_block32_bf16<kV8>(xr + blk * 32, w);
    if (kQ == 2) q.sb = quant_block32_bf16_fp4(w, *reinterpret_cast<uint32_t(*)[4]>(&q.o[0]));
    else q.sb = quant_block32_bf16(w, q.o);
  }
  q.sw = q.sb;
  q.sw |= __shfl_down_sync(0xffffffffu, q.sb, 1) << 8;
  q.sw |= __shfl_down_sync(0xffffffffu, q.sb, 2) << 16;
  q.sw |= __shfl_down_sync(0xffffffffu, q.sb, 3) << 24;
}

template <int kQ, bool kTiled, bool kV8>
__device__ __forceinline__ void store_chunk(const QuantChunk& q, int H, int k, int j0, int lane,
                                            const int64_t* dest, const int64_t* sfrow,
                                            uint8_t* __restrict__ xq, uint8_t* __restrict__ xs) {
  const int H32 = H / 32;
  const int blk = j0 + lane;
  if (blk >= H32) return;
  const bool words = kTiled || (H32 & 3) == 0;
  const bool lead = (lane & 3) == 0;
  for (int j = 0; j < k; ++j) {
    const int64_t d = dest[j];
    if (kQ == 2)
      st_cs_v4(xq + d * (H / 2) + blk * 16, make_uint4(q.o[0], q.o[1], q.o[2], q.o[3]));
    else
      store_block32_e4m3<kV8>(xq + d * H + blk * 32, q.o);
    if (words) {
      if (lead) {
        const int64_t off = kTiled ? tiled_scale_offset(sfrow[j], blk, H / 128) : d * H32 + blk;
        *reinterpret_cast<uint32_t*>(xs + off) = q.sw;
      }
    } else {
      xs[d * H32 + blk] = (uint8_t)q.sb;
    }
  }
}

// Chunks [c0, ...) of the row: load, quantize (or copy) and store.
template <int kQ, bool kTiled, bool kV8>
__device__ __forceinline__ void permute_token_row(const uint16_t* __restrict__ xr, int H, int k,
                                                  int lane, const int64_t* dest,
                                                  const int64_t* sfrow, uint8_t* __restrict__ xq,
                                                  uint8_t* __restrict__ xs,
                                                  uint16_t* __restrict__ xp, int c0 = 0,
                                                  int cstep = 1) {
  const int H32 = H / 32;
  for (int j0 = 32 * c0; j0 < H32; j0 += 32 * cstep) {  // warp-uniform
    if (kQ == 0) {
      const int blk = j0 + lane;
      if (blk >= H32) continue;
      uint32_t w[16];
      load_block32_bf16<kV8>(xr + blk * 32, w);
      for (int j = 0; j < k; ++j) {
        uint16_t* dst = xp + dest[j] * H + blk * 32;
        if (kV8) {
          st_cs_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(&w[0]));
          st_cs_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(&w[8]));
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_cs_v4(dst + 8 * i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
        }
      }
      continue;
    }
    QuantChunk q;
    quant_chunk<kQ, kV8>(xr, H32, j0, lane, q);
    store_chunk<kQ, kTiled, kV8>(q, H, k, j0, lane, dest, sfrow, xq, xs);
  }
}

// The permutation: a warp per token computes its k destination rows (offset
// + the block's base inside the expert + the in-block rank) and moves the row.
// The row x[t] is an input of the routing step, complete before its first
// kernel (an ordinary launch) started, and this kernel starts only after that
// one did: so the first kPermPre chunks of the row are loaded and quantized
// before the wait for the routing results, while the kernels before finish.
constexpr int kPermPre = 1;

template <int kQ, bool kTiled, bool kV8>
__global__ void __launch_bounds__(kRouteThreads) route_permute_kernel(
    const uint16_t* __restrict__ x, int T, int H, int E, int k,
    const int32_t* __restrict__ topk_ids, const int32_t* __restrict__ block_base,
    const int64_t* __restrict__ offsets, const int32_t* __restrict__ tile_base,
    int32_t* __restrict__ src_to_sorted, int32_t* __restrict__ sorted_to_src,
    uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, uint16_t* __restrict__ xp) {
  __shared__ int64_t s_dest[kRouteWarps][32];
  __shared__ int64_t s_sfrow[kRouteWarps][32];  // tiled layout: 128-row block and row
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;  // warp-uniform
  const uint16_t* xr = x + (int64_t)t * H;
  const int H32 = H / 32;
  QuantChunk pre[kPermPre];
  if constexpr (kQ != 0) {
#pragma unroll
    for (int c = 0; c < kPermPre; ++c)
      if (32 * c < H32) quant_chunk<kQ, kV8>(xr, H32, 32 * c, lane, pre[c]);  // warp-uniform
  }
  pdl_wait();  // ids, ranks, block bases and offsets of the two kernels before
  const int b = t / kRouteTokensPerBlock;
  const int nbk = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  if (lane < k) {
    const int64_t f = (int64_t)t * k + lane;
    const int e = topk_ids[f];
    const int64_t dest = offsets[e] + block_base[(int64_t)e * nbk + b] + src_to_sorted[f];
    src_to_sorted[f] = (int32_t)dest;
    sorted_to_src[dest] = (int32_t)f;
    s_dest[warp][lane] = dest;
    if (kTiled) {
      const int64_t within = dest - offsets[e];
      s_sfrow[warp][lane] = ((int64_t)tile_base[e] + within / 128) * 128 + (within % 128);
    }
  }
  __syncwarp();
  if constexpr (kQ != 0) {
#pragma unroll
    for (int c = 0; c < kPermPre; ++c)
      if (32 * c < H32)
        store_chunk<kQ, kTiled, kV8>(pre[c], H, k, 32 * c, lane, s_dest[warp], s_sfrow[warp], xq,
                                     xs);
  }
  permute_token_row<kQ, kTiled, kV8>(xr, H, k, lane, s_dest[warp], s_sfrow[warp], xq, xs, xp,
                                     kQ != 0 ? kPermPre : 0);
}

// Small batches (T <= one 64-token routing block): the whole routing step in
// one kernel, launched as one cluster of G = ceil(T / TPC) <= 8 CTAs with
// TPC = ceil(T / 8) tokens each.  CTA c takes the top-k of its tokens
// c TPC, c TPC + 1, ... (a warp per token), writes their ids and weights and
// marks them in its expert masks; after a cluster barrier every CTA ORs the G
// masks (distributed shared memory) into the expert counts, offsets and
// tiled-scale row-block bases, and permutes its own tokens, each row split
// over kSplit warps by 32-block chunk (p, p + kSplit, ...).  CTA 0 writes the
// counts, offsets and tile bases.  Same selection, weights, in-block ranks
// and offsets as the three-kernel path.
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallMaxCtas = 8;  // portable cluster size
constexpr int kSmallMaxE = 256;

__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 64-bit load from the shared memory of CTA `rank` of the cluster, at the
// offset of this CTA's `p`
__device__ __forceinline__ unsigned long long ld_peer_u64(const void* p, uint32_t rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t ra;
  unsigned long long v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(ra) : "memory");
  return v;
}

template <int EPL, int kQ, bool kTiled, bool kV8>
__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ logits, int T, int H, int E, int k,
    int renormalize, int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
    int32_t* __restrict__ src_to_sorted, int32_t* __restrict__ sorted_to_src,
    int64_t* __restrict__ counts, int64_t* __restrict__ offsets, int32_t* __restrict__ tile_base,
    uint8_t* __restrict__ xq, uint8_t* __restrict__ xs, uint16_t* __restrict__ xp, int tpc,
    int kSplit, int32_t* __restrict__ zero_e) {
  __shared__ unsigned long long s_mine[kSmallMaxE];  // bit t: this CTA's token t chose e
  __shared__ unsigned long long s_mask[kSmallMaxE];  // bit t: token t chose e (all CTAs)
  __shared__ int s_ids[kSmallWarps][32];             // this CTA's tokens' experts
  __shared__ int s_off[kSmallMaxE];
  __shared__ int s_tb[kSmallMaxE];
  __shared__ int s_warp[33];
  __shared__ int64_t s_dest[kSmallWarps][32];
  __shared__ int64_t s_sfrow[kSmallWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t_first = (int)blockIdx.x * tpc;
  // the grouped GEMM after the routing may be scheduled now (its CTAs set
  // up on the free SMs and wait for this grid's results before reading them)
  pdl_launch_dependents();
  // this CTA's rows start their way into L2 now, so the DRAM latency of
  // their loads hides behind the top-k and the scan
  if (lane == 0 && warp < tpc && t_first + warp < T)
    prefetch_l2_bulk(x + (int64_t)(t_first + warp) * H, (uint32_t)H * 2u);
  if (tid < E) s_mine[tid] = 0ull;
  __syncthreads();
  // ---- top-k of this CTA's tokens, a warp per token
  if (warp < tpc && t_first + warp < T) {  // warp-uniform
    const int t = t_first + warp;
    const float* rows[1] = {logits + (int64_t)t * E};
    int c[1];
    float v[1], w[1];
    warp_topk_softmax<EPL, 1>(rows, E, k, renormalize != 0, lane, c, v, w);
    if (lane < k) {
      s_ids[warp][lane] = c[0];
      atomicOr(&s_mine[c[0]], 1ull << t);
      topk_ids[(int64_t)t * k + lane] = c[0];
      topk_w[(int64_t)t * k + lane] = w[0];
    }
  }
  // every CTA's masks are complete; OR them together, then a second barrier
  // keeps each CTA's masks alive until all the others have read them
  __syncwarp();
  cluster_barrier();
  if (tid < E) {
    unsigned long long m = 0ull;
    for (uint32_t r = 0; r < gridDim.x; ++r) m |= ld_peer_u64(&s_mine[tid], r);
    s_mask[tid] = m;
  }
  __syncwarp();
  cluster_barrier();
  // ---- expert counts -> offsets and tiled-scale row-block bases (one
  // expert per thread, E <= 256)
  const int c0 = tid < E ? __popcll(s_mask[tid]) : 0;
  int sum = 0;
  const int ex = block_excl_scan(c0, s_warp, &sum);
  if (tid < E) s_off[tid] = ex;
  __syncthreads();
  const int t0c = (c0 + 127) / 128;
  int tsum = 0;
  const int tex = block_excl_scan(t0c, s_warp, &tsum);
  if (tid < E) s_tb[tid] = tex;
  if (blockIdx.x == 0) {
    if (tid < E) { counts[tid] = c0; offsets[tid] = ex; if (tile_base) tile_base[tid] = tex; }
    if (tid == 0) { offsets[E] = sum; if (tile_base) tile_base[E] = tsum; }
    if (zero_e != nullptr && tid < E) zero_e[tid] = 0;
  }
  __syncthreads();
  // ---- the permutation: token t = this CTA's token warp % tpc, row part
  // warp / tpc of kSplit (every part's warp computes the destinations; part
  // 0 writes the index maps)
  const int part = warp / tpc, tl = warp % tpc;
  const int t = t_first + tl;
  if (part >= kSplit || t >= T) return;  // warp-uniform
  if (lane < k) {
    const int e = s_ids[tl][lane];
    const int64_t f = (int64_t)t * k + lane;
    const int64_t rank = __popcll(s_mask[e] & ((1ull << t) - 1ull));
    const int64_t dest = s_off[e] + rank;
    if (part == 0) {
      src_to_sorted[f] = (int32_t)dest;
      sorted_to_src[dest] = (int32_t)f;
    }
    s_dest[warp][lane] = dest;
    if (kTiled) s_sfrow[warp][lane] = ((int64_t)s_tb[e] + rank / 128) * 128 + (rank % 128);
  }
  __syncwarp();
  permute_token_row<kQ, kTiled, kV8>(x + (int64_t)t * H, H, k, lane, s_dest[warp], s_sfrow[warp],
                                     xq, xs, xp, part, kSplit);
}

template <int EPL, int kQ, bool kTiled, bool kV8>
static cudaError_t launch_small(int grid, int tpc, int split, cudaStream_t stream,
                                const uint16_t* x, const float* logits, int T, int H, int E,
                                int k, int rn, int32_t* ids, float* w, int32_t* s2s,
                                int32_t* src2s, int64_t* counts, int64_t* offsets, int32_t* tb,
                                uint8_t* xq, uint8_t* xs, uint16_t* xp, int32_t* zero_e) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)grid;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_small_kernel<EPL, kQ, kTiled, kV8>, x, logits, T, H, E,
                            k, rn, ids, w, s2s, src2s, counts, offsets, tb, xq, xs, xp, tpc,
                            split, zero_e);
}

// Routing scratch: the histograms [E][nb], then the scan's block bases
// [E][nb], each piece 256-byte aligned.
size_t route_hist_bytes(int T, int E) {
  const int64_t nb = ceil_div(T, kRouteTokensPerBlock);
  const size_t b = (size_t)(nb > 0 ? nb : 1) * (size_t)E * sizeof(int32_t);
  return (b + 255) & ~(size_t)255;
}
size_t route_workspace_bytes(int T, int E) { return 2 * route_hist_bytes(T, E); }

template <int EPL>
static void launch_topk(int nb, size_t smem, cudaStream_t stream, const float* logits, int T,
                        int E, int k, int renorm, int32_t* ids, float* w, int32_t* rank,
                        int32_t* hist) {
  constexpr int threads = 32 * (kRouteTokensPerBlock / topk_tokens_per_warp<EPL>());
  if (k == 8)  // the common top-8: its selection rounds unrolled
    route_topk_rank_kernel<EPL, topk_tokens_per_warp<EPL>(), 8>
        <<<nb, threads, smem, stream>>>(logits, T, E, k, renorm, ids, w, rank, hist);
  else
    route_topk_rank_kernel<EPL><<<nb, threads, smem, stream>>>(logits, T, E, k, renorm, ids, w,
                                                               rank, hist);
}

cudaError_t launch_route(const uint16_t* x, const float* logits, int T, int H, int E, int k,
                         bool renormalize, int quant, uint8_t* xq, uint8_t* xs, uint16_t* xp,
                         int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                         int32_t* src_to_sorted, int64_t* counts, int64_t* offsets,
                         int32_t* block_hist, cudaStream_t stream, int32_t* tile_base,
                         bool topk_done, int32_t* zero_e) {
  if (quant == 2 && !tile_base) return cudaErrorNotSupported;  // MXFP4 rows: tiled scales only
  if (T == 0) {
    cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int64_t) * E, stream);
    if (err != cudaSuccess) return err;
    return cudaMemsetAsync(offsets, 0, sizeof(int64_t) * (E + 1), stream);
  }
  const int nb = (int)ceil_div(T, kRouteTokensPerBlock);
  if (!topk_done && nb == 1 && E <= kSmallMaxE) {
    // one routing block: the single-kernel path (one cluster)
    const int epl_s = (E + 31) / 32;
    const int tpc = (int)ceil_div(T, kSmallMaxCtas);
    const int grid = (int)ceil_div(T, tpc);
    const int rn_s = renormalize ? 1 : 0;
    // warps per token row in the permutation: one per 32-block chunk
    const int split = (int)std::min<int64_t>(kSmallWarps / tpc, ceil_div(H / 32, 32));
    // 32-byte loads and stores (half the store instructions, which bound the
    // permutation here) when the rows allow them
    const bool v8s = ((uintptr_t)x & 31u) == 0 &&
                     ((uintptr_t)(quant ? (const void*)xq : (const void*)xp) & 31u) == 0;
    cudaError_t err;
#define MXMOE_SMALL_V(EPL, Q, TL, V)                                                              \
  err = launch_small<EPL, Q, TL, V>(grid, tpc, split, stream, x, logits, T, H, E, k, rn_s,       \
                                    topk_ids, topk_w, src_to_sorted, sorted_to_src, counts,      \
                                    offsets, tile_base, Q ? xq : nullptr, Q ? xs : nullptr,      \
                                    Q ? nullptr : xp, zero_e)
#define MXMOE_SMALL(EPL, Q, TL)                                                                   \
  do {                                                                                            \
    if (v8s) MXMOE_SMALL_V(EPL, Q, TL, true);                                                     \
    else MXMOE_SMALL_V(EPL, Q, TL, false);                                                        \
  } while (0)
#define MXMOE_SMALL_Q(EPL)                                                                        \
  if (quant == 2) MXMOE_SMALL(EPL, 2, true);                                                      \
  else if (quant && tile_base) MXMOE_SMALL(EPL, 1, true);                                         \
  else if (quant) MXMOE_SMALL(EPL, 1, false);                                                     \
  else MXMOE_SMALL(EPL, 0, false)
    if (epl_s <= 1) { MXMOE_SMALL_Q(1); }
    else if (epl_s <= 2) { MXMOE_SMALL_Q(2); }
    else if (epl_s <= 4) { MXMOE_SMALL_Q(4); }
    else { MXMOE_SMALL_Q(8); }
#undef MXMOE_SMALL_Q
#undef MXMOE_SMALL
#undef MXMOE_SMALL_V
    return err;
  }
  if (zero_e) {
    const cudaError_t zerr = cudaMemsetAsync(zero_e, 0, sizeof(int32_t) * (size_t)E, stream);
    if (zerr != cudaSuccess) return zerr;
  }
  const size_t smem1 = sizeof(unsigned long long) * (size_t)E;
  const int epl = (E + 31) / 32;
  const int rn = renormalize ? 1 : 0;
  // src_to_sorted holds the in-block rank between kernels 1 and 3.  topk_done:
  // the fused router (router.cu) already wrote ids, weights, ranks and
  // histograms.
  if (topk_done) {
  } else if (epl <= 1)       launch_topk<1>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist);
  else if (epl <= 2)  launch_topk<2>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist);
  else if (epl <= 4)  launch_topk<4>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist);
  else if (epl <= 8)  launch_topk<8>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist);
  else if (epl <= 16) launch_topk<16>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist);
  else                launch_topk<32>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  // the scan and the permutation start early (programmatic dependent
  // launch) and wait on the device for their predecessor's results
  int32_t* block_base = block_hist + route_hist_bytes(T, E) / sizeof(int32_t);
  err = launch_pdl(route_scan_kernel, dim3((unsigned)ceil_div(E, kScanWarps) + 1u),
                   dim3(kScanThreads), 0, stream, (const int32_t*)block_hist, nb, E, block_base,
                   counts, offsets, tile_base);
  if (err != cudaSuccess) return err;

  const int nb3 = (int)ceil_div(T, kRouteWarps);
  const bool v8 = ((uintptr_t)x & 31u) == 0 && ((uintptr_t)(quant ? (const void*)xq : (const void*)xp) & 31u) == 0;
#define MXMOE_PERMUTE(Q, TL, V)                                                                   \
  err = launch_pdl(route_permute_kernel<Q, TL, V>, dim3(nb3), dim3(kRouteThreads), 0, stream,  \
      x, T, H, E, k, (const int32_t*)topk_ids, (const int32_t*)block_base,                     \
      (const int64_t*)offsets, (const int32_t*)(TL ? tile_base : nullptr), src_to_sorted,     \
      sorted_to_src, Q ? xq : nullptr, Q ? xs : nullptr, Q ? nullptr : xp)
  if (quant == 2) {
    if (v8) MXMOE_PERMUTE(2, true, true); else MXMOE_PERMUTE(2, true, false);
  } else if (quant && tile_base) {
    if (v8) MXMOE_PERMUTE(1, true, true); else MXMOE_PERMUTE(1, true, false);
  } else if (quant) {
    if (v8) MXMOE_PERMUTE(1, false, true); else MXMOE_PERMUTE(1, false, false);
  } else {
    if (v8) MXMOE_PERMUTE(0, false, true); else MXMOE_PERMUTE(0, false, false);
  }
#undef MXMOE_PERMUTE
  return err;
}

}  // namespace mxmoe
