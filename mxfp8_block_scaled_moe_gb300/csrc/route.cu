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
//      block's base row inside each expert) and of the expert totals (offsets).
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


// TPW tokens per warp (kRouteTokensPerBlock / TPW warps per block): four for
// narrow rows, whose warp reductions interleave; two for wide rows, where
// more would not fit in the registers.
template <int EPL>
constexpr int topk_tokens_per_warp() { return EPL <= 4 ? 4 : 2; }

template <int EPL, int TPW = topk_tokens_per_warp<EPL>()>  // logits per lane: E <= 32 * EPL
__global__ void __launch_bounds__(32 * (kRouteTokensPerBlock / TPW)) route_topk_rank_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renormalize,
    int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
    int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
    const uint16_t* __restrict__ x_prefetch, int H) {
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
  // the block's hidden-state rows (contiguous) head for L2 while the top-k
  // runs, so the permutation reads them from L2 instead of HBM
  if (x_prefetch && threadIdx.x == 0)
    prefetch_l2_bulk(x_prefetch + (int64_t)t0 * H, (uint64_t)nt * H * 2);

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
    warp_topk_softmax<EPL, NT>(rows, E, k, renormalize != 0, lane, c, v, w);
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

// One block of 1024 threads over the expert-major histogram hist[e][b] (nb
// blocks per row).  Each warp takes whole expert rows (e = warp, warp + 32,
// ...): 32 consecutive blocks per load, a shuffle scan per 32, and the row is
// rewritten as its exclusive prefix (the block's base row inside expert e).
// Then the expert totals are scanned into counts, offsets and the experts'
// first 128-row blocks of the tiled scale layout.
constexpr int kScanThreads = 1024;

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Exclusive scan of one value per thread over the block (values of threads
// >= n count as 0); *total receives the sum.  s_warp: 32 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int incl = warp_incl_scan(v, lane);
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = s_warp[lane];
    const int xi = warp_incl_scan(x, lane);
    s_warp[lane] = xi - x;
    if (lane == 31) s_warp[32] = xi;
  }
  __syncthreads();
  const int r = incl - v + s_warp[w];
  *total = s_warp[32];
  return r;
}

__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(int32_t* __restrict__ hist,
                                                                  int nb, int E,
                                                                  int64_t* __restrict__ counts,
                                                                  int64_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ tile_base) {
  pdl_launch_dependents();
  pdl_wait();  // the top-k kernel's histograms
  __shared__ int s_tot[1024];
  __shared__ int s_warp[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int U = 8;  // 32-block chunks loaded together
  for (int e = warp; e < E; e += kScanThreads / 32) {
    int32_t* row = hist + (int64_t)e * nb;
    int run = 0;
    for (int c0 = 0; c0 < nb; c0 += 32 * U) {
      int v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int b = c0 + 32 * u + lane;
        v[u] = b < nb ? row[b] : 0;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int b = c0 + 32 * u + lane;
        const int incl = warp_incl_scan(v[u], lane);
        if (b < nb) row[b] = run + incl - v[u];
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) s_tot[e] = run;
  }
  __syncthreads();
  // expert totals -> counts and offsets (E <= 1024: one expert per thread)
  const int v = tid < E ? s_tot[tid] : 0;
  int sum = 0;
  const int excl = block_excl_scan(v, s_warp, &sum);
  if (tid < E) {
    counts[tid] = v;
    offsets[tid] = excl;
  }
  if (tid == 0) offsets[E] = sum;
  if (tile_base == nullptr) return;
  // exclusive prefix of the experts' 128-row tile counts (tiled scale layout)
  __syncthreads();
  const int tv = (v + 127) / 128;
  int tsum = 0;
  const int texcl = block_excl_scan(tv, s_warp, &tsum);
  if (tid < E) tile_base[tid] = texcl;
  if (tid == 0) tile_base[E] = tsum;
}

// kQ: 0 = bf16 rows to xp; 1 = MXFP8 (xq [M, H] e4m3); 2 = MXFP4 (xq [M, H/2]
// packed e2m1, the W4A4 path).  kTiled: xs goes to the MMA-ready tiled scale
// layout (tiled_scales.h) instead of [M, H/32]; requires H % 128 == 0 and the
// experts' tile bases.
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
  pdl_wait();  // ids, ranks, block bases and offsets of the two kernels before
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;  // warp-uniform
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
  // one lane = one 32-element block of the row: quantized once, written to
  // the k destination rows (32 B of payload + 1 scale byte each)
  const uint16_t* xr = x + (int64_t)t * H;
  const int H32 = H / 32;
  for (int j0 = 0; j0 < H32; j0 += 32) {
    const int blk = j0 + lane;
    if (blk >= H32) break;
    uint32_t w[16];
    load_block32_bf16<kV8>(xr + blk * 32, w);
    if (kQ == 2) {
      uint32_t o[4];
      const uint32_t sb = quant_block32_bf16_fp4(w, o);
      for (int j = 0; j < k; ++j) {
        const int64_t d = s_dest[warp][j];
        st_cs_v4(xq + d * (H / 2) + blk * 16, make_uint4(o[0], o[1], o[2], o[3]));
        if (kTiled)
          xs[tiled_scale_offset(s_sfrow[warp][j], blk, H / 128)] = (uint8_t)sb;
        else
          xs[d * H32 + blk] = (uint8_t)sb;
      }
    } else if (kQ == 1) {
      uint32_t o[8];
      const uint32_t sb = quant_block32_bf16(w, o);
      for (int j = 0; j < k; ++j) {
        const int64_t d = s_dest[warp][j];
        store_block32_e4m3<kV8>(xq + d * H + blk * 32, o);
        if (kTiled)
          xs[tiled_scale_offset(s_sfrow[warp][j], blk, H / 128)] = (uint8_t)sb;
        else
          xs[d * H32 + blk] = (uint8_t)sb;
      }
    } else {
      for (int j = 0; j < k; ++j) {
        uint16_t* dst = xp + s_dest[warp][j] * H + blk * 32;
        if (kV8) {
          st_cs_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(&w[0]));
          st_cs_v8(dst + 16, *reinterpret_cast<const uint32_t(*)[8]>(&w[8]));
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_cs_v4(dst + 8 * i, make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]));
        }
      }
    }
  }
}

size_t route_workspace_bytes(int T, int E) {
  const int64_t nb = ceil_div(T, kRouteTokensPerBlock);
  const size_t b = (size_t)(nb > 0 ? nb : 1) * (size_t)E * sizeof(int32_t);
  return (b + 255) & ~(size_t)255;
}

template <int EPL>
static void launch_topk(int nb, size_t smem, cudaStream_t stream, const float* logits, int T,
                        int E, int k, int renorm, int32_t* ids, float* w, int32_t* rank,
                        int32_t* hist, const uint16_t* x, int H) {
  constexpr int threads = 32 * (kRouteTokensPerBlock / topk_tokens_per_warp<EPL>());
  route_topk_rank_kernel<EPL><<<nb, threads, smem, stream>>>(logits, T, E, k, renorm, ids,
                                                                   w, rank, hist, x, H);
}

cudaError_t launch_route(const uint16_t* x, const float* logits, int T, int H, int E, int k,
                         bool renormalize, int quant, uint8_t* xq, uint8_t* xs, uint16_t* xp,
                         int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                         int32_t* src_to_sorted, int64_t* counts, int64_t* offsets,
                         int32_t* block_hist, cudaStream_t stream, int32_t* tile_base,
                         bool topk_done) {
  if (quant == 2 && !tile_base) return cudaErrorNotSupported;  // MXFP4 rows: tiled scales only
  if (T == 0) {
    cudaError_t err = cudaMemsetAsync(counts, 0, sizeof(int64_t) * E, stream);
    if (err != cudaSuccess) return err;
    return cudaMemsetAsync(offsets, 0, sizeof(int64_t) * (E + 1), stream);
  }
  const int nb = (int)ceil_div(T, kRouteTokensPerBlock);
  const size_t smem1 = sizeof(unsigned long long) * (size_t)E;
  const int epl = (E + 31) / 32;
  const int rn = renormalize ? 1 : 0;
  // src_to_sorted holds the in-block rank between kernels 1 and 3.  topk_done:
  // the fused router (router.cu) already wrote ids, weights, ranks and
  // histograms.
  if (topk_done) {
  } else if (epl <= 1)       launch_topk<1>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist, x, H);
  else if (epl <= 2)  launch_topk<2>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist, x, H);
  else if (epl <= 4)  launch_topk<4>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist, x, H);
  else if (epl <= 8)  launch_topk<8>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist, x, H);
  else if (epl <= 16) launch_topk<16>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist, x, H);
  else                launch_topk<32>(nb, smem1, stream, logits, T, E, k, rn, topk_ids, topk_w, src_to_sorted, block_hist, x, H);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  // the scan and the permutation start early (programmatic dependent
  // launch) and wait on the device for their predecessor's results
  err = launch_pdl(route_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, block_hist, nb, E,
                   counts, offsets, tile_base);
  if (err != cudaSuccess) return err;

  const int nb3 = (int)ceil_div(T, kRouteWarps);
  const bool v8 = ((uintptr_t)x & 31u) == 0 && ((uintptr_t)(quant ? (const void*)xq : (const void*)xp) & 31u) == 0;
#define MXMOE_PERMUTE(Q, TL, V)                                                                   \
  err = launch_pdl(route_permute_kernel<Q, TL, V>, dim3(nb3), dim3(kRouteThreads), 0, stream,  \
      x, T, H, E, k, (const int32_t*)topk_ids, (const int32_t*)block_hist,                     \
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
