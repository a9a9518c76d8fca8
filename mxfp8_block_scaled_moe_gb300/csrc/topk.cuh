// Warp-cooperative top-k softmax of router logits, shared by the logits-input
// routing kernel (route.cu) and the fused router gate (router.cu), so both
// give the same bytes on the same fp32 logits.
//
// Top-k routing ("Quantization on Ascend", MoE forward: routing; the
// softmax / renormalise form of Qwen3-MoE): the k largest logits, ties to the
// lower expert id, in descending order; weights softmax(logits)[e] of the
// chosen experts, divided by their own sum when `renormalize`.
#pragma once

#include "common.cuh"

namespace mxmoe {

// Exact rounding error of h = fl(a + b) (Knuth's two-sum; no ordering
// condition on |a|, |b|), written with explicit round-to-nearest adds so the
// compiler cannot reassociate them.
__device__ __forceinline__ float two_sum_err(float a, float b, float h) {
  const float bb = __fsub_rn(h, a);
  return __fadd_rn(__fsub_rn(a, __fsub_rn(h, bb)), __fsub_rn(b, bb));
}

// e^(v - m) with the difference carried exactly: hi = fl(v - m), lo its
// rounding error, e^(hi + lo) = e^hi + e^hi * lo to first order in lo.
__device__ __forceinline__ float exp_of_difference(float v, float m) {
  const float hi = __fsub_rn(v, m);
  const float lo = two_sum_err(v, -m, hi);
  const float e = expf(hi);
  return __fmaf_rn(e, lo, e);
}

// NT tokens per call, each with the same arithmetic as a call for that token
// alone (the tokens only share the warp's instruction stream, so the latency
// of one token's warp reductions hides behind the others').  rows[n] points
// at token n's E fp32 logits (global or shared memory), or is null for no
// token; lane l reads experts l, l + 32, ..., l + 32 (EPL - 1).  On lanes
// j < k: ids[n] / vals[n] / ws[n] are token n's j-th chosen expert, its logit
// and its weight.
//
// Selection: k rounds of the warp's largest remaining key (redux max), ties
// to the lowest expert id among the lanes holding it (redux min).  For
// EPL <= 4 each lane first sorts its own EPL (key, id) pairs (descending key,
// ties to the lower id, i.e. a stable sort of the lane's experts), so a round
// reads the lane's head and, on a win, shifts the lane's list by one; wider
// rows rescan the lane's live entries every round.  KC > 0: the caller
// guarantees k == KC, and the EPL <= 4 rounds are unrolled (measured on
// GB300 with k = 8: the 16K-token route+quant 76.3 against 77.2-78.0 us).
template <int EPL, int NT, int KC = 0>
__device__ __forceinline__ void warp_topk_softmax(const float* const (&rows)[NT], int E, int k_rt,
                                                  bool renormalize, int lane, int (&ids)[NT],
                                                  float (&vals)[NT], float (&ws)[NT]) {
  const int k = KC > 0 ? KC : k_rt;  // a compile-time constant when KC > 0
  float v[NT][EPL];
  uint32_t key[NT][EPL];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      const bool in = rows[n] != nullptr && e < E;
      v[n][i] = in ? rows[n][e] : 0.f;
      key[n][i] = in ? order_key(v[n][i]) : 0u;  // 0: below every finite key
    }
  uint32_t my_key[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) { my_key[n] = 0; ids[n] = 0; }
  if constexpr (EPL <= 4) {
    // the lane's sorted list: sk[n][0] is its current head
    uint32_t sk[NT][EPL], si[NT][EPL];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        sk[n][i] = key[n][i];
        si[n][i] = lane + 32 * i < E ? (uint32_t)(lane + 32 * i) : 0xFFFFFFFFu;
      }
      // stable bubble sort, descending (strict compare keeps the lower id first)
#pragma unroll
      for (int a = 0; a < EPL - 1; ++a)
#pragma unroll
        for (int b = 0; b < EPL - 1 - a; ++b) {
          const bool sw = sk[n][b + 1] > sk[n][b];
          const uint32_t k0 = sk[n][b], k1 = sk[n][b + 1], i0 = si[n][b], i1 = si[n][b + 1];
          sk[n][b] = sw ? k1 : k0;
          sk[n][b + 1] = sw ? k0 : k1;
          si[n][b] = sw ? i1 : i0;
          si[n][b + 1] = sw ? i0 : i1;
        }
    }
#pragma unroll
    for (int j = 0; j < k; ++j) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const uint32_t hk = sk[n][0], hid = si[n][0];
        const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t id = __reduce_min_sync(0xffffffffu, hk == m ? hid : 0xFFFFFFFFu);
        const bool win = hid == id;
#pragma unroll
        for (int i = 0; i < EPL - 1; ++i) {
          sk[n][i] = win ? sk[n][i + 1] : sk[n][i];
          si[n][i] = win ? si[n][i + 1] : si[n][i];
        }
        if (win) { sk[n][EPL - 1] = 0u; si[n][EPL - 1] = 0xFFFFFFFFu; }
        if (lane == j) { ids[n] = (int)id; my_key[n] = m; }
      }
    }
  } else {
    // within a lane the lowest index wins a tie (strict compare in increasing i)
    uint32_t taken[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) taken[n] = 0;
    for (int j = 0; j < k; ++j) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        uint32_t hk = 0u, hid = 0xFFFFFFFFu;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const bool live = lane + 32 * i < E && !((taken[n] >> i) & 1u);
          if (live && (hid == 0xFFFFFFFFu || key[n][i] > hk)) {
            hk = key[n][i];
            hid = (uint32_t)(lane + 32 * i);
          }
        }
        const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t id = __reduce_min_sync(0xffffffffu, hk == m ? hid : 0xFFFFFFFFu);
        if (hid == id) taken[n] |= 1u << (id >> 5);
        if (lane == j) { ids[n] = (int)id; my_key[n] = m; }
      }
    }
  }
  // softmax weights of the chosen experts.  Every exponent argument
  // a = v - vmax is carried exactly as an fp32 pair (hi + lo, Knuth's
  // two-sum), e^a = e^hi (1 + lo) to first order, and the denominator is a
  // compensated sum (each addition's exact rounding error kept in a second
  // fp32 word), so the weights carry only the fp32 exp error and the final
  // roundings: a few 1e-7 relative to the exact softmax.  xor butterflies
  // leave the same bits on every lane (fp32 addition and the two-sum error
  // are both symmetric in their operands); renormalized sums run only the
  // butterfly levels that lanes 0..k-1 need.
  int kp = 1;
  while (kp < k) kp <<= 1;
  if (NT == 2 && renormalize && k <= 16) {
    // both tokens in one pass: token n's slot j on lane 16 n + j (the
    // butterfly's levels below kp <= 16 stay inside each half, so every
    // weight gets the bits of the one-token pass)
    const int j = lane & 15;
    const float a = __shfl_sync(0xffffffffu, key_value(my_key[0]), j);
    const float b = __shfl_sync(0xffffffffu, key_value(my_key[NT - 1]), j);
    const float val = lane < 16 ? a : b;
    const float vmax = __shfl_sync(0xffffffffu, val, lane & 16);
    const float mine = j < k ? exp_of_difference(val, vmax) : 0.f;
    float s_hi = mine, s_lo = 0.f;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
      if (off >= kp) continue;  // warp-uniform
      const float oh = __shfl_xor_sync(0xffffffffu, s_hi, off);
      const float ol = __shfl_xor_sync(0xffffffffu, s_lo, off);
      const float h = __fadd_rn(s_hi, oh);
      s_lo = __fadd_rn(__fadd_rn(s_lo, ol), two_sum_err(s_hi, oh, h));
      s_hi = h;
    }
    const float w = __fdiv_rn(mine, __fadd_rn(s_hi, s_lo));
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      vals[n] = key_value(my_key[n]);
      ws[n] = __shfl_sync(0xffffffffu, w, 16 * n + j);
    }
    return;
  }
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    vals[n] = key_value(my_key[n]);
    const float vmax = __shfl_sync(0xffffffffu, vals[n], 0);
    const float mine = lane < k ? exp_of_difference(vals[n], vmax) : 0.f;
    float s_hi = 0.f, s_lo = 0.f;
    if (renormalize) {
      s_hi = mine;
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          const float t = exp_of_difference(v[n][i], vmax);
          const float h = __fadd_rn(s_hi, t);
          s_lo = __fadd_rn(s_lo, two_sum_err(s_hi, t, h));
          s_hi = h;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      if (renormalize && off >= kp) continue;  // warp-uniform
      const float oh = __shfl_xor_sync(0xffffffffu, s_hi, off);
      const float ol = __shfl_xor_sync(0xffffffffu, s_lo, off);
      const float h = __fadd_rn(s_hi, oh);
      s_lo = __fadd_rn(__fadd_rn(s_lo, ol), two_sum_err(s_hi, oh, h));
      s_hi = h;
    }
    const float denom = __fadd_rn(s_hi, s_lo);
    ws[n] = __fdiv_rn(mine, denom);
  }
}

}  // namespace mxmoe
