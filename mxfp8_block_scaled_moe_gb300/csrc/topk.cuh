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

// NT tokens per call, each with the same arithmetic as a call for that token
// alone (the tokens only share the warp's instruction stream, so the latency
// of one token's warp reductions hides behind the others').  rows[n] points
// at token n's E fp32 logits (global or shared memory), or is null for no
// token; lane l reads experts l, l + 32, ..., l + 32 (EPL - 1).  On lanes
// j < k: ids[n] / vals[n] / ws[n] are token n's j-th chosen expert, its logit
// and its weight.  The softmax sums run per lane in increasing expert order,
// then over the lanes by an xor butterfly.
template <int EPL, int NT>
__device__ __forceinline__ void warp_topk_softmax(const float* const (&rows)[NT], int E, int k,
                                                  bool renormalize, int lane, int (&ids)[NT],
                                                  float (&vals)[NT], float (&ws)[NT]) {
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
  // k rounds: the warp's largest remaining key (redux max), ties to the
  // lowest expert id among the lanes holding it (redux min); within a lane
  // the lowest index wins a tie (strict compare in increasing i).
  uint32_t taken[NT], my_key[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) { taken[n] = 0; my_key[n] = 0; ids[n] = 0; }
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
  // softmax weights of the chosen experts
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    vals[n] = key_value(my_key[n]);
    const float vmax = __shfl_sync(0xffffffffu, vals[n], 0);
    float denom;
    if (renormalize) {
      float ej = lane < k ? expf(vals[n] - vmax) : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ej += __shfl_xor_sync(0xffffffffu, ej, off);
      denom = ej;
    } else {
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) sum += expf(v[n][i] - vmax);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      denom = sum;
    }
    ws[n] = expf(vals[n] - vmax) / denom;
  }
}

}  // namespace mxmoe
