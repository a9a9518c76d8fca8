// Router gate GEMM fused with softmax top-k (the step upstream of the MoE
// routing: "Quantization on Ascend", MoE MXFP8 notes on the router gate, a
// ReplicatedLinear kept in bf16 online and dequantized on the offline path;
// sglang PR #32266, router-gate commit note).
//
//   logits[t, e] = sum_h x[t, h] * gate[e, h]          bf16 inputs, fp32 accumulate
//   top-k of logits[t, :] (ties to the lower expert id), softmax weights of
//   the chosen experts, renormalized over the k when asked.
//
// One CTA per 128 tokens: warp 0 streams x and gate tiles (64 bf16 of K per
// stage, 128-byte swizzle) by TMA, warp 1 issues tcgen05.mma kind::f16 (M=128
// tokens, N = E rounded up to 16 experts, the gate rows past E zero-filled by
// the TMA, K=16) into a TMEM accumulator, warps 2-17 (four per TMEM
// lane quarter) move the accumulator into shared memory, then take the tokens
// warp by warp with the routing kernel's top-k (topk.cuh) and write ids,
// weights and, when asked, the logits.  The same warps then build the routing
// step's per-64-token expert masks in shared memory and write the in-block
// ranks and per-block histograms, so the permutation continues from here
// (route.cu, scan and permute kernels).
//
// Roofline: HBM-bound on x (2 B per element, read once); the gate (E x H
// bf16) stays in L2 and is re-read by every CTA.
#include "gemm_common.cuh"
#include "topk.cuh"

namespace mxmoe {
namespace router {

using gemm::mbar_arrive_expect_tx;
using gemm::mbar_init;
using gemm::smem_u32;
using gemm::tc_commit;
using gemm::tc_fence_after;
using gemm::tc_fence_before;
using gemm::tma_load_2d;
using gemm::wait_bar;

constexpr int TOK = 128;            // tokens per CTA (the MMA's M)
constexpr int KS = 64;              // bf16 elements of K per stage (one 128-byte row)
constexpr int STAGES = 4;
constexpr int EPI = 16;             // epilogue warps (four per TMEM lane quarter)
constexpr int THREADS = 64 + 32 * EPI;  // producer, MMA, epilogue
constexpr int A_BYTES = TOK * 128;  // 16 KB
constexpr int MAX_E = 256;
constexpr int STAGE_MAX = A_BYTES + MAX_E * 128;
constexpr int OFF_BAR = STAGES * STAGE_MAX;
// epilogue scratch over the stages: fp32 logits [TOK][E | 1], chosen ids [TOK][32]
constexpr int OFF_IDS = TOK * (MAX_E + 1) * 4;
static_assert(OFF_IDS + TOK * 32 * 4 <= OFF_BAR, "epilogue scratch fits in the stages");
constexpr int OFF_MASK = OFF_BAR + 128;                  // uint64 [2][MAX_E]
constexpr int OFF_TMEM = OFF_MASK + 2 * MAX_E * 8;
constexpr int ALLOC = OFF_TMEM + 16 + 1024;              // + alignment slack
static_assert(ALLOC <= 232448, "shared memory");

struct Params {
  int T, H, E, k, renormalize, n_blocks;
  float* logits;
  int32_t* topk_ids;
  float* topk_w;
  int32_t* local_rank;
  int32_t* block_hist;
  int* status;
  long long wait_limit;
};

// kind::f16 instruction descriptor: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 and 10-12 = 1), both K-major, N >> 3 at 17-22, M >> 4 at 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// KC > 0: k == KC (the top-k selection rounds unrolled)
template <int EPL, int KC = 0>
__global__ void __launch_bounds__(THREADS, 1)
    router_gate_topk_kernel(const __grid_constant__ CUtensorMap tmX,
                            const __grid_constant__ CUtensorMap tmG, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int NE = (E + 15) & ~15;  // the MMA's N
  const int stage_bytes = A_BYTES + NE * 128;
  auto bar_full = [&](int s) { return sbase + OFF_BAR + 8u * s; };
  auto bar_empty = [&](int s) { return sbase + OFF_BAR + 8u * (STAGES + s); };
  const uint32_t bar_acc = sbase + OFF_BAR + 8u * (2 * STAGES);
  unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(smem + OFF_MASK);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_TMEM + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_acc, 1);
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < 2 * MAX_E; i += THREADS) s_mask[i] = 0ull;
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(256)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int KT = p.H / KS;
  const int t0 = blockIdx.x * TOK;

  if (warp == 0) {
    // ================= producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      for (int kt = 0; kt < KT; ++kt) {
        if (!wait_bar(bar_empty(stage), phase ^ 1, p.wait_limit, p.status, s_abort)) break;
        const uint32_t sA = sbase + stage * STAGE_MAX;
        mbar_arrive_expect_tx(bar_full(stage), (uint32_t)stage_bytes);
        tma_load_2d(sA, &tmX, kt * KS, t0, bar_full(stage));
        tma_load_2d(sA + A_BYTES, &tmG, kt * KS, 0, bar_full(stage));
        armed |= 1u << stage;
        if (phase) armed_parity |= 1u << stage; else armed_parity &= ~(1u << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      // drain: every copy this thread issued has landed before the CTA exits
      // (returns at once for copies the MMA thread already waited for)
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) {
          volatile int no_abort = 0;
          wait_bar(bar_full(s), (armed_parity >> s) & 1u, 1ll << 32, nullptr, &no_abort);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(TOK, NE);
      int stage = 0;
      uint32_t phase = 0;
      bool issued = false;
      for (int kt = 0; kt < KT; ++kt) {
        if (!wait_bar(bar_full(stage), phase, p.wait_limit, p.status, s_abort)) break;
        tc_fence_after();
        const uint32_t sA = sbase + stage * STAGE_MAX;
        const uint64_t adesc = gemm::make_sdesc(sA, 16, 1024, 2);
        const uint64_t bdesc = gemm::make_sdesc(sA + A_BYTES, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < KS / 16; ++kk)
          mma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) != 0 ? 1u : 0u);
        issued = true;
        tc_commit(bar_empty(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      // the accumulator is complete (or, after an abort, every issued MMA is);
      // this thread also waits, so no MMA is in flight at the teardown
      if (issued) {
        tc_commit(bar_acc);
        volatile int no_abort = 0;
        wait_bar(bar_acc, 0, 1ll << 32, nullptr, &no_abort);
      } else {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar_acc) : "memory");
      }
    }
    __syncwarp();
  } else {
    // ================= epilogue warps: the accumulator goes to shared memory
    // (over the stages, idle once every MMA is done), then each warp takes
    // tokens ew, ew + EPI, ... with the routing kernel's warp top-k (one warp
    // per token is latency-bound: the token count per warp sets the time)
    const int q = warp & 3;        // TMEM lane quarter
    const int r = q * 32 + lane;   // token row this thread moves out of TMEM
    const int ew = warp - 2;       // 0..EPI-1
    const int cg = ew >> 2;        // column group: 32-column chunks cg, cg + EPI/4, ...
    const bool got = wait_bar(bar_acc, 0, p.wait_limit, p.status, s_abort);
    const bool ok = __all_sync(0xffffffffu, got) && !*s_abort;
    tc_fence_after();
    const int LD = E | 1;  // odd row stride: the row-per-lane writes hit 32 banks
    float* s_log = reinterpret_cast<float*>(smem);                  // [TOK][LD]
    int* s_ids = reinterpret_cast<int*>(smem + OFF_IDS);            // [TOK][32]
    if (ok) {
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
      for (int c = 32 * cg; c < E; c += 32 * (EPI / 4)) {
        uint32_t v[32];
        gemm::tmem_ld_32(t_row + c, v);
        gemm::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)  // columns at and past E are not experts
          if (c + i < E) s_log[r * LD + c + i] = __uint_as_float(v[i]);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI) : "memory");
    const int k = p.k;
    if (ok) {
      // NT tokens per call: tl = ew + EPI * (g * NT + n)
      constexpr int NT = EPL <= 4 ? TOK / EPI / 2 : TOK / EPI / 4;  // registers
#pragma unroll
      for (int g = 0; g < TOK / EPI / NT; ++g) {
        const float* rows[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int tl = ew + EPI * (g * NT + n);
          rows[n] = t0 + tl < p.T ? s_log + tl * LD : nullptr;
          if (rows[n] && p.logits)
            for (int e = lane; e < E; e += 32) p.logits[(int64_t)(t0 + tl) * E + e] = rows[n][e];
        }
        int ids[NT];
        float vals[NT], ws[NT];
        warp_topk_softmax<EPL, NT, KC>(rows, E, k, p.renormalize != 0, lane, ids, vals, ws);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int tl = ew + EPI * (g * NT + n);
          if (rows[n] && lane < k) {
            const int64_t f = (int64_t)(t0 + tl) * k + lane;
            p.topk_ids[f] = ids[n];
            p.topk_w[f] = ws[n];
            if (p.local_rank) {
              atomicOr(&s_mask[(tl >> 6) * MAX_E + ids[n]], 1ull << (tl & 63));
              s_ids[tl * 32 + lane] = ids[n];
            }
          }
        }
      }
    }
    // ranks inside each 64-token routing block and its expert histogram
    asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI) : "memory");
    if (ok && p.local_rank) {
      for (int tl = ew; tl < TOK; tl += EPI) {
        const int t = t0 + tl;
        if (t >= p.T) break;
        if (lane < k)
          p.local_rank[(int64_t)t * k + lane] =
              __popcll(s_mask[(tl >> 6) * MAX_E + s_ids[tl * 32 + lane]] &
                       ((1ull << (tl & 63)) - 1ull));
      }
      for (int i = threadIdx.x - 64; i < 2 * E; i += 32 * EPI) {
        const int half = i / E, e = i - half * E;
        const int b = 2 * blockIdx.x + half;
        if (b < p.n_blocks)
          p.block_hist[(int64_t)e * p.n_blocks + b] = __popcll(s_mask[half * MAX_E + e]);
      }
    }
  }

  // ---- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256)
                 : "memory");
  }
}

// bf16 [outer, inner] with a 64-element (128-byte) swizzled box.
static bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                          uint32_t box_outer) {
  auto fn = gemm::encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)KS, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace router

template <int EPL, int KC = 0>
static cudaError_t launch_router_epl(const CUtensorMap& tmX, const CUtensorMap& tmG,
                                     const router::Params& p, int grid, cudaStream_t stream) {
  using namespace router;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static uint64_t configured[64] = {0};  // context id the attribute was set in
  const uint64_t ctx = context_id();
  if (ctx == 0 || configured[dev] != ctx) {
    const cudaError_t err = cudaFuncSetAttribute(router_gate_topk_kernel<EPL, KC>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, ALLOC);
    if (err != cudaSuccess) return err;
    configured[dev] = context_id();
  }
  router_gate_topk_kernel<EPL, KC><<<grid, THREADS, ALLOC, stream>>>(tmX, tmG, p);
  return cudaGetLastError();
}

cudaError_t launch_router_gate_topk(const uint16_t* x, const uint16_t* gate, int T, int H, int E,
                                    int k, bool renormalize, float* logits, int32_t* topk_ids,
                                    float* topk_w, int32_t* local_rank, int32_t* block_hist,
                                    cudaStream_t stream) {
  using namespace router;
  if (T == 0) return cudaSuccess;
  if (H % KS != 0 || E < 1 || E > MAX_E || k < 1 || k > 32 || k > E) return cudaErrorInvalidValue;
  CUtensorMap tmX, tmG;
  if (!make_map_bf16(&tmX, x, (uint64_t)H, (uint64_t)T, TOK)) return cudaErrorInvalidValue;
  // the box covers the MMA's N rows; rows past E read the zero fill
  if (!make_map_bf16(&tmG, gate, (uint64_t)H, (uint64_t)E, (uint32_t)((E + 15) & ~15)))
    return cudaErrorInvalidValue;
  Params p;
  p.T = T;
  p.H = H;
  p.E = E;
  p.k = k;
  p.renormalize = renormalize ? 1 : 0;
  p.n_blocks = (int)ceil_div(T, kRouteTokensPerBlock);
  p.logits = logits;
  p.topk_ids = topk_ids;
  p.topk_w = topk_w;
  p.local_rank = local_rank;
  p.block_hist = block_hist;
  p.status = device_status_ptr();
  p.wait_limit = wait_limit_cycles();
  const int grid = (int)ceil_div(T, TOK);
  const int epl = (E + 31) / 32;
  if (epl <= 1) return launch_router_epl<1>(tmX, tmG, p, grid, stream);
  if (epl <= 2) return launch_router_epl<2>(tmX, tmG, p, grid, stream);
  if (epl <= 4 && k == 8) return launch_router_epl<4, 8>(tmX, tmG, p, grid, stream);  // top-8
  if (epl <= 4) return launch_router_epl<4>(tmX, tmG, p, grid, stream);
  return launch_router_epl<8>(tmX, tmG, p, grid, stream);
}

// ---------------------------------------------------------------- dequant

// e4m3 code -> fp32 from its bit fields: sign | 4 exponent bits (bias 7) |
// 3 mantissa bits, exponent 0 subnormal (m * 2^-9).  The NaN codes are outside
// the contract.
__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
  return __uint_as_float(__float_as_uint(mag) | ((c & 0x80u) << 24));
}

// One thread per 32-element block: 32 e4m3 codes x 2^(s - 127) -> bf16.
__global__ void __launch_bounds__(256) mx_dequantize_bf16_kernel(const uint8_t* __restrict__ q,
                                                                 const uint8_t* __restrict__ s,
                                                                 int64_t n_blocks,
                                                                 uint16_t* __restrict__ out) {
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks;
       b += (int64_t)gridDim.x * blockDim.x) {
    // 2^(s - 127) as an fp32 (s = 0 gives 2^-127, a subnormal; exact)
    const int e = (int)s[b] - 127;
    const float scale = ldexpf(1.f, e);
    const uint4 c0 = ld_nc_v4(q + b * 32), c1 = ld_nc_v4(q + b * 32 + 16);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t wi = w[i];
      o[2 * i] = cvt_bf16x2(e4m3_to_float(wi & 0xFFu) * scale, e4m3_to_float((wi >> 8) & 0xFFu) * scale);
      o[2 * i + 1] =
          cvt_bf16x2(e4m3_to_float((wi >> 16) & 0xFFu) * scale, e4m3_to_float(wi >> 24) * scale);
    }
    uint16_t* dst = out + b * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      st_v4(dst + 8 * i, make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]));
  }
}

cudaError_t launch_mx_dequantize_bf16(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K,
                                      uint16_t* out, cudaStream_t stream) {
  const int64_t n = rows * (K / 32);
  if (n == 0) return cudaSuccess;
  int64_t blocks = ceil_div(n, 256);
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  mx_dequantize_bf16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(q, s, n, out);
  return cudaGetLastError();
}

}  // namespace mxmoe
