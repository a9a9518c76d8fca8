// C ABI of the MXFP8 MoE library: argument validation, the device status
// word, workspace carving and the layer orchestration (moe_forward_mxfp8).
// The declarations and their contracts are in include/mxmoe.h.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "internal.h"
#include "mxmoe.h"

namespace mxmoe {

// Library status word (one per device the library is loaded on).  Kernels get
// its device address as a parameter; they only ever write a non-zero error.
__device__ int g_device_status = 0;

static std::atomic<long long> g_wait_limit{0};
// grouped GEMM kernel choice: 0 = 1-SM, 1 = 2-SM, 2 (default) = 2-SM for the
// bf16-output GEMM when experts average at least 4 m-tiles, and for the SwiGLU
// GEMM when they average at least 8.  A CTA pair computes two m-tiles of one
// expert, so an expert with an odd m-tile count pays a padded tile; with few
// m-tiles per expert that outweighs the pair's third less L2 traffic
// (measured on GB300: gmm2 gains on the 16K-token Qwen3-30B-A3B and 8K-token
// Qwen3-235B-A22B prefills and loses at decode; gmm1 gains 1-3% at 16K
// tokens, plain or skewed, is even on the 235B prefill and loses 12% at 4K
// skewed tokens).
static std::atomic<int> g_use_2sm{2};
// small batches: both grouped GEMMs of an MXFP8 layer in one kernel (1, the
// default) or one kernel each (0); both give the same bytes
static std::atomic<int> g_use_chain{1};

bool use_two_sm_gemm(bool swiglu, int64_t M, int E) {
  const int m = g_use_2sm.load();
  return m == 1 || (m == 2 && M >= (swiglu ? 1024 : 512) * (int64_t)E);
}
constexpr long long kDefaultWaitLimit = 1ll << 32;  // ~2 s at 2 GHz

long long wait_limit_cycles() {
  const long long v = g_wait_limit.load();
  return v > 0 ? v : kDefaultWaitLimit;
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices] = {0};
int* g_status_ptr[kMaxDevices] = {nullptr};
uint64_t g_status_ctx[kMaxDevices] = {0};  // context id the cached address belongs to
}  // namespace

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

uint64_t context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return (uint64_t)id;
}

int* device_status_ptr() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  const uint64_t ctx = context_id();
  if (!g_status_ptr[dev] || ctx == 0 || ctx != g_status_ctx[dev]) {
    // (the lookup makes the device's primary context current, so the id is
    // taken again afterwards)
    void* p = nullptr;
    g_status_ptr[dev] = cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess ? (int*)p : nullptr;
    g_status_ctx[dev] = context_id();
  }
  return g_status_ptr[dev];
}

static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
static inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace mxmoe

using namespace mxmoe;

#define MXMOE_CHECK_PTR(p)                 \
  do {                                     \
    if ((p) == nullptr) return MXMOE_ERR_NULL; \
    if (!aligned16(p)) return MXMOE_ERR_ALIGN; \
  } while (0)

static mxmoe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MXMOE_OK : MXMOE_ERR_CUDA; }

extern "C" {

const char* mxmoe_status_string(mxmoe_status s) {
  switch (s) {
    case MXMOE_OK: return "MXMOE_OK";
    case MXMOE_ERR_NULL: return "MXMOE_ERR_NULL: a required pointer is NULL";
    case MXMOE_ERR_ALIGN: return "MXMOE_ERR_ALIGN: a pointer is misaligned (16 bytes; 32 for GEMM outputs)";
    case MXMOE_ERR_SHAPE: return "MXMOE_ERR_SHAPE: a size is out of range or inconsistent";
    case MXMOE_ERR_UNSUPPORTED: return "MXMOE_ERR_UNSUPPORTED: not supported by this build";
    case MXMOE_ERR_WORKSPACE: return "MXMOE_ERR_WORKSPACE: workspace missing or too small";
    case MXMOE_ERR_CUDA: return "MXMOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MXMOE_ERR_DEVICE_TIMEOUT: return "MXMOE_ERR_DEVICE_TIMEOUT: a device-side wait timed out";
    case MXMOE_ERR_DEVICE_CHECK: return "MXMOE_ERR_DEVICE_CHECK: a device-side check failed";
  }
  return "MXMOE_ERR_UNKNOWN";
}

const char* mxmoe_version(void) { return "mxmoe 0.1.0 (sm_103a)"; }

void mxmoe_set_wait_limit_cycles(long long cycles) { g_wait_limit.store(cycles > 0 ? cycles : 0); }

void mxmoe_set_gemm_2sm(int mode) { g_use_2sm.store(mode < 0 || mode > 2 ? 2 : mode); }

void mxmoe_set_gemm_chain(int enable) { g_use_chain.store(enable ? 1 : 0); }

mxmoe_status mxmoe_get_device_status(int32_t* status_out, int clear) {
  if (!status_out) return MXMOE_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return MXMOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return MXMOE_ERR_CUDA;
  *status_out = v;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return MXMOE_ERR_CUDA;
  }
  return MXMOE_OK;
}

mxmoe_status mx_quantize_3d(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint8_t* q,
                            uint8_t* scale, void* stream) {
  if (E < 0 || N < 0 || K <= 0 || K % 16 != 0) return MXMOE_ERR_SHAPE;
  if (E == 0 || N == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(w);
  MXMOE_CHECK_PTR(q);
  if (!scale) return MXMOE_ERR_NULL;
  return from_cuda(launch_mx_quantize(w, E * N, K, q, scale, (cudaStream_t)stream));
}

size_t moe_route_quant_mxfp8_workspace_size(int T, int E) {
  if (T < 0 || E <= 0) return 0;
  return route_workspace_bytes(T, E);
}

static mxmoe_status check_route(const uint16_t* x, const float* logits, int T, int H, int E, int k,
                                int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                                int32_t* src_to_sorted, int64_t* counts, int64_t* offsets,
                                void* ws, size_t ws_bytes) {
  if (T < 0 || H <= 0 || H % 32 != 0 || E <= 0 || E > 1024 || k < 1 || k > 32 || k > E)
    return MXMOE_ERR_SHAPE;
  if ((int64_t)T * k >= (1ll << 31)) return MXMOE_ERR_SHAPE;
  MXMOE_CHECK_PTR(counts);
  MXMOE_CHECK_PTR(offsets);
  if (T == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(x);
  MXMOE_CHECK_PTR(logits);
  MXMOE_CHECK_PTR(topk_ids);
  MXMOE_CHECK_PTR(topk_w);
  MXMOE_CHECK_PTR(sorted_to_src);
  MXMOE_CHECK_PTR(src_to_sorted);
  if (!ws) return MXMOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MXMOE_ERR_ALIGN;
  if (ws_bytes < route_workspace_bytes(T, E)) return MXMOE_ERR_WORKSPACE;
  return MXMOE_OK;
}

mxmoe_status moe_route_quant_mxfp8(const uint16_t* x, const float* logits, int T, int H, int E,
                                   int k, int renormalize, uint8_t* xq, uint8_t* xs,
                                   int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
                                   int32_t* src_to_sorted, int64_t* expert_counts,
                                   int64_t* expert_offsets, void* ws, size_t ws_bytes,
                                   void* stream) {
  mxmoe_status st = check_route(x, logits, T, H, E, k, topk_ids, topk_w, sorted_to_src,
                                src_to_sorted, expert_counts, expert_offsets, ws, ws_bytes);
  if (st != MXMOE_OK) return st;
  if (T > 0) {
    MXMOE_CHECK_PTR(xq);
    if (!xs) return MXMOE_ERR_NULL;
  }
  return from_cuda(launch_route(x, logits, T, H, E, k, renormalize != 0, true, xq, xs, nullptr,
                                topk_ids, topk_w, sorted_to_src, src_to_sorted, expert_counts,
                                expert_offsets, (int32_t*)ws, (cudaStream_t)stream));
}

mxmoe_status moe_route_permute_bf16(const uint16_t* x, const float* logits, int T, int H, int E,
                                    int k, int renormalize, uint16_t* xp, int32_t* topk_ids,
                                    float* topk_w, int32_t* sorted_to_src, int32_t* src_to_sorted,
                                    int64_t* expert_counts, int64_t* expert_offsets, void* ws,
                                    size_t ws_bytes, void* stream) {
  mxmoe_status st = check_route(x, logits, T, H, E, k, topk_ids, topk_w, sorted_to_src,
                                src_to_sorted, expert_counts, expert_offsets, ws, ws_bytes);
  if (st != MXMOE_OK) return st;
  if (T > 0) MXMOE_CHECK_PTR(xp);
  return from_cuda(launch_route(x, logits, T, H, E, k, renormalize != 0, false, nullptr, nullptr,
                                xp, topk_ids, topk_w, sorted_to_src, src_to_sorted, expert_counts,
                                expert_offsets, (int32_t*)ws, (cudaStream_t)stream));
}

static mxmoe_status check_gemm(const uint8_t* a, const uint8_t* sa, const uint8_t* w,
                               const uint8_t* sw, const int64_t* offsets, int64_t M, int E, int K,
                               int N, const void* out) {
  if (M < 0 || M >= (1ll << 31) || E < 1 || K <= 0 || N <= 0) return MXMOE_ERR_SHAPE;
  if (E > 256) return MXMOE_ERR_UNSUPPORTED;
  if (K % 128 != 0 || N % 128 != 0) return MXMOE_ERR_UNSUPPORTED;
  MXMOE_CHECK_PTR(offsets);
  if (M == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(a);
  MXMOE_CHECK_PTR(w);
  MXMOE_CHECK_PTR(out);
  if ((uintptr_t)out & 31u) return MXMOE_ERR_ALIGN;  // 32-byte sector stores
  if (!sa || !sw) return MXMOE_ERR_NULL;
  if (((uintptr_t)sa & 3u) || ((uintptr_t)sw & 3u)) return MXMOE_ERR_ALIGN;
  return MXMOE_OK;
}

mxmoe_status grouped_gemm_swiglu_quant_mxfp8(const uint8_t* xq, const uint8_t* xs,
                                             const uint8_t* w13q, const uint8_t* w13s,
                                             const int64_t* expert_offsets, int64_t M, int E,
                                             int H, int I, uint8_t* aq, uint8_t* as,
                                             void* stream) {
  mxmoe_status st = check_gemm(xq, xs, w13q, w13s, expert_offsets, M, E, H, I, aq);
  if (st != MXMOE_OK) return st;
  if (M > 0 && !as) return MXMOE_ERR_NULL;
  if ((int64_t)E * 2 * I >= (1ll << 31)) return MXMOE_ERR_SHAPE;
  return from_cuda(launch_gemm_swiglu_quant(xq, xs, w13q, w13s, expert_offsets, M, E, H, I, aq, as,
                                            (cudaStream_t)stream));
}

mxmoe_status grouped_gemm_mxfp8(const uint8_t* aq, const uint8_t* as, const uint8_t* w2q,
                                const uint8_t* w2s, const int64_t* expert_offsets, int64_t M,
                                int E, int I, int H, uint16_t* y, void* stream) {
  mxmoe_status st = check_gemm(aq, as, w2q, w2s, expert_offsets, M, E, I, H, y);
  if (st != MXMOE_OK) return st;
  if ((int64_t)E * H >= (1ll << 31)) return MXMOE_ERR_SHAPE;
  return from_cuda(
      launch_gemm_bf16(aq, as, w2q, w2s, expert_offsets, M, E, I, H, y, (cudaStream_t)stream));
}

mxmoe_status moe_finalize_routing(const uint16_t* y, const float* topk_w,
                                  const int32_t* src_to_sorted, int T, int k, int H,
                                  uint16_t* out, void* stream) {
  if (T < 0 || k < 1 || k > 32 || H <= 0 || H % 8 != 0) return MXMOE_ERR_SHAPE;
  if (T == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(y);
  MXMOE_CHECK_PTR(topk_w);
  MXMOE_CHECK_PTR(src_to_sorted);
  MXMOE_CHECK_PTR(out);
  return from_cuda(launch_finalize(y, topk_w, src_to_sorted, T, k, H, out, (cudaStream_t)stream));
}

// Workspace of the whole layer, in this order (each 256-byte aligned):
// xq [M,H] | xs tiled | topk_ids [T,k] | topk_w [T,k] | sorted_to_src [M] |
// src_to_sorted [M] | counts [E] | offsets [E+1] | tile bases [E+1] |
// route histograms | aq [M,I] | as tiled | y [M,H] bf16 | w13s tiled | w2s tiled.
// Tiled activation scales hold at most ceil(M/128) + E row blocks.
struct FwdLayout {
  size_t xq, xs, ids, w, s2s, src2s, counts, offs, tbase, hist, aq, as, y, w13s, w2s, done, total;
};

static FwdLayout fwd_layout(int T, int H, int E, int k, int I) {
  FwdLayout L;
  const size_t M = (size_t)T * k;
  const size_t blocks = (M + 127) / 128 + (size_t)E;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += align256(bytes); return at; };
  L.xq = take(M * H);
  L.xs = take(blocks * 128 * (H / 32));
  L.ids = take(M * 4);
  L.w = take(M * 4);
  L.s2s = take(M * 4);
  L.src2s = take(M * 4);
  L.counts = take((size_t)E * 8);
  L.offs = take((size_t)(E + 1) * 8);
  L.tbase = take((size_t)(E + 1) * 4);
  L.hist = take(route_workspace_bytes(T, E));
  L.aq = take(M * I);
  L.as = take(blocks * 128 * (I / 32));
  L.y = take(M * H * 2);
  L.w13s = take((size_t)E * 2 * I * (H / 32));
  L.w2s = take((size_t)E * H * (I / 32));
  L.done = take((size_t)E * 4);
  L.total = o;
  return L;
}

size_t moe_forward_mxfp8_workspace_size(int T, int H, int E, int k, int I) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || I <= 0) return 0;
  return fwd_layout(T, H, E, k, I).total;
}

mxmoe_status mx_scales_to_mma_layout(const uint8_t* scale, int64_t E, int64_t N, int64_t K,
                                     uint8_t* out, void* stream) {
  if (E < 0 || N < 0 || K <= 0 || K % 16 != 0) return MXMOE_ERR_SHAPE;
  if (E > 1 && N % 128 != 0) return MXMOE_ERR_UNSUPPORTED;  // experts start whole row blocks
  if (E == 0 || N == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(scale);
  MXMOE_CHECK_PTR(out);
  return from_cuda(launch_scales_to_tiled(scale, E * N, K, out, (cudaStream_t)stream));
}

// Opt-in per-kernel timing of the layer call: events recorded on the call's
// stream between its kernels (one set per device, reused by every call).
namespace {
constexpr int kProfEvents = 6;
std::atomic<int> g_prof_enabled{0};
cudaEvent_t g_prof_ev[kMaxDevices][kProfEvents] = {};
bool g_prof_valid[kMaxDevices] = {false};
int g_prof_mode[kMaxDevices] = {0};  // mode of the last profiled call

// Mode 1 records an event at every kernel boundary; mode 2 only around the
// dominant GEMM (events 2 and 3), so the other boundaries keep their
// programmatic dependent launches (an event between two kernels makes the
// second wait for the first to finish).
struct LayerProfiler {
  int dev = -1;
  int mode = 0;
  cudaStream_t s;
  explicit LayerProfiler(cudaStream_t st) : s(st) {
    const int m = g_prof_enabled.load();
    if (!m) return;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < kProfEvents; ++i)
      if (!g_prof_ev[dev][i] && cudaEventCreate(&g_prof_ev[dev][i]) != cudaSuccess) return;
    g_prof_valid[dev] = false;
    mode = m;
  }
  void mark(int i) {
    if (mode == 1 || (mode == 2 && (i == 2 || i == 3))) cudaEventRecord(g_prof_ev[dev][i], s);
  }
  void done() {
    if (mode) {
      g_prof_valid[dev] = true;
      g_prof_mode[dev] = mode;
    }
  }
};
}  // namespace

mxmoe_status mxmoe_layer_profile_enable(int enable) {
  if (enable < 0 || enable > 2) return MXMOE_ERR_SHAPE;
  g_prof_enabled.store(enable);
  return MXMOE_OK;
}

mxmoe_status mxmoe_layer_profile_read(float* ms, int n) {
  if (!ms || n < 1) return MXMOE_ERR_NULL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MXMOE_ERR_CUDA;
  if (!g_prof_valid[dev]) return MXMOE_ERR_UNSUPPORTED;
  const bool full = g_prof_mode[dev] == 1;
  const int last = full ? kProfEvents - 1 : 3;
  if (cudaEventSynchronize(g_prof_ev[dev][last]) != cudaSuccess) return MXMOE_ERR_CUDA;
  for (int i = 0; i < n && i < kProfEvents - 1; ++i) {
    float t = 0.f;
    if ((full || i == 2) &&
        cudaEventElapsedTime(&t, g_prof_ev[dev][i], g_prof_ev[dev][i + 1]) != cudaSuccess)
      return MXMOE_ERR_CUDA;
    ms[i] = t;
  }
  return MXMOE_OK;
}

// fmt: 0 = W8A8; 1 = W4A8 (w13q / w2q packed MXFP4); 2 = W4A4 (the expert
// inputs of both grouped GEMMs are MXFP4 as well).  1 and 2 require mma_scales.
static mxmoe_status forward_impl(const uint16_t* x, const float* logits, const uint8_t* w13q,
                                 const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                                 bool mma_scales, int T, int H, int E, int k, int I,
                                 int renormalize, uint16_t* out, void* ws, size_t ws_bytes,
                                 void* stream, int fmt = 0, const uint16_t* gate = nullptr) {
  const bool fp4_weights = fmt != 0;
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > 32 || k > E || I <= 0) return MXMOE_ERR_SHAPE;
  if (E > 256 || H % 128 != 0 || I % 128 != 0) return MXMOE_ERR_UNSUPPORTED;
  if ((int64_t)T * k >= (1ll << 31)) return MXMOE_ERR_SHAPE;
  if (T == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(x);
  if (gate) MXMOE_CHECK_PTR(gate); else MXMOE_CHECK_PTR(logits);
  MXMOE_CHECK_PTR(w13q);
  MXMOE_CHECK_PTR(w2q);
  MXMOE_CHECK_PTR(out);
  if (!w13s || !w2s) return MXMOE_ERR_NULL;
  if (mma_scales && (!aligned16(w13s) || !aligned16(w2s))) return MXMOE_ERR_ALIGN;
  if (fp4_weights && (!mma_scales || ((uintptr_t)w13q & 31u) || ((uintptr_t)w2q & 31u)))
    return mma_scales ? MXMOE_ERR_ALIGN : MXMOE_ERR_UNSUPPORTED;
  if (!mma_scales && (((uintptr_t)w13s & 3u) || ((uintptr_t)w2s & 3u))) return MXMOE_ERR_ALIGN;
  if (!ws) return MXMOE_ERR_WORKSPACE;
  if ((uintptr_t)ws & 255u) return MXMOE_ERR_ALIGN;
  const FwdLayout L = fwd_layout(T, H, E, k, I);
  if (ws_bytes < L.total) return MXMOE_ERR_WORKSPACE;
  uint8_t* b = (uint8_t*)ws;
  const int64_t M = (int64_t)T * k;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* xq = b + L.xq;
  uint8_t* xs = b + L.xs;
  int32_t* ids = (int32_t*)(b + L.ids);
  float* w = (float*)(b + L.w);
  int32_t* s2s = (int32_t*)(b + L.s2s);
  int32_t* src2s = (int32_t*)(b + L.src2s);
  int64_t* counts = (int64_t*)(b + L.counts);
  int64_t* offs = (int64_t*)(b + L.offs);
  int32_t* tbase = (int32_t*)(b + L.tbase);
  uint8_t* aq = b + L.aq;
  uint8_t* as = b + L.as;
  uint16_t* y = (uint16_t*)(b + L.y);
  const uint8_t* w13s_t = w13s;
  const uint8_t* w2s_t = w2s;
  cudaError_t e;
  LayerProfiler prof(s);
  prof.mark(0);
  if (!mma_scales) {
    e = launch_scales_to_tiled(w13s, (int64_t)E * 2 * I, H, b + L.w13s, s);
    if (e != cudaSuccess) return MXMOE_ERR_CUDA;
    e = launch_scales_to_tiled(w2s, (int64_t)E * H, I, b + L.w2s, s);
    if (e != cudaSuccess) return MXMOE_ERR_CUDA;
    w13s_t = b + L.w13s;
    w2s_t = b + L.w2s;
  }
  prof.mark(1);
  if (gate) {
    // the fused router leaves ids, weights, in-block ranks and histograms
    e = launch_router_gate_topk(x, gate, T, H, E, k, renormalize != 0, nullptr, ids, w, src2s,
                                (int32_t*)(b + L.hist), s);
    if (e != cudaSuccess) return MXMOE_ERR_CUDA;
  }
  // small MXFP8 batches: both grouped GEMMs in one kernel, whose per-expert
  // completion counters the routing kernel zeroes
  const bool chain = fmt == 0 && !gate && g_use_chain.load() != 0 &&
                     T <= kRouteTokensPerBlock && E <= 256 && gemm_chain_supported(T, H, I);
  int* done = chain ? (int*)(b + L.done) : nullptr;
  e = launch_route(x, logits, T, H, E, k, renormalize != 0, fmt == 2 ? 2 : 1, xq, xs, nullptr, ids,
                   w, s2s, src2s, counts, offs, (int32_t*)(b + L.hist), s, tbase, gate != nullptr,
                   done);
  if (e != cudaSuccess) return MXMOE_ERR_CUDA;
  prof.mark(2);
  // an expert's rows are at most T (the k experts of a token are distinct)
  if (chain) {
    // one kernel: its time is reported as gmm1's, gmm2's as zero
    e = launch_gemm_chain(xq, xs, w13q, w13s_t, w2q, w2s_t, offs, M, E, H, I, aq, as, y, done, s,
                          T);
    if (e != cudaSuccess) return MXMOE_ERR_CUDA;
    prof.mark(3);
    prof.mark(4);
  } else {
    e = launch_gemm_swiglu_quant(xq, xs, w13q, w13s_t, offs, M, E, H, I, aq, as, s, true, fmt, T);
    if (e != cudaSuccess) return MXMOE_ERR_CUDA;
    prof.mark(3);
    e = launch_gemm_bf16(aq, as, w2q, w2s_t, offs, M, E, I, H, y, s, true, fmt, 1, nullptr, T);
    if (e != cudaSuccess) return MXMOE_ERR_CUDA;
    prof.mark(4);
  }
  e = launch_finalize(y, w, src2s, T, k, H, out, s);
  if (e != cudaSuccess) return MXMOE_ERR_CUDA;
  prof.mark(5);
  prof.done();
  return MXMOE_OK;
}

mxmoe_status moe_forward_mxfp8(const uint16_t* x, const float* logits, const uint8_t* w13q,
                               const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                               int T, int H, int E, int k, int I, int renormalize,
                               uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(x, logits, w13q, w13s, w2q, w2s, false, T, H, E, k, I, renormalize, out, ws,
                      ws_bytes, stream);
}

mxmoe_status moe_forward_mxfp8_mma_scales(const uint16_t* x, const float* logits,
                                          const uint8_t* w13q, const uint8_t* w13s_mma,
                                          const uint8_t* w2q, const uint8_t* w2s_mma, int T,
                                          int H, int E, int k, int I, int renormalize,
                                          uint16_t* out, void* ws, size_t ws_bytes,
                                          void* stream) {
  return forward_impl(x, logits, w13q, w13s_mma, w2q, w2s_mma, true, T, H, E, k, I, renormalize,
                      out, ws, ws_bytes, stream);
}

mxmoe_status moe_forward_w4a8_mma_scales(const uint16_t* x, const float* logits,
                                         const uint8_t* w13p, const uint8_t* w13s_mma,
                                         const uint8_t* w2p, const uint8_t* w2s_mma, int T, int H,
                                         int E, int k, int I, int renormalize, uint16_t* out,
                                         void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(x, logits, w13p, w13s_mma, w2p, w2s_mma, true, T, H, E, k, I, renormalize,
                      out, ws, ws_bytes, stream, 1);
}

mxmoe_status moe_forward_w4a4_mma_scales(const uint16_t* x, const float* logits,
                                         const uint8_t* w13p, const uint8_t* w13s_mma,
                                         const uint8_t* w2p, const uint8_t* w2s_mma, int T, int H,
                                         int E, int k, int I, int renormalize, uint16_t* out,
                                         void* ws, size_t ws_bytes, void* stream) {
  return forward_impl(x, logits, w13p, w13s_mma, w2p, w2s_mma, true, T, H, E, k, I, renormalize,
                      out, ws, ws_bytes, stream, 2);
}

mxmoe_status moe_forward_mxfp8_gated_mma_scales(const uint16_t* x, const uint16_t* gate,
                                                const uint8_t* w13q, const uint8_t* w13s_mma,
                                                const uint8_t* w2q, const uint8_t* w2s_mma, int T,
                                                int H, int E, int k, int I, int renormalize,
                                                uint16_t* out, void* ws, size_t ws_bytes,
                                                void* stream) {
  return forward_impl(x, nullptr, w13q, w13s_mma, w2q, w2s_mma, true, T, H, E, k, I, renormalize,
                      out, ws, ws_bytes, stream, 0, gate);
}

mxmoe_status moe_router_gate_topk(const uint16_t* x, const uint16_t* gate, int T, int H, int E,
                                  int k, int renormalize, float* logits_out, int32_t* topk_ids,
                                  float* topk_w, void* stream) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E) return MXMOE_ERR_SHAPE;
  if (H % 64 != 0 || E > 256 || k > 32) return MXMOE_ERR_UNSUPPORTED;
  if (T == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(x);
  MXMOE_CHECK_PTR(gate);
  MXMOE_CHECK_PTR(topk_ids);
  MXMOE_CHECK_PTR(topk_w);
  if (logits_out && !aligned16(logits_out)) return MXMOE_ERR_ALIGN;
  return from_cuda(launch_router_gate_topk(x, gate, T, H, E, k, renormalize != 0, logits_out,
                                           topk_ids, topk_w, nullptr, nullptr,
                                           (cudaStream_t)stream));
}

mxmoe_status mx_dequantize_bf16_2d(const uint8_t* q, const uint8_t* scale, int64_t rows,
                                   int64_t K, uint16_t* out, void* stream) {
  if (rows < 0 || K <= 0 || K % 32 != 0) return MXMOE_ERR_SHAPE;
  if (rows == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(q);
  MXMOE_CHECK_PTR(out);
  if (!scale) return MXMOE_ERR_NULL;
  return from_cuda(launch_mx_dequantize_bf16(q, scale, rows, K, out, (cudaStream_t)stream));
}

mxmoe_status mx_quantize_fp4_3d(const uint16_t* w, int64_t E, int64_t N, int64_t K, uint8_t* q,
                                uint8_t* scale, void* stream) {
  if (E < 0 || N < 0 || K <= 0 || K % 32 != 0) return MXMOE_ERR_SHAPE;
  if (E == 0 || N == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(w);
  MXMOE_CHECK_PTR(q);
  if (!scale) return MXMOE_ERR_NULL;
  return from_cuda(launch_mx_quantize_fp4(w, E * N, K, q, scale, (cudaStream_t)stream));
}

// Dense linear workspace, each part 256-byte aligned:
// xq [M, K] | xs tiled (ceil(M/128) + 1 row blocks) | offsets [2] | w scales
// tiled (ceil(N/128) row blocks; the row-major-scale entry point only) |
// split-K partial sums fp32 [ksplit][M][N] (small M only).
struct LinearLayout {
  size_t xq, xs, offs, ws, partial, total;
  int ksplit;
};

static LinearLayout linear_layout(int64_t M, int64_t N, int64_t K, bool w_scales) {
  LinearLayout L;
  const size_t slice_bytes = (size_t)((K + 127) / 128) * 512;  // one row block, one K slice each
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += align256(bytes); return at; };
  L.xq = take((size_t)M * K);
  L.xs = take(((size_t)(M + 127) / 128 + 1) * slice_bytes);
  L.offs = take(2 * sizeof(int64_t));
  L.ws = w_scales ? take((size_t)(N + 127) / 128 * slice_bytes) : 0;
  L.ksplit = M > 0 ? gemm_bf16_ksplit(M, (int)N, (int)K) : 1;
  L.partial = L.ksplit > 1 ? take((size_t)L.ksplit * M * N * sizeof(float)) : 0;
  L.total = o;
  return L;
}

static bool linear_shape_ok(int64_t M, int64_t N, int64_t K) {
  return M >= 0 && M < (1ll << 31) && N > 0 && N < (1ll << 31) && K > 0 && K < (1ll << 31) &&
         N % 16 == 0 && K % 16 == 0;
}

size_t mxfp8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (!linear_shape_ok(M, N, K)) return 0;
  return linear_layout(M, N, K, true).total;
}

// fp4: W4A4 (packed MXFP4 weights [N, K/2], 32-byte aligned; activations
// quantized to MXFP4), K % 128 == 0: every k-slice of the packed GEMM holds
// one or two whole 128-element scale chunks.
static mxmoe_status linear_impl(const uint16_t* x, const uint8_t* wq, const uint8_t* ws,
                                bool ws_tiled, int64_t M, int64_t N, int64_t K, uint16_t* out,
                                void* workspace, size_t ws_bytes, void* stream, bool fp4 = false) {
  if (!linear_shape_ok(M, N, K) || (fp4 && K % 128 != 0)) return MXMOE_ERR_SHAPE;
  if (M == 0) return MXMOE_OK;
  MXMOE_CHECK_PTR(x);
  MXMOE_CHECK_PTR(wq);
  if (fp4 && ((uintptr_t)wq & 31u)) return MXMOE_ERR_ALIGN;
  MXMOE_CHECK_PTR(out);
  if ((uintptr_t)out & 31u) return MXMOE_ERR_ALIGN;  // 32-byte sector stores
  if (!ws) return MXMOE_ERR_NULL;
  if (ws_tiled && !aligned16(ws)) return MXMOE_ERR_ALIGN;  // bulk copies
  const LinearLayout L = linear_layout(M, N, K, !ws_tiled);
  if (!workspace || ws_bytes < L.total) return MXMOE_ERR_WORKSPACE;
  if ((uintptr_t)workspace & 255u) return MXMOE_ERR_ALIGN;
  // the workspace holds L.ksplit partial planes, at least the W4A4 count
  const int ksplit = fp4 ? gemm_bf16_ksplit(M, (int)N, (int)K, true) : L.ksplit;
  if (ksplit > L.ksplit) return MXMOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* base = (uint8_t*)workspace;
  uint8_t* xq = base + L.xq;
  uint8_t* xs = base + L.xs;
  int64_t* offs = (int64_t*)(base + L.offs);
  const uint8_t* wst = ws;
  cudaError_t err;
  LayerProfiler prof(st);
  prof.mark(0);
  if (!ws_tiled) {
    err = launch_scales_to_tiled(ws, N, K, base + L.ws, st);
    if (err != cudaSuccess) return MXMOE_ERR_CUDA;
    wst = base + L.ws;
  }
  prof.mark(1);
  err = launch_mx_quantize_tiled(x, M, K, xq, xs, offs, st, fp4);
  if (err != cudaSuccess) return MXMOE_ERR_CUDA;
  prof.mark(2);
  err = launch_gemm_bf16(xq, xs, wq, wst, offs, M, 1, (int)K, (int)N, out, st, true, fp4 ? 2 : 0,
                         ksplit, ksplit > 1 ? (float*)(base + L.partial) : nullptr);
  if (err != cudaSuccess) return MXMOE_ERR_CUDA;
  for (int i = 3; i < kProfEvents; ++i) prof.mark(i);
  prof.done();
  return MXMOE_OK;
}

mxmoe_status mxfp8_linear(const uint16_t* x, const uint8_t* wq, const uint8_t* ws, int64_t M,
                          int64_t N, int64_t K, uint16_t* out, void* workspace, size_t ws_bytes,
                          void* stream) {
  return linear_impl(x, wq, ws, false, M, N, K, out, workspace, ws_bytes, stream);
}

mxmoe_status mxfp8_linear_mma_scales(const uint16_t* x, const uint8_t* wq, const uint8_t* ws_mma,
                                     int64_t M, int64_t N, int64_t K, uint16_t* out,
                                     void* workspace, size_t ws_bytes, void* stream) {
  return linear_impl(x, wq, ws_mma, true, M, N, K, out, workspace, ws_bytes, stream);
}

mxmoe_status mxfp4_linear(const uint16_t* x, const uint8_t* wp, const uint8_t* ws, int64_t M,
                          int64_t N, int64_t K, uint16_t* out, void* workspace, size_t ws_bytes,
                          void* stream) {
  return linear_impl(x, wp, ws, false, M, N, K, out, workspace, ws_bytes, stream, true);
}

mxmoe_status mxfp4_linear_mma_scales(const uint16_t* x, const uint8_t* wp, const uint8_t* ws_mma,
                                     int64_t M, int64_t N, int64_t K, uint16_t* out,
                                     void* workspace, size_t ws_bytes, void* stream) {
  return linear_impl(x, wp, ws_mma, true, M, N, K, out, workspace, ws_bytes, stream, true);
}

// ---------------------------------------------------------------- host-buffer layer

// Device staging of one chunk slot: x | logits | out | layer workspace.
constexpr int kMaxHostChunks = 1024;

struct HostChunkLayout {
  size_t x, logits, out, ws, ws_bytes, slot;
};

static HostChunkLayout host_chunk_layout(int Tc, int H, int E, int k, int I) {
  HostChunkLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o += align256(bytes); return at; };
  L.x = take((size_t)Tc * H * 2);
  L.logits = take((size_t)Tc * E * 4);
  L.out = take((size_t)Tc * H * 2);
  L.ws_bytes = fwd_layout(Tc, H, E, k, I).total;
  L.ws = take(L.ws_bytes);
  L.slot = o;
  return L;
}

// Chunk plans.  n_chunks > 0: that many near-equal chunks.  n_chunks <= 0:
// the default plan, chosen from measurements on GB300 (16K-token
// Qwen3-30B-A3B layer; host links ~0.2 TB/s each way): every chunk re-reads
// all experts' weights, so chunks should be few and large, while the first
// chunk's copy-in and the last chunk's copy-out are not overlapped with any
// compute, so those two should be small.  Up to 4096 tokens: one chunk;
// beyond: three chunks, the outer two of 3/16 of the tokens each (measured:
// 1.17 ms per call against 1.28 ms for two equal chunks and 1.51 ms for one).
static int host_chunk_plan(int T, int n_chunks, int* sizes) {
  if (T <= 0) { sizes[0] = 0; return 1; }
  if (n_chunks <= 0) {
    if (T <= 4096) { sizes[0] = T; return 1; }
    const int a = std::max(64, (T * 3 / 16) / 64 * 64);
    sizes[0] = a;
    sizes[1] = T - 2 * a;
    sizes[2] = a;
    return 3;
  }
  if (n_chunks > kMaxHostChunks) n_chunks = kMaxHostChunks;
  if (n_chunks > T) n_chunks = T;
  for (int i = 0; i < n_chunks; ++i)
    sizes[i] = (int)((int64_t)T * (i + 1) / n_chunks - (int64_t)T * i / n_chunks);
  return n_chunks;
}

size_t moe_forward_mxfp8_host_workspace_size(int T, int H, int E, int k, int I, int n_chunks) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || I <= 0) return 0;
  int sizes[kMaxHostChunks];
  const int n = host_chunk_plan(T, n_chunks, sizes);
  int Tc = 0;
  for (int i = 0; i < n; ++i) Tc = std::max(Tc, sizes[i]);
  return 2 * host_chunk_layout(Tc, H, E, k, I).slot;
}

namespace {
struct HostPipe {
  cudaStream_t s[3] = {nullptr, nullptr, nullptr};  // h2d, compute, d2h
  cudaEvent_t ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {}, ev_start = {}, ev_done = {};
  bool ok = false;
};
HostPipe g_pipe[kMaxDevices];
}  // namespace

static HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  HostPipe& P = g_pipe[dev];
  if (!P.ok) {
    for (auto& st : P.s)
      if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    cudaEvent_t* evs[] = {&P.ev_in[0], &P.ev_in[1], &P.ev_comp[0], &P.ev_comp[1],
                          &P.ev_out[0], &P.ev_out[1], &P.ev_start, &P.ev_done};
    for (cudaEvent_t* e : evs)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    P.ok = true;
  }
  return &P;
}

// The pipeline over an explicit chunk plan (sizes[0..n), summing to T).
static mxmoe_status host_pipeline(const uint16_t* x_host, const float* logits_host,
                                  const uint8_t* w13q, const uint8_t* w13s_mma,
                                  const uint8_t* w2q, const uint8_t* w2s_mma, int T, int H, int E,
                                  int k, int I, int renormalize, uint16_t* out_host,
                                  const int* sizes, int n, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > 32 || k > E || I <= 0) return MXMOE_ERR_SHAPE;
  if (E > 256 || H % 128 != 0 || I % 128 != 0) return MXMOE_ERR_UNSUPPORTED;
  if ((int64_t)T * k >= (1ll << 31)) return MXMOE_ERR_SHAPE;
  if (T == 0) return MXMOE_OK;
  if (!x_host || !logits_host || !out_host) return MXMOE_ERR_NULL;
  MXMOE_CHECK_PTR(w13q);
  MXMOE_CHECK_PTR(w2q);
  MXMOE_CHECK_PTR(w13s_mma);
  MXMOE_CHECK_PTR(w2s_mma);
  if (!ws) return MXMOE_ERR_WORKSPACE;
  if ((uintptr_t)ws & 255u) return MXMOE_ERR_ALIGN;
  int64_t sum = 0;
  int Tc = 0;
  for (int i = 0; i < n; ++i) {
    if (sizes[i] <= 0) return MXMOE_ERR_SHAPE;
    sum += sizes[i];
    Tc = std::max(Tc, sizes[i]);
  }
  if (n <= 0 || sum != T) return MXMOE_ERR_SHAPE;
  const HostChunkLayout CL = host_chunk_layout(Tc, H, E, k, I);
  if (ws_bytes < 2 * CL.slot) return MXMOE_ERR_WORKSPACE;
  HostPipe* P = host_pipe();
  if (!P) return MXMOE_ERR_CUDA;
  cudaStream_t user = (cudaStream_t)stream;
  auto ck = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ck(cudaEventRecord(P->ev_start, user))) return MXMOE_ERR_CUDA;
  for (auto st : P->s)
    if (!ck(cudaStreamWaitEvent(st, P->ev_start, 0))) return MXMOE_ERR_CUDA;
  uint8_t* base = (uint8_t*)ws;
  int t0 = 0;
  for (int c = 0; c < n; t0 += sizes[c], ++c) {
    const int tc = sizes[c];
    const int slot = c & 1;
    uint8_t* sb = base + (size_t)slot * CL.slot;
    uint16_t* xd = (uint16_t*)(sb + CL.x);
    float* ld = (float*)(sb + CL.logits);
    uint16_t* od = (uint16_t*)(sb + CL.out);
    // h2d: the slot's inputs are free once chunk c-2's compute is done
    if (c >= 2 && !ck(cudaStreamWaitEvent(P->s[0], P->ev_comp[slot], 0))) return MXMOE_ERR_CUDA;
    if (!ck(cudaMemcpyAsync(xd, x_host + (size_t)t0 * H, (size_t)tc * H * 2,
                            cudaMemcpyHostToDevice, P->s[0])) ||
        !ck(cudaMemcpyAsync(ld, logits_host + (size_t)t0 * E, (size_t)tc * E * 4,
                            cudaMemcpyHostToDevice, P->s[0])) ||
        !ck(cudaEventRecord(P->ev_in[slot], P->s[0])))
      return MXMOE_ERR_CUDA;
    // compute: needs this chunk's inputs and the slot's output buffer back
    if (!ck(cudaStreamWaitEvent(P->s[1], P->ev_in[slot], 0))) return MXMOE_ERR_CUDA;
    if (c >= 2 && !ck(cudaStreamWaitEvent(P->s[1], P->ev_out[slot], 0))) return MXMOE_ERR_CUDA;
    const mxmoe_status st =
        forward_impl(xd, ld, w13q, w13s_mma, w2q, w2s_mma, true, tc, H, E, k, I, renormalize, od,
                     sb + CL.ws, CL.ws_bytes, P->s[1]);
    if (st != MXMOE_OK) return st;
    if (!ck(cudaEventRecord(P->ev_comp[slot], P->s[1]))) return MXMOE_ERR_CUDA;
    // d2h
    if (!ck(cudaStreamWaitEvent(P->s[2], P->ev_comp[slot], 0)) ||
        !ck(cudaMemcpyAsync(out_host + (size_t)t0 * H, od, (size_t)tc * H * 2,
                            cudaMemcpyDeviceToHost, P->s[2])) ||
        !ck(cudaEventRecord(P->ev_out[slot], P->s[2])))
      return MXMOE_ERR_CUDA;
  }
  // the caller's stream continues once every copy back has been issued and done
  if (!ck(cudaEventRecord(P->ev_done, P->s[2])) || !ck(cudaStreamWaitEvent(user, P->ev_done, 0)))
    return MXMOE_ERR_CUDA;
  return MXMOE_OK;
}

mxmoe_status moe_forward_mxfp8_host(const uint16_t* x_host, const float* logits_host,
                                    const uint8_t* w13q, const uint8_t* w13s_mma,
                                    const uint8_t* w2q, const uint8_t* w2s_mma, int T, int H,
                                    int E, int k, int I, int renormalize, uint16_t* out_host,
                                    int n_chunks, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0) return MXMOE_ERR_SHAPE;
  int sizes[kMaxHostChunks];
  const int n = host_chunk_plan(T, n_chunks, sizes);
  return host_pipeline(x_host, logits_host, w13q, w13s_mma, w2q, w2s_mma, T, H, E, k, I,
                       renormalize, out_host, sizes, n, ws, ws_bytes, stream);
}

mxmoe_status moe_forward_mxfp8_host_plan(const uint16_t* x_host, const float* logits_host,
                                         const uint8_t* w13q, const uint8_t* w13s_mma,
                                         const uint8_t* w2q, const uint8_t* w2s_mma, int T, int H,
                                         int E, int k, int I, int renormalize, uint16_t* out_host,
                                         const int32_t* chunk_tokens, int n_chunks, void* ws,
                                         size_t ws_bytes, void* stream) {
  if (!chunk_tokens || n_chunks <= 0 || n_chunks > kMaxHostChunks) return MXMOE_ERR_SHAPE;
  int sizes[kMaxHostChunks];
  for (int i = 0; i < n_chunks; ++i) sizes[i] = chunk_tokens[i];
  return host_pipeline(x_host, logits_host, w13q, w13s_mma, w2q, w2s_mma, T, H, E, k, I,
                       renormalize, out_host, sizes, n_chunks, ws, ws_bytes, stream);
}

}  // extern "C"
