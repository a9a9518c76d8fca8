// moe_route_quant_mxfp8_noalloc: the fused route + MX quant without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// layer: an inference runtime that hands every byte of HBM to its own pool at
// start-up and forbids cudaMalloc afterwards (a cudaMalloc there can
// synchronize the device and fragments the pool), a plug-in whose host
// framework owns device memory and offers no workspace hook, or a
// latency-critical path that must not pay cudaMalloc's cost.  They still own
// their inputs and outputs, but not a scratch buffer.  For them the routing
// step's only scratch -- the per-block expert histograms and their scanned
// block bases -- lives in the
// file-scope device array below, which every GPU that loads this library
// holds until the process exits.
#include <mutex>

#include "internal.h"
#include "mxmoe.h"

namespace mxmoe {

// Scratch for ceil(T / 64) * E <= 262144 histogram entries (1 MiB) and as
// many block bases.
constexpr int64_t kNoAllocHistInts = 262144;
constexpr size_t kNoAllocScratchInts = 2 * kNoAllocHistInts;
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};
uint64_t g_scratch_ctx[kMaxDevices] = {0};  // context id the cached address belongs to

// Device address of g_route_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, never a device address, so the
// address is looked up with that device current: once per device and
// context (after cudaDeviceReset the device's new primary context holds a
// new copy of the array, and the address is looked up again).
cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  const uint64_t ctx = context_id();
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    g_scratch_ctx[dev] = context_id();
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}
}  // namespace

}  // namespace mxmoe

using namespace mxmoe;

extern "C" mxmoe_status moe_route_quant_mxfp8_noalloc(
    const uint16_t* x, const float* logits, int T, int H, int E, int k, int renormalize,
    uint8_t* xq, uint8_t* xs, int32_t* topk_ids, float* topk_w, int32_t* sorted_to_src,
    int32_t* src_to_sorted, int64_t* expert_counts, int64_t* expert_offsets, void* stream) {
  if (T < 0 || H <= 0 || H % 32 != 0 || E <= 0 || E > 1024 || k < 1 || k > 32 || k > E)
    return MXMOE_ERR_SHAPE;
  if ((int64_t)T * k >= (1ll << 31)) return MXMOE_ERR_SHAPE;
  // the built-in scratch is the workspace: reject sizes it cannot hold
  const int64_t nb = ceil_div(T, kRouteTokensPerBlock);
  if (nb * (int64_t)E > kNoAllocHistInts) return MXMOE_ERR_WORKSPACE;
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MXMOE_ERR_CUDA;
  return moe_route_quant_mxfp8(x, logits, T, H, E, k, renormalize, xq, xs, topk_ids, topk_w,
                               sorted_to_src, src_to_sorted, expert_counts, expert_offsets,
                               scratch, kNoAllocScratchInts * sizeof(int32_t), stream);
}
