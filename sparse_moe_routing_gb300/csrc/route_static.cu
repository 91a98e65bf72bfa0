// moe_route_static: routing that needs no caller-provided workspace.
//
// Some callers cannot call cudaMalloc: a plugin run by a host framework that
// owns every device allocation and hands its plugins no allocator, or a
// serving loop that must not allocate once it is running (an allocation can
// synchronise the device and adds latency jitter). moe_route needs a
// workspace for its fp32 router logits; this variant keeps those logits in a
// fixed array in the library's own device memory instead, so the caller
// passes only the inputs and the outputs. It runs moe_route's CUDA-core
// router kernels at every batch size (moe_route itself switches to the
// tensor-core router contraction from 128 bf16 tokens, whose logits can
// differ from these in the last bits).
//
// The array is a file-scope static __device__ object of kStaticLogits floats
// (4 MiB). Every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it; make that first call before any stream
// capture. A device reset (cudaDeviceReset) unloads the library's module and
// leaves the cached address stale: a process that resets a device must not
// call this entry point on it again. All calls share the one array and it
// keeps the last call's contents; nothing in it has to start at zero because
// every call overwrites the logits it reads. Calls whose kernels overlap on
// the GPU (two streams, or two threads) race on the array and must be
// serialised by the caller.
#include "moe_route.h"

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kStaticLogits = (size_t)1 << 20;  // floats: T * (E + 1) at most

static __device__ __align__(256) float g_route_logits[kStaticLogits];

// Device address of g_route_logits per device ordinal (< 64), looked up once
// with that device current; null until then. Concurrent first calls on one
// device may both look it up and store the same address.
std::atomic<float*> g_logits_addr[64];

// The array's device address on the current device, or null (with the CUDA
// error recorded) if the lookup fails.
float* static_logits() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    set_last_cuda_error(cudaErrorInvalidDevice);
    return nullptr;
  }
  float* a = g_logits_addr[dev].load(std::memory_order_acquire);
  if (!a) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_logits);
    if (e != cudaSuccess || !p) {
      set_last_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return nullptr;
    }
    a = static_cast<float*>(p);
    g_logits_addr[dev].store(a, std::memory_order_release);
  }
  return a;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_static(const void* x, const void* W_router,
                                         const float* expert_bias, const void* w_shared,
                                         const moe_cfg_t* cfg, int32_t* topk_ids, float* weights,
                                         float* s_shared, void* stream) {
  using namespace moe;
  // moe_route's checks in moe_route's order, without the workspace check
  moe_status_t s = validate_route_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !W_router || !topk_ids || !weights) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W_router) || !aligned16(topk_ids) || !aligned16(weights))
    return MOE_ERR_INVALID_ARG;
  if (s_shared && (!w_shared || !aligned16(w_shared) || !aligned16(s_shared)))
    return MOE_ERR_INVALID_ARG;
  if (expert_bias && !aligned16(expert_bias)) return MOE_ERR_INVALID_ARG;
  // the one limit of its own: the logits must fit the array
  if ((size_t)cfg->T * (size_t)(cfg->n_experts + 1) > kStaticLogits) return MOE_ERR_UNSUPPORTED;
  float* logits = static_logits();
  if (!logits) return MOE_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouterArgs ra{x, W_router, s_shared ? w_shared : nullptr, logits, cfg->T, cfg->d_model,
                cfg->n_experts};
  TopkArgs ta{};
  ta.logits = logits;
  ta.bias = cfg->router == MOE_ROUTER_SIGMOID_GROUP_TOPK ? expert_bias : nullptr;
  ta.topk_ids = topk_ids;
  ta.weights = weights;
  ta.s_shared = s_shared;
  ta.T = cfg->T;
  ta.E = cfg->n_experts;
  ta.k = cfg->top_k;
  ta.kind = cfg->router;
  ta.n_group = cfg->n_group;
  ta.topk_group = cfg->topk_group;
  ta.has_shared_logit = ra.w_shared ? 1 : 0;
  ta.routed_scaling = cfg->routed_scaling;
  ta.renorm_clamp = cfg->renorm_clamp;
  cudaError_t e = launch_router_logits(ra, cfg->act_dtype == MOE_BF16, st);
  if (e == cudaSuccess) e = launch_router_topk(ta, st);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
