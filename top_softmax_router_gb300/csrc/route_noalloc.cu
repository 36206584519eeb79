// moe_route_noalloc: the router for callers that cannot allocate device memory.
//
// moe_route needs a caller-provided workspace for the fp32 logits.  Some
// callers have no way to provide one: a serving process that hands all device
// memory to its own pool at start-up (so any later cudaMalloc fails or
// fragments that pool), or a plugin running inside a host framework that owns
// the device allocator and gives extensions no way to borrow from it.  This
// entry point keeps the logits in a fixed array that lives in the library's
// own device image instead, so it allocates nothing at call time.
//
// The array below is sized for MOE_ROUTE_NOALLOC_MAX_LOGITS fp32 logits
// (16 MiB).  Every GPU on which the library is loaded holds it until the
// process exits.  All calls share it: two calls whose kernels overlap on the
// GPU (different streams, or different host threads) race on it and give
// undefined results; calls on one stream are ordered and safe.  Each call
// writes every logit it later reads, so nothing in it has to start at zero.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace {

static __device__ __align__(256) float g_route_logits[MOE_ROUTE_NOALLOC_MAX_LOGITS];

// Device address of g_route_logits, looked up once per device with that device
// current (in host code the symbol is only a host-side stand-in).
constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_addr[kMaxDevices] = {nullptr};

int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_logits) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_addr[dev] = static_cast<float*>(p);
  }
  *out = g_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_route_noalloc(const moe_config* cfg, const uint16_t* X, const float* Wr, const float* bias,
                                 int32_t* topk_idx, float* gates, void* stream) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  if (c.N < 0 || c.H <= 0 || c.E <= 0 || c.k <= 0 || c.I <= 0 || c.c <= 0 || c.K_max <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c.H % 64 != 0 || c.I % 64 != 0 || c.E > 1024 || c.k > c.E || c.k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)c.N * c.E > (int64_t)MOE_ROUTE_NOALLOC_MAX_LOGITS) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.N == 0) return MOE_OK;
  if (!aligned16(X) || !aligned16(Wr) || !aligned16(topk_idx) || !aligned16(gates)) return MOE_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  float* logits = nullptr;
  const int r = scratch_for_current_device(&logits);
  if (r != MOE_OK) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (moe::launch_router_logits(X, Wr, bias, logits, c.N, c.H, c.E, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_router_topk(logits, topk_idx, gates, c.N, c.E, c.k, nullptr, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
