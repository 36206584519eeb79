// Offloaded optimizer step ("bounded-streaming operators" summary, Methodology 4,
// OffloadStreamAdamW, eq. (5)) and the fused AdamW update it runs on each bucket.
//
// The update is elementwise and streams 30 bytes per parameter (p, m, v and an fp32
// gradient in; p, m, v and the bf16 working weight out), so the kernel is a plain
// bandwidth kernel: 16-byte vector accesses with streaming cache hints, several
// independent vectors in flight per thread, and a grid of a few resident blocks per SM.
// The same kernel serves state in HBM, in a staging slot, or in page-locked host memory
// that the GPU addresses across the host link.
#include <cuda_runtime.h>

#include <cmath>
#include <deque>

#include "../../include/moe.h"
#include "../../include/moe_adamw.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 4;
constexpr int kUnroll = 2;  // float4 groups per thread per iteration (no spills at 64 registers)

// One element of the AdamW update with decoupled weight decay, in the order the
// header states: decay, moments, bias-corrected step.
__device__ __forceinline__ void adam_elem(float& p, float& m, float& v, float g, const AdamConst& c) {
  p *= c.decay;
  m = fmaf(c.beta1, m, c.omb1 * g);
  v = fmaf(c.beta2, v, c.omb2 * g * g);
  const float denom = fmaf(sqrtf(v), c.inv_sqrt_bc2, c.eps);
  p = fmaf(-c.step_size, m / denom, p);
}

template <int GRAD>
__device__ __forceinline__ float4 load_grad4(const void* G, int64_t i) {
  if constexpr (GRAD == MOE_GRAD_F32) {
    return __ldcs(reinterpret_cast<const float4*>(G) + i);
  } else {
    const uint2 b = __ldcs(reinterpret_cast<const uint2*>(G) + i);
    return make_float4(bf16_lo(b.x), bf16_hi(b.x), bf16_lo(b.y), bf16_hi(b.y));
  }
}

template <int GRAD>
__device__ __forceinline__ float load_grad1(const void* G, int64_t i) {
  if constexpr (GRAD == MOE_GRAD_F32) {
    return reinterpret_cast<const float*>(G)[i];
  } else {
    return bf16_lo(reinterpret_cast<const uint16_t*>(G)[i]);
  }
}

template <int GRAD>
__global__ void __launch_bounds__(kThreads, kBlocksPerSm)
    adamw_kernel(float* __restrict__ P, float* __restrict__ M, float* __restrict__ V, const void* __restrict__ G,
                 uint16_t* __restrict__ W, int64_t n, AdamConst c) {
  const int64_t n4 = n >> 2;
  const int64_t nthreads = (int64_t)gridDim.x * kThreads;
  const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  float4* P4 = reinterpret_cast<float4*>(P);
  float4* M4 = reinterpret_cast<float4*>(M);
  float4* V4 = reinterpret_cast<float4*>(V);
  uint2* W4 = reinterpret_cast<uint2*>(W);
  for (int64_t base = tid; base < n4; base += nthreads * kUnroll) {
    float4 p[kUnroll], m[kUnroll], v[kUnroll], g[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + u * nthreads;
      if (i < n4) {
        p[u] = __ldcs(P4 + i);
        m[u] = __ldcs(M4 + i);
        v[u] = __ldcs(V4 + i);
        g[u] = load_grad4<GRAD>(G, i);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + u * nthreads;
      if (i < n4) {
        adam_elem(p[u].x, m[u].x, v[u].x, g[u].x, c);
        adam_elem(p[u].y, m[u].y, v[u].y, g[u].y, c);
        adam_elem(p[u].z, m[u].z, v[u].z, g[u].z, c);
        adam_elem(p[u].w, m[u].w, v[u].w, g[u].w, c);
        __stcs(P4 + i, p[u]);
        __stcs(M4 + i, m[u]);
        __stcs(V4 + i, v[u]);
        __stcs(W4 + i, make_uint2(pack_bf16(p[u].x, p[u].y), pack_bf16(p[u].z, p[u].w)));
      }
    }
  }
  // the last n mod 4 parameters
  const int64_t t = 4 * n4 + tid;
  if (t < n) {
    float p = P[t], m = M[t], v = V[t];
    adam_elem(p, m, v, load_grad1<GRAD>(G, t), c);
    P[t] = p;
    M[t] = m;
    V[t] = v;
    W[t] = static_cast<uint16_t>(pack_bf16(p, 0.0f) & 0xFFFFu);
  }
}

cudaError_t launch_adamw(float* P, float* M, float* V, const void* G, int grad_dtype, uint16_t* W, int64_t n,
                         const AdamConst& c, cudaStream_t s) {
  const int64_t groups = (n >> 2) + 1;
  const int64_t want = (groups + (int64_t)kThreads * kUnroll - 1) / ((int64_t)kThreads * kUnroll);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)device_sm_count() * kBlocksPerSm));
  if (grad_dtype == MOE_GRAD_F32)
    adamw_kernel<MOE_GRAD_F32><<<blocks, kThreads, 0, s>>>(P, M, V, G, W, n, c);
  else
    adamw_kernel<MOE_GRAD_BF16><<<blocks, kThreads, 0, s>>>(P, M, V, G, W, n, c);
  return cudaGetLastError();
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_hparams(const moe_adamw_hparams* h) {
  if (!h || h->step < 1) return false;
  if (!std::isfinite(h->lr) || !std::isfinite(h->weight_decay) || !std::isfinite(h->eps) || h->eps < 0.0) return false;
  if (!(h->beta1 >= 0.0 && h->beta1 < 1.0 && h->beta2 >= 0.0 && h->beta2 < 1.0)) return false;
  return true;
}

// Bias corrections and the other per-step scalars, formed in double and rounded once to fp32.
AdamConst constants(const moe_adamw_hparams& h) {
  const double t = (double)h.step;
  const double bc1 = 1.0 - std::pow(h.beta1, t);
  const double bc2 = 1.0 - std::pow(h.beta2, t);
  AdamConst c;
  c.decay = (float)(1.0 - h.lr * h.weight_decay);
  c.beta1 = (float)h.beta1;
  c.omb1 = (float)(1.0 - h.beta1);
  c.beta2 = (float)h.beta2;
  c.omb2 = (float)(1.0 - h.beta2);
  c.step_size = (float)(h.lr / bc1);
  c.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  c.eps = (float)h.eps;
  return c;
}

// Memory kind of a pointer as the runtime sees it; cudaMemoryTypeUnregistered for pageable memory.
cudaMemoryType kind_of(const void* p, void** dev_ptr = nullptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return cudaMemoryTypeUnregistered;
  }
  if (dev_ptr) *dev_ptr = a.devicePointer;
  return a.type;
}

bool device_addressable(const void* p) { return kind_of(p) != cudaMemoryTypeUnregistered; }

size_t slot_part_bytes(int64_t bucket) { return ((size_t)bucket * 4 + 255) / 256 * 256; }

// The library's three pipeline streams and their per-slot events, one set per (host thread, device).
struct OffloadStreams {
  int dev = -1;
  cudaStream_t h2d = nullptr, upd = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[MOE_ADAMW_MAX_SLOTS], updated[MOE_ADAMW_MAX_SLOTS], stored[MOE_ADAMW_MAX_SLOTS];
};
thread_local std::deque<OffloadStreams> g_off;   // indexed by device; created on first use, kept (stable addresses)

cudaError_t offload_streams(OffloadStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((int)g_off.size() <= dev) g_off.resize(dev + 1);
  OffloadStreams& o = g_off[dev];
  if (o.dev != dev) {
    for (cudaStream_t* s : {&o.h2d, &o.upd, &o.d2h})
      if ((e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    for (cudaEvent_t* ev : {&o.start, &o.done})
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < MOE_ADAMW_MAX_SLOTS; ++i)
      for (cudaEvent_t* ev : {&o.loaded[i], &o.updated[i], &o.stored[i]})
        if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    o.dev = dev;
  }
  *out = &o;
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_adamw_staging_bytes(int64_t bucket, int32_t slots, size_t* bytes) {
  if (!bytes || bucket < 4 || bucket % 4 != 0 || slots < 1 || slots > MOE_ADAMW_MAX_SLOTS)
    return MOE_ERR_INVALID_ARG;
  *bytes = (size_t)slots * 3 * slot_part_bytes(bucket);
  return MOE_OK;
}

int moe_adamw_offload_step(const moe_adamw_hparams* hp, int64_t n, int64_t bucket, int32_t slots, float* master,
                           float* exp_avg, float* exp_avg_sq, const void* grad, int32_t grad_dtype,
                           uint16_t* weight, void* staging, size_t staging_bytes, void* stream) {
  size_t need = 0;
  if (!valid_hparams(hp) || n < 0 || (grad_dtype != MOE_GRAD_F32 && grad_dtype != MOE_GRAD_BF16))
    return MOE_ERR_INVALID_ARG;
  if (moe_adamw_staging_bytes(bucket, slots, &need) != MOE_OK) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  for (const void* p : {(const void*)master, (const void*)exp_avg, (const void*)exp_avg_sq, grad,
                        (const void*)weight, (const void*)staging})
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  for (const void* p : {(const void*)master, (const void*)exp_avg, (const void*)exp_avg_sq})
    if (kind_of(p) != cudaMemoryTypeHost) return MOE_ERR_INVALID_ARG;
  if (!device_addressable(grad) || !device_addressable(weight) || !device_addressable(staging))
    return MOE_ERR_INVALID_ARG;
  if (staging_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;

  OffloadStreams* o = nullptr;
  cudaError_t e = offload_streams(&o);
  if (e != cudaSuccess) return record_cuda_error(e, "optimizer streams");
  const cudaStream_t caller = static_cast<cudaStream_t>(stream);
  const AdamConst c = constants(*hp);
  const size_t part = slot_part_bytes(bucket);
  const size_t gsize = grad_dtype == MOE_GRAD_F32 ? 4 : 2;
  float* host[3] = {master, exp_avg, exp_avg_sq};

  e = cudaEventRecord(o->start, caller);
  for (cudaStream_t s : {o->h2d, o->upd, o->d2h})
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, o->start, 0);
  if (e != cudaSuccess) return record_cuda_error(e, "fork optimizer streams");

  const int64_t G = (n + bucket - 1) / bucket;
  for (int64_t b = 0; b < G; ++b) {
    const int slot = (int)(b % slots);
    const int64_t off = b * bucket;
    const int64_t len = std::min(bucket, n - off);
    char* base = static_cast<char*>(staging) + (size_t)slot * 3 * part;
    float* dev[3] = {reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + part),
                     reinterpret_cast<float*>(base + 2 * part)};
    // (i) host to device, once the write-back of bucket b - slots has left the slot
    if (b >= slots) e = cudaStreamWaitEvent(o->h2d, o->stored[slot], 0);
    for (int a = 0; a < 3 && e == cudaSuccess; ++a)
      e = cudaMemcpyAsync(dev[a], host[a] + off, (size_t)len * 4, cudaMemcpyHostToDevice, o->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(o->loaded[slot], o->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(o->upd, o->loaded[slot], 0);
    if (e != cudaSuccess) return record_cuda_error(e, "bucket host-to-device copy");
    // (ii) fused update and bf16 working-weight refresh
    const void* g = static_cast<const char*>(grad) + (size_t)off * gsize;
    const int rc = timed_launch(MOE_K_ADAMW, "adamw update", o->upd, [&] {
      return launch_adamw(dev[0], dev[1], dev[2], g, grad_dtype, weight + off, len, c, o->upd);
    });
    if (rc != MOE_OK) return rc;
    e = cudaEventRecord(o->updated[slot], o->upd);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(o->d2h, o->updated[slot], 0);
    // (iii) write-back
    for (int a = 0; a < 3 && e == cudaSuccess; ++a)
      e = cudaMemcpyAsync(host[a] + off, dev[a], (size_t)len * 4, cudaMemcpyDeviceToHost, o->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(o->stored[slot], o->d2h);
    if (e != cudaSuccess) return record_cuda_error(e, "bucket write-back");
  }
  // the write-back stream is last in every bucket's chain, so its final event covers the step
  e = cudaEventRecord(o->done, o->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(caller, o->done, 0);
  if (e != cudaSuccess) return record_cuda_error(e, "join optimizer streams");
  return MOE_OK;
}

int moe_adamw_step(const moe_adamw_hparams* hp, int64_t n, float* master, float* exp_avg, float* exp_avg_sq,
                   const void* grad, int32_t grad_dtype, uint16_t* weight, void* stream) {
  if (!valid_hparams(hp) || n < 0 || (grad_dtype != MOE_GRAD_F32 && grad_dtype != MOE_GRAD_BF16))
    return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  float* state[3] = {master, exp_avg, exp_avg_sq};
  float* dstate[3];
  cudaMemoryType kind0 = cudaMemoryTypeUnregistered;
  for (int a = 0; a < 3; ++a) {
    if (!aligned16(state[a])) return MOE_ERR_INVALID_ARG;
    void* dp = nullptr;
    const cudaMemoryType k = kind_of(state[a], &dp);
    const bool host = k == cudaMemoryTypeHost;
    if (k == cudaMemoryTypeUnregistered || (a > 0 && host != (kind0 == cudaMemoryTypeHost)))
      return MOE_ERR_INVALID_ARG;
    if (a == 0) kind0 = k;
    dstate[a] = host ? static_cast<float*>(dp) : state[a];
    if (!aligned16(dstate[a])) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(grad) || !aligned16(weight) || !device_addressable(grad) || !device_addressable(weight))
    return MOE_ERR_INVALID_ARG;
  const AdamConst c = constants(*hp);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  return timed_launch(MOE_K_ADAMW, "adamw update", s, [&] {
    return launch_adamw(dstate[0], dstate[1], dstate[2], grad, grad_dtype, weight, n, c, s);
  });
}

}  // extern "C"
