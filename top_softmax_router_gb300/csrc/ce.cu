// Vocabulary-projection cross-entropy head with a bounded logit working set (include/moe_ce.h).
//
// "bounded-streaming operators" summary, Methodology 2 (Ring-DTP), eqs. (2)-(3); "Training
// Trillion-Parameter MoE ..." blog, section 3.5 (vocabulary-axis chunking, two-pass scan).
//
// Forward: one persistent grouped-GEMM launch (a single "expert", W) whose epilogue turns each
// 128-token x 256-class logit tile, straight from tensor memory, into per-token (max, sum of exp)
// pairs; ce_merge_kernel folds each token's pairs in class order by the online-softmax recurrence.
// Backward, per vocabulary strip: recompute the strip's logits and write d (bf16) for the strip,
// then dX += d W_strip (fp32, TMA store on the first strip and reduce-add after) and
// dW_strip = d^T X (fp32, contraction over the tokens).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <string>

#include "../../include/moe.h"
#include "../../include/moe_ce.h"
#include "common.cuh"
#include "gemm_launch.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

thread_local moe_ce_stats g_ce_stats = {};
// The logit GEMMs have hundreds of 256-class column tiles: walked tile-major, every CTA would stream
// its own slab of W from HBM.  Bands of 8 row tiles make the CTAs at work share ~19 W tiles and 8 X
// tiles at a time.
constexpr int kBand = 8;

struct CeLayout {
  int T;       // 128-token row tiles
  int NT;      // 256-class tiles over the whole vocabulary (forward partials per token)
  int Vs;      // classes per backward strip (multiple of 256)
  int S;       // strips
  int nctr;    // work counters
  size_t tiles, tile_count, active, active_count, expert_off, ctr;
  size_t part_m, part_z, tgt, fwd_total;
  size_t dlog, dxacc, bwd_total;
};

CeLayout ce_layout(const moe_ce_config& c) {
  CeLayout L = {};
  const int64_t N = c.N, H = c.H, V = c.V;
  L.T = (int)((N + 127) / 128);
  L.NT = (int)((V + 255) / 256);
  const int64_t per = (V + c.P - 1) / c.P;
  L.Vs = (int)((per + 255) / 256 * 256);
  L.S = (int)((V + L.Vs - 1) / L.Vs);
  L.nctr = 1 + 3 * L.S;
  size_t o = align_up(sizeof(WsHeader));
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.tiles = take((size_t)L.T * 8);
  L.tile_count = take(4);
  L.active = take(4);
  L.active_count = take(4);
  L.expert_off = take(8);
  L.ctr = take((size_t)L.nctr * 4);
  const size_t common = o;
  L.part_m = take((size_t)N * L.NT * 4);
  L.part_z = take((size_t)N * L.NT * 4);
  L.tgt = take((size_t)N * 4);
  L.fwd_total = o;
  o = common;
  L.dlog = take((size_t)N * L.Vs * 2);
  L.dxacc = take((size_t)N * H * 4);
  L.bwd_total = o;
  return L;
}

int ce_validate(const moe_ce_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->N < 0 || c->H < 0 || c->V < 0 || c->P < 0) return MOE_ERR_INVALID_ARG;
  if (c->H < 64 || c->H % 64 != 0 || c->V < 1 || c->P < 1 || c->P > c->V) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The row-tile list (one "expert", 0), the single-expert segment arrays of the weight-gradient GEMM,
// and zeroed work counters.
__global__ void ce_setup_kernel(int2* tiles, int* tile_count, int* active, int* active_count, int* expert_off,
                                int* ctr, int nctr, int N, int T) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    const int rows = min(128, N - 128 * t);
    tiles[t] = make_int2(128 * t, rows << 16);
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < nctr; i += blockDim.x) ctr[i] = 0;
    if (threadIdx.x == 0) {
      *tile_count = T;
      active[0] = 0;
      *active_count = 1;
      expert_off[0] = 0;
      expert_off[1] = N;
    }
  }
}

// eq. (3) for two partial states: (m, z) with z = sum of exp(y - m) over the classes seen.
__device__ __forceinline__ void fold(float& m, float& z, float m2, float z2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    z = z2;
    return;
  }
  const float mn = fmaxf(m, m2);
  z = z * expf(m - mn) + z2 * expf(m2 - mn);
  m = mn;
}

// One warp per token: lane l folds tiles l, l+32, ... in order, then the lanes are folded by a
// butterfly (the fold is commutative, so every lane ends with the same bits).
__global__ void __launch_bounds__(256) ce_merge_kernel(const float* __restrict__ pm, const float* __restrict__ pz,
                                                       const float* __restrict__ tgt, const int* __restrict__ targets,
                                                       float* __restrict__ loss, float* __restrict__ lse, int N,
                                                       int NT, int V, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (n >= N) return;
  float m = -INFINITY, z = 0.0f;
  for (int i = lane; i < NT; i += 32) fold(m, z, pm[n * NT + i], pz[n * NT + i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, off);
    fold(m, z, m2, z2);
  }
  if (lane == 0) {
    const float l = m + logf(z);
    const int t = targets[n];
    const bool ok = t >= 0 && t < V;
    if (!ok) report(status, MOE_ERR_DEVICE_CHECK, 401);
    lse[n] = l;
    loss[n] = ok ? l - tgt[n] : l;
  }
}

// sum_n loss[n] / N in a fixed order: strided per-thread sums, then a tree over the block.
__global__ void __launch_bounds__(1024) ce_mean_kernel(const float* __restrict__ loss, float* out, int N) {
  __shared__ float s[1024];
  float a = 0.0f;
  for (int i = threadIdx.x; i < N; i += 1024) a += loss[i];
  s[threadIdx.x] = a;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) s[threadIdx.x] += s[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = N > 0 ? s[0] / (float)N : 0.0f;
}

GemmParams ce_params(const CeLayout& L, uint8_t* w, int* status, int ctr_slot) {
  GemmParams p = {};
  p.tiles = reinterpret_cast<const int2*>(w + L.tiles);
  p.tile_count = reinterpret_cast<const int*>(w + L.tile_count);
  p.active = reinterpret_cast<const int*>(w + L.active);
  p.active_count = reinterpret_cast<const int*>(w + L.active_count);
  p.expert_off = reinterpret_cast<const int*>(w + L.expert_off);
  p.work_ctr = reinterpret_cast<int*>(w + L.ctr) + ctr_slot;
  p.status = status;
  p.n_problems = 1;
  return p;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_ce_workspace_bytes(const moe_ce_config* cfg, size_t* fwd_bytes, size_t* bwd_bytes) {
  const int v = ce_validate(cfg);
  if (v != MOE_OK) return v;
  const CeLayout L = ce_layout(*cfg);
  if (fwd_bytes) *fwd_bytes = L.fwd_total;
  if (bwd_bytes) *bwd_bytes = L.bwd_total;
  return MOE_OK;
}

int moe_ce_forward(const moe_ce_config* cfg, const uint16_t* X, const uint16_t* W, const int32_t* targets,
                   float* loss, float* lse, float* loss_mean, void* ws, size_t ws_bytes, void* stream) {
  int v = ce_validate(cfg);
  if (v != MOE_OK) return v;
  const moe_ce_config& c = *cfg;
  const CeLayout L = ce_layout(c);
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.fwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(W) || (c.N > 0 && (!aligned16(X) || !aligned16(targets) || !aligned16(loss) || !aligned16(lse))))
    return MOE_ERR_INVALID_ARG;
  if (loss_mean && (reinterpret_cast<uintptr_t>(loss_mean) & 3u)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  int launches = 0;
  if (c.N > 0) {
    auto run = [&](int kind, const char* what, const std::function<cudaError_t()>& f) {
      const int rc = timed_launch(kind, what, s, f);
      if (rc == MOE_OK) ++launches;
      return rc;
    };
    if ((v = run(MOE_K_PLAN, "ce setup", [&] {
           ce_setup_kernel<<<(L.T + 255) / 256, 256, 0, s>>>(
               reinterpret_cast<int2*>(w + L.tiles), reinterpret_cast<int*>(w + L.tile_count),
               reinterpret_cast<int*>(w + L.active), reinterpret_cast<int*>(w + L.active_count),
               reinterpret_cast<int*>(w + L.expert_off), reinterpret_cast<int*>(w + L.ctr), L.nctr, c.N, L.T);
           return cudaGetLastError();
         })) != MOE_OK)
      return v;
    CUtensorMap a, b;
    if (!make_map_2d(&a, X, c.H, c.N, 64, 128) || !make_map_3d(&b, W, c.H, c.V, 1, 64, 256))
      return record_cuda_error(cudaErrorInvalidValue, "ce tensor maps");
    GemmParams p = ce_params(L, w, status, 0);
    p.nk = c.H / GEMM_BK;
    p.n_tiles = L.NT;
    p.N = c.V;
    p.targets = targets;
    p.part_m = reinterpret_cast<float*>(w + L.part_m);
    p.part_z = reinterpret_cast<float*>(w + L.part_z);
    p.tgt_logit = reinterpret_cast<float*>(w + L.tgt);
    p.col0 = 0;
    p.ldp = L.NT;
    p.band = kBand;
    p.limit_ns = wait_limit_ns();
    if ((v = run(MOE_K_CE_LOGITS, "ce logits", [&] {
           return launch_grouped_gemm<EPI_LSE, false, false, false, 256, false, false>(a, a, b, b, p,
                                                                                     device_sm_count(), s);
         })) != MOE_OK)
      return v;
    if ((v = run(MOE_K_CE_MERGE, "ce merge", [&] {
           ce_merge_kernel<<<(c.N + 7) / 8, 256, 0, s>>>(p.part_m, p.part_z, p.tgt_logit, targets, loss, lse, c.N,
                                                         L.NT, c.V, status);
           return cudaGetLastError();
         })) != MOE_OK)
      return v;
  }
  if (loss_mean) {
    const int rc = timed_launch(MOE_K_CE_MERGE, "ce mean", s, [&] {
      ce_mean_kernel<<<1, 1024, 0, s>>>(loss, loss_mean, c.N);
      return cudaGetLastError();
    });
    if (rc != MOE_OK) return rc;
    ++launches;
  }
  moe_ce_stats st = {};
  st.strips = L.S;
  st.strip_classes = L.Vs;
  st.strip_bytes = 0;
  st.strip_bound_bytes = (int64_t)c.N * ((c.V + c.P - 1) / c.P) * 2;
  st.partial_bytes = (int64_t)c.N * L.NT * 8;
  st.workspace_bytes = (int64_t)L.fwd_total;
  st.kernel_launches = launches;
  g_ce_stats = st;
  return MOE_OK;
}

int moe_ce_backward(const moe_ce_config* cfg, const uint16_t* X, const uint16_t* W, const int32_t* targets,
                    const float* lse, const float* dloss, uint16_t* dX, float* dW, void* ws, size_t ws_bytes,
                    void* stream) {
  int v = ce_validate(cfg);
  if (v != MOE_OK) return v;
  const moe_ce_config& c = *cfg;
  const CeLayout L = ce_layout(c);
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.bwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(W) || !aligned16(dW)) return MOE_ERR_INVALID_ARG;
  if (c.N > 0 && (!aligned16(X) || !aligned16(targets) || !aligned16(lse) || !aligned16(dloss) || !aligned16(dX)))
    return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  int launches = 0;
  if (c.N == 0) {
    const cudaError_t e = cudaMemsetAsync(dW, 0, (size_t)c.V * c.H * 4, s);
    if (e != cudaSuccess) return record_cuda_error(e, "clear dW");
  } else {
    auto run = [&](int kind, const char* what, const std::function<cudaError_t()>& f) {
      const int rc = timed_launch(kind, what, s, f);
      if (rc == MOE_OK) ++launches;
      return rc;
    };
    if ((v = run(MOE_K_PLAN, "ce setup", [&] {
           ce_setup_kernel<<<(L.T + 255) / 256, 256, 0, s>>>(
               reinterpret_cast<int2*>(w + L.tiles), reinterpret_cast<int*>(w + L.tile_count),
               reinterpret_cast<int*>(w + L.active), reinterpret_cast<int*>(w + L.active_count),
               reinterpret_cast<int*>(w + L.expert_off), reinterpret_cast<int*>(w + L.ctr), L.nctr, c.N, L.T);
           return cudaGetLastError();
         })) != MOE_OK)
      return v;
    uint16_t* dlog = reinterpret_cast<uint16_t*>(w + L.dlog);
    float* dxacc = reinterpret_cast<float*>(w + L.dxacc);
    const int sms = device_sm_count();
    CUtensorMap xa, xb;   // X as the A operand (K-major rows) and as the B operand of dW (MN-major)
    if (!make_map_2d(&xa, X, c.H, c.N, 64, 128) || !make_map_2d(&xb, X, c.H, c.N, 64, 64))
      return record_cuda_error(cudaErrorInvalidValue, "ce tensor maps");
    CUtensorMap dxo;
    if (!make_map_3d_f32(&dxo, dxacc, c.H, c.N, 1, 32, 32))
      return record_cuda_error(cudaErrorInvalidValue, "ce tensor maps");
    for (int st = 0; st < L.S; ++st) {
      const int v0 = st * L.Vs;
      const int width = std::min(L.Vs, c.V - v0);
      const uint16_t* Ws = W + (size_t)v0 * c.H;
      CUtensorMap wk, wm, da, dm, dwo;
      if (!make_map_3d(&wk, Ws, c.H, width, 1, 64, 256) || !make_map_3d(&wm, Ws, c.H, width, 1, 64, 64) ||
          !make_map_2d_strided(&da, dlog, width, c.N, L.Vs, 64, 128) ||
          !make_map_2d_strided(&dm, dlog, width, c.N, L.Vs, 64, 64) ||
          !make_map_3d_f32(&dwo, dW + (size_t)v0 * c.H, c.H, width, 1, 32, 32))
        return record_cuda_error(cudaErrorInvalidValue, "ce tensor maps");
      // d for this strip
      GemmParams p = ce_params(L, w, status, 1 + 3 * st);
      p.nk = c.H / GEMM_BK;
      p.n_tiles = (width + 255) / 256;
      p.N = width;
      p.ldo = L.Vs;
      p.out0 = dlog;
      p.targets = targets;
      p.lse = lse;
      p.rowscale = dloss;
      p.col0 = v0;
      p.band = kBand;
      p.limit_ns = wait_limit_ns();
      if ((v = run(MOE_K_CE_DLOGIT, "ce dlogit", [&] {
             return launch_grouped_gemm<EPI_DLOGIT, false, false, false, 256, false, false>(xa, xa, wk, wk, p, sms,
                                                                                          s);
           })) != MOE_OK)
        return v;
      // dX (+)= d W_strip: A = d [N, width] K-major, B = W_strip [width, H] MN-major
      GemmParams q = ce_params(L, w, status, 2 + 3 * st);
      q.nk = (width + GEMM_BK - 1) / GEMM_BK;
      q.n_tiles = (c.H + 255) / 256;
      q.N = c.H;
      q.chunk = st;
      q.limit_ns = wait_limit_ns();
      if ((v = run(MOE_K_CE_DX, "ce dX", [&] {
             return launch_grouped_gemm<EPI_ACC, false, true, false, 256, false, false>(da, da, wm, wm, q, sms, s,
                                                                                      &dxo);
           })) != MOE_OK)
        return v;
      // dW_strip = d^T X: contraction over the tokens; A = d (MN-major, M = classes), B = X (MN-major)
      GemmParams r = ce_params(L, w, status, 3 + 3 * st);
      r.m_tiles = (width + GEMM_BM - 1) / GEMM_BM;
      r.n_tiles = (c.H + 255) / 256;
      r.M = width;
      r.N = c.H;
      r.first_touch = nullptr;   // every strip's rows are written once: plain stores
      r.limit_ns = wait_limit_ns();
      if ((v = run(MOE_K_CE_DW, "ce dW", [&] {
             return launch_grouped_gemm<EPI_DW, true, true, true, 256, false, false>(dm, dm, xb, xb, r, sms, s,
                                                                                   &dwo);
           })) != MOE_OK)
        return v;
    }
    if ((v = run(MOE_K_FINAL, "ce dX to bf16",
                 [&] { return launch_to_bf16(dxacc, dX, (int64_t)c.N * c.H, s); })) != MOE_OK)
      return v;
  }
  moe_ce_stats st = {};
  st.strips = L.S;
  st.strip_classes = L.Vs;
  st.strip_bytes = (int64_t)c.N * L.Vs * 2;
  st.strip_bound_bytes = (int64_t)c.N * ((c.V + c.P - 1) / c.P) * 2;
  st.partial_bytes = 0;
  st.workspace_bytes = (int64_t)L.bwd_total;
  st.kernel_launches = launches;
  g_ce_stats = st;
  return MOE_OK;
}

int moe_ce_last_stats(moe_ce_stats* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = g_ce_stats;
  return MOE_OK;
}

}  // extern "C"
