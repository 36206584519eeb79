// C ABI of libmoe.so (declared in include/moe.h): argument checks, workspace
// layout and the chunk schedule of the bounded-streaming MoE block.
//
// Schedule ("bounded-streaming operators" summary, Methodology 1,
// PipelinedLLEP): K = min(ceil(N/c), K_max) chunks, c_eff = ceil(N/K), chunk i
// holds tokens i, i+K, ...  Forward runs chunks 0..K-1; backward runs K-1..0
// and recomputes each chunk's expert intermediates into the same workspace
// slots, so at most one chunk's routed buffers are ever live.  The dispatch
// gather either fills a permuted buffer (MOE_DISPATCH_GATHER: the chunk's two
// routed buffers, {Xp, Op} forward and {Xp, dYp/dXp} backward) or is fused
// into the expert GEMMs' operand loads (MOE_DISPATCH_ON_LOAD: only the expert
// output, Op forward and dXp backward, is materialised).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <deque>
#include <functional>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Wait-accounting counters of the diagnostic build (moe_diag_gemm_wait_stats); NULL until first enabled.
std::atomic<unsigned long long*> g_wait_stats{nullptr};
unsigned long long* gemm_wait_stats_buffer() { return g_wait_stats.load(); }

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

thread_local std::string g_err;
thread_local moe_stats g_stats = {};
std::atomic<int64_t> g_limit_ns{2000000000LL};
constexpr int64_t kDefaultLimitNs = 2000000000LL;

// ------------------------------------------------------------------ profiling
struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_free_events;
int g_prof_launches[MOE_K_COUNT];
double g_prof_ms[MOE_K_COUNT];
const char* kKernelNames[MOE_K_COUNT] = {"router_logits", "router_topk", "plan",      "gather",
                                         "gemm_gateup",   "gemm_down",   "combine",   "gemm_dact",
                                         "gemm_dw",       "gemm_dx",     "unpermute", "router_dw",
                                         "zero",          "hop_plan",    "finalize",  "adamw",
                                         "ce_logits",     "ce_merge",    "ce_dlogit", "ce_dx",
                                         "ce_dw",         "route_grad"};

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

int cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return MOE_ERR_CUDA;
}

// Runs one launch, bracketed by events when profiling is on.
struct Launcher {
  cudaStream_t s;
  int launches = 0;
  template <class F>
  int operator()(int kind, const char* what, F&& f) {
    cudaEvent_t a = nullptr, b = nullptr;
    if (g_prof_on) {
      std::lock_guard<std::mutex> g(g_prof_mu);
      a = take_event();
      b = take_event();
    }
    if (a) cudaEventRecord(a, s);
    cudaError_t e = f();
    if (b) cudaEventRecord(b, s);
    if (a) {
      std::lock_guard<std::mutex> g(g_prof_mu);
      g_prof.push_back({kind, a, b});
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    ++launches;
    return MOE_OK;
  }
};

// ------------------------------------------------------------------ shapes
int validate(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->N < 0 || c->H <= 0 || c->E <= 0 || c->k <= 0 || c->I <= 0 || c->c <= 0 || c->K_max <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->H % 64 != 0 || c->I % 64 != 0 || c->E > 1024 || c->k > c->E || c->k > 32)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((int64_t)c->N * c->k > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

void chunk_plan(const moe_config& c, int* K, int* c_eff) {
  if (c.N == 0) {
    *K = 0;
    *c_eff = 0;
    return;
  }
  const int64_t need = ((int64_t)c.N + c.c - 1) / c.c;
  *K = (int)(need < c.K_max ? need : c.K_max);
  *c_eff = (int)(((int64_t)c.N + *K - 1) / *K);
}

struct Layout {
  int K, c_eff, kc_max, T_max, T2_max, n_dact;
  size_t expert_off, row_route, row_of, tiles, tile_count, tiles2, tile2_count, active, active_count, first_touch;
  size_t work_ctr;                                  // [K][GEMM_CTR_SLOTS] GEMM work counters
  size_t plan_counts;                               // multi-block plan scratch (K = 1 only)
  int count_blocks;
  size_t logits;
  bool on_load;                                     // MOE_DISPATCH_ON_LOAD: no Xp / dYp buffers
  size_t xp, op, act;                               // forward (xp unused on load)
  size_t b_xp, b_dyp, b_gate, b_up, b_gact, b_dgp, b_dlogit, b_dlrow, b_rdw;  // backward (b_rdw: router dW partials;
                                                    // b_dyp holds dYp, then dXp; on load only dXp)
  size_t route_total, fwd_total, bwd_total;
};

std::atomic<int> g_dispatch{MOE_DISPATCH_GATHER};

Layout make_layout(const moe_config& c) {
  Layout L = {};
  L.on_load = g_dispatch.load() == MOE_DISPATCH_ON_LOAD;
  chunk_plan(c, &L.K, &L.c_eff);
  const int64_t K = L.K, E = c.E, k = c.k, N = c.N, H = c.H, I = c.I;
  L.kc_max = (int)(k * L.c_eff);
  L.T_max = (L.kc_max + 127) / 128 + c.E;
  L.T2_max = (L.kc_max + 255) / 256 + c.E;
  L.n_dact = dgate_partials(c.I);
  size_t o = align_up(sizeof(WsHeader));
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.expert_off = take(K * (E + 1) * 4);
  L.row_route = take(K * (size_t)L.kc_max * 4);
  L.row_of = take(N * k * 4);
  L.tiles = take(K * (size_t)L.T_max * 8);
  L.tile_count = take(K * 4);
  L.tiles2 = take(K * (size_t)L.T2_max * 8);
  L.tile2_count = take(K * 4);
  L.active = take(K * E * 4);
  L.active_count = take(K * 4);
  L.first_touch = take(E * 4);
  L.work_ctr = take(K * GEMM_CTR_SLOTS * 4);
  L.count_blocks = L.K == 1 ? plan_count_blocks((int64_t)L.kc_max) : 0;
  L.plan_counts = take((size_t)L.count_blocks * E * 4);
  const size_t common = o;
  L.logits = take(N * E * 4);
  L.route_total = o;
  o = common;
  const size_t kc = (size_t)L.kc_max;
  if (!L.on_load) L.xp = take(kc * H * 2);
  L.op = take(kc * H * 2);
  L.act = take(kc * I * 2);
  L.fwd_total = o;
  o = common;
  if (!L.on_load) L.b_xp = take(kc * H * 2);
  L.b_dyp = take(kc * H * 2);
  L.b_gate = take(kc * I * 2);
  L.b_up = take(kc * I * 2);
  L.b_gact = take(kc * I * 2);
  L.b_dgp = take(kc * L.n_dact * 4);
  L.b_dlogit = take(N * k * 4);
  L.b_dlrow = take(kc * 4);
  L.b_rdw = take((size_t)L.T_max * H * 4);
  L.bwd_total = o;
  return L;
}

PlanPtrs plan_ptrs(const moe_config& c, const Layout& L, uint8_t* ws) {
  PlanPtrs p;
  p.expert_off = reinterpret_cast<int*>(ws + L.expert_off);
  p.row_route = reinterpret_cast<int*>(ws + L.row_route);
  p.row_of = reinterpret_cast<int*>(ws + L.row_of);
  p.tiles = reinterpret_cast<int2*>(ws + L.tiles);
  p.tile_count = reinterpret_cast<int*>(ws + L.tile_count);
  p.tiles2 = reinterpret_cast<int2*>(ws + L.tiles2);
  p.tile2_count = reinterpret_cast<int*>(ws + L.tile2_count);
  p.active = reinterpret_cast<int*>(ws + L.active);
  p.active_count = reinterpret_cast<int*>(ws + L.active_count);
  p.first_touch = reinterpret_cast<int*>(ws + L.first_touch);
  p.block_counts = reinterpret_cast<int*>(ws + L.plan_counts);
  p.count_blocks = L.count_blocks;
  p.N = c.N;
  p.E = c.E;
  p.k = c.k;
  p.K = L.K;
  p.c_eff = L.c_eff;
  p.kc_max = L.kc_max;
  p.T_max = L.T_max;
  p.T2_max = L.T2_max;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

void set_stats(const moe_config& c, const Layout& L, int launches, size_t ws_used, int routed_buffers,
               int inter_buffers) {
  moe_stats s = {};
  s.K = L.K;
  s.c_eff = L.c_eff;
  s.routed_rows = (int64_t)L.kc_max;
  s.routed_bytes_peak = (int64_t)routed_buffers * L.kc_max * c.H * 2;
  s.routed_bytes_bound = 2LL * c.k * L.c_eff * c.H * 2;
  s.inter_bytes_peak = (int64_t)inter_buffers * L.kc_max * c.I * 2;
  s.inter_bytes_bound = 3LL * c.k * L.c_eff * c.I * 2;
  s.workspace_bytes = (int64_t)ws_used;
  s.kernel_launches = launches;
  g_stats = s;
}

// A library-owned side stream per (host thread, device), with its fork/join events.  The router
// weight gradient of chunk i only reads inputs and per-chunk arrays that no later kernel of the
// backward pass writes, so it runs there, overlapping the next chunk's GEMMs.
struct SideStream {
  int dev = -1;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local std::deque<SideStream> g_side;   // indexed by device; created on first use, kept (stable addresses)

cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((int)g_side.size() <= dev) g_side.resize(dev + 1);
  SideStream& ss = g_side[dev];
  if (ss.dev != dev) {
    if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    ss.dev = dev;
  }
  *out = &ss;
  return cudaSuccess;
}

// CTA-pair GEMMs pay off when expert segments are long: with 256-row pair tiles the padding of an
// expert's last tile doubles, so short segments (a few hundred rows) run faster on single CTAs.
std::atomic<int> g_gemm_form{MOE_GEMM_AUTO};
bool use_pairs(int64_t rows, int E) {
  if (g_gemm_form == MOE_GEMM_SINGLE) return false;
  if (g_gemm_form == MOE_GEMM_PAIR) return true;
  return rows >= 512LL * E;
}

// GEMM work items are handed out dynamically (a work counter per GEMM); MOE_GEMM_STATIC builds the
// round-robin form instead.
inline int* gemm_counters(int* base) {
#ifdef MOE_GEMM_STATIC
  (void)base;
  return nullptr;
#else
  return base;
#endif
}

ChunkGemm chunk_gemm(const moe_config& c, const Layout& L, const PlanPtrs& p, int i, int* status, int* ctr) {
  ChunkGemm g;
  g.work_ctr = gemm_counters(ctr + (size_t)i * GEMM_CTR_SLOTS);
  g.late_wait = false;
  g.trigger_early = false;
  g.pair = use_pairs((int64_t)L.kc_max, c.E);
  const int n_i = (c.N - i + L.K - 1) / L.K;
  g.tiles = p.tiles + (size_t)i * L.T_max;
  g.tile_count = p.tile_count + i;
  g.tiles2 = p.tiles2 + (size_t)i * L.T2_max;
  g.tile2_count = p.tile2_count + i;
  g.active = p.active + (size_t)i * c.E;
  g.active_count = p.active_count + i;
  g.expert_off = p.expert_off + (size_t)i * (c.E + 1);
  g.row_route = p.row_route + (size_t)i * L.kc_max;
  g.rows = n_i * c.k;
  g.chunk = i;
  g.N = c.N;
  g.k = c.k;
  g.on_load = L.on_load;
  g.E = c.E;
  g.H = c.H;
  g.I = c.I;
  g.num_sms = num_sms();
  g.status = status;
  g.limit_ns = g_limit_ns;
  return g;
}

// ------------------------------------------------------------------ hop schedule
struct HopLayout {
  int P, cap, Tg, Tg2, Th, Th2, n_dact;
  bool on_load;
  // global plan (one chunk over all routes)
  size_t expert_off, row_route, row_of, tiles_g, tile_count_g, tiles2_g, tile2_count_g, active_g, active_count_g,
      first_touch, ft_zero;
  // per-hop plan arrays, one set per hop (all hops are planned in one launch)
  size_t h_tiles, h_tile_count, h_tiles2, h_tile2_count, h_active, h_active_count, h_expert_off, h_row_route,
      h_base, h_rows;
  size_t work_ctr;   // [P][GEMM_CTR_SLOTS]
  size_t plan_counts;  // multi-block global plan scratch
  int count_blocks;
  // forward (xp unused on load)
  size_t yacc, xp, op, act;
  // backward: b_xp holds Xp, then dXp; b_dyp holds dYp (both unused on load, where b_dxp holds dXp)
  size_t dxacc, dg_route, dlogit, b_xp, b_dyp, b_dxp, b_gate, b_up, b_gact, b_dgp, b_rdw;
  size_t fwd_total, bwd_total;
};

int hop_rows_worst(const moe_config& c, int P) {
  const int per = (c.E + P - 1) / P;
  return (int)std::min<int64_t>((int64_t)c.N * std::min(c.k, per), (int64_t)INT32_MAX / 2);
}

HopLayout make_hop_layout(const moe_config& c, int P, int cap) {
  HopLayout L = {};
  L.on_load = g_dispatch.load() == MOE_DISPATCH_ON_LOAD;
  L.P = P;
  L.cap = cap;
  const int64_t E = c.E, k = c.k, N = c.N, H = c.H, I = c.I, Nk = N * k;
  L.Tg = (int)((Nk + 127) / 128 + E);
  L.Tg2 = (int)((Nk + 255) / 256 + E);
  L.Th = (cap + 127) / 128 + c.E;
  L.Th2 = (cap + 255) / 256 + c.E;
  L.n_dact = dgate_partials(c.I);
  size_t o = align_up(sizeof(WsHeader));
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.expert_off = take((E + 1) * 4);
  L.row_route = take(Nk * 4);
  L.row_of = take(Nk * 4);
  L.tiles_g = take((size_t)L.Tg * 8);
  L.tile_count_g = take(4);
  L.tiles2_g = take((size_t)L.Tg2 * 8);
  L.tile2_count_g = take(4);
  L.active_g = take(E * 4);
  L.active_count_g = take(4);
  L.first_touch = take(E * 4);
  L.ft_zero = take(E * 4);
  L.h_tiles = take((size_t)P * L.Th * 8);
  L.h_tile_count = take((size_t)P * 4);
  L.h_tiles2 = take((size_t)P * L.Th2 * 8);
  L.h_tile2_count = take((size_t)P * 4);
  L.h_active = take((size_t)P * E * 4);
  L.h_active_count = take((size_t)P * 4);
  L.h_expert_off = take((size_t)P * (E + 1) * 4);
  L.h_row_route = take((size_t)P * cap * 4);
  L.h_base = take((size_t)P * 4);
  L.h_rows = take((size_t)P * 4);
  L.work_ctr = take((size_t)P * GEMM_CTR_SLOTS * 4);
  L.count_blocks = plan_count_blocks(Nk);
  L.plan_counts = take((size_t)L.count_blocks * E * 4);
  const size_t common = o;
  L.yacc = take(N * H * 4);
  if (!L.on_load) L.xp = take((size_t)cap * H * 2);
  L.op = take((size_t)cap * H * 2);
  L.act = take((size_t)cap * I * 2);
  L.fwd_total = o;
  o = common;
  L.dxacc = take(N * H * 4);
  L.dg_route = take(Nk * 4);
  L.dlogit = take(Nk * 4);
  if (!L.on_load) {
    L.b_xp = take((size_t)cap * H * 2);
    L.b_dyp = take((size_t)cap * H * 2);
    L.b_dxp = L.b_xp;
  } else {
    L.b_dxp = take((size_t)cap * H * 2);
  }
  L.b_gate = take((size_t)cap * I * 2);
  L.b_up = take((size_t)cap * I * 2);
  L.b_gact = take((size_t)cap * I * 2);
  L.b_dgp = take((size_t)cap * L.n_dact * 4);
  L.b_rdw = take((size_t)L.Tg * H * 4);
  L.bwd_total = o;
  return L;
}

// The global plan: the chunk plan with one chunk over all N*k routes.
PlanPtrs global_plan(const moe_config& c, const HopLayout& L, uint8_t* w) {
  PlanPtrs p;
  p.expert_off = reinterpret_cast<int*>(w + L.expert_off);
  p.row_route = reinterpret_cast<int*>(w + L.row_route);
  p.row_of = reinterpret_cast<int*>(w + L.row_of);
  p.tiles = reinterpret_cast<int2*>(w + L.tiles_g);
  p.tile_count = reinterpret_cast<int*>(w + L.tile_count_g);
  p.tiles2 = reinterpret_cast<int2*>(w + L.tiles2_g);
  p.tile2_count = reinterpret_cast<int*>(w + L.tile2_count_g);
  p.active = reinterpret_cast<int*>(w + L.active_g);
  p.active_count = reinterpret_cast<int*>(w + L.active_count_g);
  p.first_touch = reinterpret_cast<int*>(w + L.first_touch);
  p.block_counts = reinterpret_cast<int*>(w + L.plan_counts);
  p.count_blocks = L.count_blocks;
  p.N = c.N;
  p.E = c.E;
  p.k = c.k;
  p.K = 1;
  p.c_eff = c.N;
  p.kc_max = c.N * c.k;
  p.T_max = L.Tg;
  p.T2_max = L.Tg2;
  return p;
}

HopSets hop_sets(const moe_config& c, const HopLayout& L, uint8_t* w) {
  HopSets S;
  HopPtrs& h = S.h0;
  h.tiles = reinterpret_cast<int2*>(w + L.h_tiles);
  h.tile_count = reinterpret_cast<int*>(w + L.h_tile_count);
  h.tiles2 = reinterpret_cast<int2*>(w + L.h_tiles2);
  h.tile2_count = reinterpret_cast<int*>(w + L.h_tile2_count);
  h.active = reinterpret_cast<int*>(w + L.h_active);
  h.active_count = reinterpret_cast<int*>(w + L.h_active_count);
  h.expert_off = reinterpret_cast<int*>(w + L.h_expert_off);
  h.first_touch = reinterpret_cast<int*>(w + L.first_touch);
  h.row_route = reinterpret_cast<int*>(w + L.h_row_route);
  h.base = reinterpret_cast<int*>(w + L.h_base);
  h.rows = reinterpret_cast<int*>(w + L.h_rows);
  S.s_tiles = L.Th;
  S.s_tiles2 = L.Th2;
  S.s_active = c.E;
  S.s_expert_off = c.E + 1;
  S.s_row_route = L.cap;
  return S;
}

// The plan arrays of hop `hop`.
HopPtrs hop_ptrs(const moe_config& c, const HopLayout& L, uint8_t* w, int hop) {
  return hop_set(hop_sets(c, L, w), hop);
}

ChunkGemm hop_gemm(const moe_config& c, const HopLayout& L, const HopPtrs& h, int hop, int* status, int* ctr) {
  ChunkGemm g;
  g.work_ctr = gemm_counters(ctr + (size_t)hop * GEMM_CTR_SLOTS);
  g.late_wait = false;
  g.trigger_early = false;
  g.pair = use_pairs((int64_t)c.N * c.k, c.E);   // a hop holds all of its experts' routes
  g.tiles = h.tiles;
  g.tile_count = h.tile_count;
  g.tiles2 = h.tiles2;
  g.tile2_count = h.tile2_count;
  g.active = h.active;
  g.active_count = h.active_count;
  g.expert_off = h.expert_off;
  g.row_route = h.row_route;
  g.rows = L.cap;
  g.chunk = hop;
  g.N = c.N;
  g.k = c.k;
  g.on_load = L.on_load;
  g.E = c.E;
  g.H = c.H;
  g.I = c.I;
  g.num_sms = num_sms();
  g.status = status;
  g.limit_ns = g_limit_ns;
  return g;
}

int validate_hops(const moe_config* cfg, int P, int cap) {
  const int v = validate(cfg);
  if (v != MOE_OK) return v;
  if (P < 1 || P > cfg->E || cap < 1) return MOE_ERR_INVALID_ARG;
  if ((int64_t)cap > (int64_t)cfg->N * cfg->k && cfg->N > 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace

int record_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
int device_sm_count() { return num_sms(); }
int64_t wait_limit_ns() { return g_limit_ns; }
int timed_launch(int kind, const char* what, cudaStream_t s, const std::function<cudaError_t()>& f) {
  Launcher L{s};
  return L(kind, what, f);
}
std::atomic<int> g_chain_mode{MOE_CHAIN_LATE};
int launch_chain_mode() { return g_chain_mode.load(std::memory_order_relaxed); }

}  // namespace moe

using namespace moe;

extern "C" {

int moe_workspace_bytes(const moe_config* cfg, size_t* route_bytes, size_t* fwd_bytes, size_t* bwd_bytes) {
  const int v = validate(cfg);
  if (v != MOE_OK) return v;
  const Layout L = make_layout(*cfg);
  if (route_bytes) *route_bytes = L.route_total;
  if (fwd_bytes) *fwd_bytes = L.fwd_total;
  if (bwd_bytes) *bwd_bytes = L.bwd_total;
  return MOE_OK;
}

int moe_chunk_plan(const moe_config* cfg, int32_t* K, int32_t* c_eff) {
  const int v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!K || !c_eff) return MOE_ERR_INVALID_ARG;
  int k_, c_;
  chunk_plan(*cfg, &k_, &c_);
  *K = k_;
  *c_eff = c_;
  return MOE_OK;
}

int moe_route(const moe_config* cfg, const uint16_t* X, const float* Wr, const float* bias, int32_t* topk_idx,
              float* gates, void* ws, size_t ws_bytes, void* stream) {
  int v = validate(cfg);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.route_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (c.N > 0 && (!ok_ptr(X) || !ok_ptr(Wr) || !ok_ptr(topk_idx) || !ok_ptr(gates))) return MOE_ERR_INVALID_ARG;
  if (bias && !aligned16(bias)) return MOE_ERR_INVALID_ARG;
  Launcher run{static_cast<cudaStream_t>(stream)};
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  float* logits = reinterpret_cast<float*>(w + L.logits);
  if (c.N > 0) {
    if ((v = run(MOE_K_ROUTER_LOGITS, "router_logits",
                 [&] { return launch_router_logits(X, Wr, bias, logits, c.N, c.H, c.E, run.s); })))
      return v;
    if ((v = run(MOE_K_ROUTER_TOPK, "router_topk",
                 [&] { return launch_router_topk(logits, topk_idx, gates, c.N, c.E, c.k, status, run.s); })))
      return v;
  }
  set_stats(c, L, run.launches, L.route_total, 0, 0);
  return MOE_OK;
}

int moe_plan(const moe_config* cfg, const int32_t* topk_idx, int32_t* row_route, int32_t* row_of,
             int32_t* expert_off, void* ws, size_t ws_bytes, void* stream) {
  int v = validate(cfg);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.fwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (c.N > 0 && (!ok_ptr(topk_idx) || !ok_ptr(row_route) || !ok_ptr(row_of) || !ok_ptr(expert_off)))
    return MOE_ERR_INVALID_ARG;
  Launcher run{static_cast<cudaStream_t>(stream)};
  uint8_t* w = static_cast<uint8_t*>(ws);
  PlanPtrs p = plan_ptrs(c, L, w);
  p.row_route = row_route;
  p.row_of = row_of;
  p.expert_off = expert_off;
  if (c.N > 0) {
    if ((v = run(MOE_K_PLAN, "plan", [&] { return launch_plan(topk_idx, p, reinterpret_cast<int*>(w), run.s); })))
      return v;
  }
  set_stats(c, L, run.launches, L.fwd_total, 0, 0);
  return MOE_OK;
}

int moe_forward(const moe_config* cfg, const uint16_t* X, const int32_t* topk_idx, const float* gates,
                const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, uint16_t* Y, void* ws, size_t ws_bytes,
                void* stream) {
  int v = validate(cfg);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.fwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (c.N > 0 && (!ok_ptr(X) || !ok_ptr(topk_idx) || !ok_ptr(gates) || !ok_ptr(Wg) || !ok_ptr(Wu) ||
                  !ok_ptr(Wd) || !ok_ptr(Y)))
    return MOE_ERR_INVALID_ARG;
  Launcher run{static_cast<cudaStream_t>(stream)};
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  const PlanPtrs p = plan_ptrs(c, L, w);
  // Xp: the permuted buffer a gather kernel fills, or (on load) X itself, which the GEMM gathers from
  uint16_t* Xp = L.on_load ? const_cast<uint16_t*>(X) : reinterpret_cast<uint16_t*>(w + L.xp);
  uint16_t* Op = reinterpret_cast<uint16_t*>(w + L.op);
  uint16_t* act = reinterpret_cast<uint16_t*>(w + L.act);
  int* ctr = reinterpret_cast<int*>(w + L.work_ctr);
  if (c.N > 0) {
    const cudaError_t e = cudaMemsetAsync(ctr, 0, (size_t)L.K * GEMM_CTR_SLOTS * 4, run.s);
    if (e != cudaSuccess) return cuda_fail(e, "clear work counters");
    if ((v = run(MOE_K_PLAN, "plan", [&] { return launch_plan(topk_idx, p, status, run.s); }))) return v;
    // Stream order per chunk i: [gather(i)] gate/up(i) down(i) combine(i).  Xp, act and Op are each written
    // by one kernel and read by the next, so the gather of chunk i+1 (into Xp, last read by gate/up(i)) runs
    // beside down(i), and gate/up(i+1) (into act, last read by down(i)) runs beside combine(i) (which reads
    // Op); both wait for the kernel they overlap at their end.  A CTA-pair gate/up waits up front.  On load
    // there is no gather kernel: gate/up gathers its rows of X itself and Op is the one H-wide buffer.
    if (!L.on_load) {
      const ChunkGemm g0 = chunk_gemm(c, L, p, 0, status, ctr);
      if ((v = run(MOE_K_GATHER, "gather X",
                   [&] { return launch_gather(X, Xp, g0.row_route, g0.rows, c.H, c.k, run.s); })))
        return v;
    }
    for (int i = 0; i < L.K; ++i) {
      ChunkGemm g = chunk_gemm(c, L, p, i, status, ctr);
      const int n_i = g.rows / c.k;
      const bool gather_next = !L.on_load && i + 1 < L.K;
      g.late_wait = i > 0 && !g.pair;
      if ((v = run(MOE_K_GEMM_GATEUP, "gemm gate/up", [&] { return gemm_gateup_fwd(g, Xp, Wg, Wu, act, run.s); })))
        return v;
      g.late_wait = false;
      g.trigger_early = gather_next;
      if ((v = run(MOE_K_GEMM_DOWN, "gemm down", [&] { return gemm_down(g, act, Wd, Op, run.s); }))) return v;
      g.trigger_early = false;
      if (gather_next) {
        const ChunkGemm gn = chunk_gemm(c, L, p, i + 1, status, ctr);
        if ((v = run(MOE_K_GATHER, "gather X",
                     [&] { return launch_gather(X, Xp, gn.row_route, gn.rows, c.H, c.k, run.s, true); })))
          return v;
      }
      if ((v = run(MOE_K_COMBINE, "combine",
                   [&] { return launch_combine(Op, gates, p.row_of, Y, i, L.K, n_i, c.H, c.k, run.s); })))
        return v;
    }
  }
  set_stats(c, L, run.launches, L.fwd_total, L.on_load ? 1 : 2, 1);
  return MOE_OK;
}

int moe_backward(const moe_config* cfg, const uint16_t* X, const float* Wr, const int32_t* topk_idx,
                 const float* gates, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd, const uint16_t* dY,
                 uint16_t* dX, float* dWr, float* dWg, float* dWu, float* dWd, float* dgates, void* ws,
                 size_t ws_bytes, void* stream) {
  int v = validate(cfg);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  const Layout L = make_layout(c);
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.bwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!ok_ptr(dWr) || !ok_ptr(dWg) || !ok_ptr(dWu) || !ok_ptr(dWd)) return MOE_ERR_INVALID_ARG;
  if (c.N > 0 && (!ok_ptr(X) || !ok_ptr(Wr) || !ok_ptr(topk_idx) || !ok_ptr(gates) || !ok_ptr(Wg) ||
                  !ok_ptr(Wu) || !ok_ptr(Wd) || !ok_ptr(dY) || !ok_ptr(dX)))
    return MOE_ERR_INVALID_ARG;
  if (dgates && !aligned16(dgates)) return MOE_ERR_INVALID_ARG;
  Launcher run{static_cast<cudaStream_t>(stream)};
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  const PlanPtrs p = plan_ptrs(c, L, w);
  // Xp, dYp: the permuted buffers the gather kernels fill, or (on load) X and dY, which the GEMMs gather from
  uint16_t* Xp = L.on_load ? const_cast<uint16_t*>(X) : reinterpret_cast<uint16_t*>(w + L.b_xp);
  uint16_t* dYp = L.on_load ? const_cast<uint16_t*>(dY) : reinterpret_cast<uint16_t*>(w + L.b_dyp);
  uint16_t* dXp = reinterpret_cast<uint16_t*>(w + L.b_dyp);   // dX's output (over dYp when materialised)
  uint16_t* gate = reinterpret_cast<uint16_t*>(w + L.b_gate); // gate, then dGate
  uint16_t* up = reinterpret_cast<uint16_t*>(w + L.b_up);     // up, then dUp
  uint16_t* gact = reinterpret_cast<uint16_t*>(w + L.b_gact);
  float* dgp = reinterpret_cast<float*>(w + L.b_dgp);
  float* dlogit = reinterpret_cast<float*>(w + L.b_dlogit);
  float* dl_row = reinterpret_cast<float*>(w + L.b_dlrow);   // router-logit gradient of each permuted row
  const size_t IH = (size_t)c.I * c.H;
  if (c.N == 0) {
    cudaStream_t s = run.s;
    cudaError_t e = cudaMemsetAsync(dWg, 0, c.E * IH * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWu, 0, c.E * IH * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWd, 0, c.E * IH * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWr, 0, (size_t)c.E * c.H * 4, s);
    if (e != cudaSuccess) return cuda_fail(e, "memset");
    set_stats(c, L, 0, L.bwd_total, L.on_load ? 1 : 2, 3);
    return MOE_OK;
  }
  int* ctr = reinterpret_cast<int*>(w + L.work_ctr);
  {
    const cudaError_t e = cudaMemsetAsync(ctr, 0, (size_t)L.K * GEMM_CTR_SLOTS * 4, run.s);
    if (e != cudaSuccess) return cuda_fail(e, "clear work counters");
  }
  if ((v = run(MOE_K_PLAN, "plan", [&] { return launch_plan(topk_idx, p, status, run.s); }))) return v;
  if ((v = run(MOE_K_PLAN, "first touch", [&] { return launch_first_touch(p, run.s); }))) return v;
  SideStream* side = nullptr;
  {
    const cudaError_t e = side_stream(&side);
    if (e != cudaSuccess) return cuda_fail(e, "side stream");
  }
  Launcher aux{side->s};
  // Stream order (backward order of chunks; K-1 first):
  //   gather X(K-1) gather dY(K-1) gate/up(K-1) dActU(K-1) route grad(K-1) dWd dWg/dWu dX(K-1) gather X(K-2)
  //   unpermute(K-1) gate/up(K-2) gather dY(K-2) [router dW(K-1) forked] dActU(K-2) ...
  // route grad turns the dActU partials into dgates, dlogit and each row's dl, which the dX GEMM uses to add
  // the router-path term dl Wr[e] to dXp.  dX writes dXp over dYp (free once dWd has read it), so the next
  // chunk's X gather (into Xp, last read by dWg/dWu) runs beside dX, and the next chunk's gate/up recompute
  // (into gate/up, last read by dX) runs beside unpermute (which reads dXp); each of the two waits for the
  // kernel it overlaps at its end (a CTA-pair recompute waits up front).  The dY gather then waits for
  // unpermute.  On load there are no gather kernels (the GEMMs gather their rows of X and dY themselves)
  // and dXp is the one H-wide buffer.
  auto fork_router_dw = [&](int i) -> int {
    // the side stream waits for chunk i's dlogit, then adds the chunk into dWr
    const ChunkGemm gi = chunk_gemm(c, L, p, i, status, ctr);
    cudaError_t e = cudaEventRecord(side->fork, run.s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "fork side stream");
    return aux(MOE_K_ROUTER_DW, "router dW", [&] {
      return launch_router_dw(X, dlogit, gi.row_route, gi.tiles, gi.tile_count, L.T_max, gi.active,
                              gi.active_count, p.first_touch, reinterpret_cast<float*>(w + L.b_rdw), dWr, i, c.E,
                              c.H, c.k, aux.s);
    });
  };
  if (!L.on_load) {
    const ChunkGemm g0 = chunk_gemm(c, L, p, L.K - 1, status, ctr);
    if ((v = run(MOE_K_GATHER, "gather X",
                 [&] { return launch_gather(X, Xp, g0.row_route, g0.rows, c.H, c.k, run.s); })))
      return v;
  }
  for (int i = L.K - 1; i >= 0; --i) {
    ChunkGemm g = chunk_gemm(c, L, p, i, status, ctr);
    const int n_i = g.rows / c.k;
    const bool first = i == L.K - 1;
    // late beside unpermute(i+1), except in the CTA-pair form: no cluster kernel waits late
    g.late_wait = !first && !g.pair;
    if ((v = run(MOE_K_GEMM_GATEUP, "gemm gate/up recompute",
                 [&] { return gemm_gateup_bwd(g, Xp, Wg, Wu, gate, up, run.s); })))
      return v;
    g.late_wait = false;
    if (!L.on_load && (v = run(MOE_K_GATHER, "gather dY",
                               [&] { return launch_gather(dY, dYp, g.row_route, g.rows, c.H, c.k, run.s); })))
      return v;
    if (!first && (v = fork_router_dw(i + 1))) return v;
    if ((v = run(MOE_K_GEMM_DACT, "gemm dact", [&] { return gemm_dact(g, dYp, Wd, gates, gate, up, gact, dgp, run.s); })))
      return v;
    // the router backward of the chunk's routes (dgates, dlogit, and each row's dl for the dX GEMM)
    if ((v = run(MOE_K_ROUTE_GRAD, "route grad", [&] {
           return launch_route_grad(dgp, L.n_dact, gates, p.row_of, dgates, dlogit, dl_row, i, L.K, n_i, c.k, run.s);
         })))
      return v;
    // dWg/dWu (dGate, dUp and Xp in; dWg, dWu out) runs beside the tail of dWd (dYp and gact in)
    g.trigger_early = true;
    if ((v = run(MOE_K_GEMM_DW, "gemm dWd", [&] { return gemm_dwd(g, dYp, gact, p.first_touch, dWd, run.s); })))
      return v;
    g.trigger_early = false;
    g.late_wait = true;
    if ((v = run(MOE_K_GEMM_DW, "gemm dWg/dWu",
                 [&] { return gemm_dwgu(g, gate, up, Xp, p.first_touch, dWg, dWu, run.s); })))
      return v;
    g.late_wait = false;
    const bool gather_next = !L.on_load && i > 0;
    g.trigger_early = gather_next;
    if ((v = run(MOE_K_GEMM_DX, "gemm dX",
                 [&] { return gemm_dx(g, gate, up, Wg, Wu, dl_row, Wr, dXp, run.s); })))
      return v;
    g.trigger_early = false;
    if (gather_next) {
      const ChunkGemm gn = chunk_gemm(c, L, p, i - 1, status, ctr);
      if ((v = run(MOE_K_GATHER, "gather X",
                   [&] { return launch_gather(X, Xp, gn.row_route, gn.rows, c.H, c.k, run.s, true); })))
        return v;
    }
    if ((v = run(MOE_K_UNPERMUTE, "unpermute", [&] {
           return launch_unpermute(dXp, p.row_of, dX, i, L.K, n_i, c.H, c.k, run.s);
         })))
      return v;
  }
  if ((v = fork_router_dw(0))) return v;
  {  // join: the caller's stream sees every router-dW update before the call's last kernel
    cudaError_t e = cudaEventRecord(side->join, side->s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(run.s, side->join, 0);
    if (e != cudaSuccess) return cuda_fail(e, "join side stream");
  }
  if ((v = run(MOE_K_ZERO, "zero untouched",
               [&] { return launch_zero_untouched(p.first_touch, dWg, dWu, dWd, dWr, c.E, c.H, c.I, run.s); })))
    return v;
  set_stats(c, L, run.launches + aux.launches, L.bwd_total, L.on_load ? 1 : 2, 3);
  return MOE_OK;
}

int moe_hop_rows_worst_case(const moe_config* cfg, int32_t P, int32_t* rows) {
  const int v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!rows || P < 1 || P > cfg->E) return MOE_ERR_INVALID_ARG;
  *rows = std::max(1, hop_rows_worst(*cfg, P));
  return MOE_OK;
}

int moe_hops_workspace_bytes(const moe_config* cfg, int32_t P, int32_t max_hop_rows, size_t* fwd_bytes,
                             size_t* bwd_bytes) {
  const int v = validate_hops(cfg, P, max_hop_rows);
  if (v != MOE_OK) return v;
  const HopLayout L = make_hop_layout(*cfg, P, max_hop_rows);
  if (fwd_bytes) *fwd_bytes = L.fwd_total;
  if (bwd_bytes) *bwd_bytes = L.bwd_total;
  return MOE_OK;
}

int moe_forward_hops(const moe_config* cfg, int32_t P, int32_t max_hop_rows, const uint16_t* X,
                     const int32_t* topk_idx, const float* gates, const uint16_t* Wg, const uint16_t* Wu,
                     const uint16_t* Wd, uint16_t* Y, void* ws, size_t ws_bytes, void* stream) {
  int v = validate_hops(cfg, P, max_hop_rows);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  const HopLayout L = make_hop_layout(c, P, max_hop_rows);
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.fwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (c.N > 0 && (!ok_ptr(X) || !ok_ptr(topk_idx) || !ok_ptr(gates) || !ok_ptr(Wg) || !ok_ptr(Wu) ||
                  !ok_ptr(Wd) || !ok_ptr(Y)))
    return MOE_ERR_INVALID_ARG;
  Launcher run{static_cast<cudaStream_t>(stream)};
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  const PlanPtrs pg = global_plan(c, L, w);
  float* Yacc = reinterpret_cast<float*>(w + L.yacc);
  uint16_t* Xp = L.on_load ? const_cast<uint16_t*>(X) : reinterpret_cast<uint16_t*>(w + L.xp);
  uint16_t* Op = reinterpret_cast<uint16_t*>(w + L.op);
  uint16_t* act = reinterpret_cast<uint16_t*>(w + L.act);
  if (c.N > 0) {
    cudaError_t e = cudaMemsetAsync(Yacc, 0, (size_t)c.N * c.H * 4, run.s);
    if (e == cudaSuccess) e = cudaMemsetAsync(w + L.work_ctr, 0, (size_t)P * GEMM_CTR_SLOTS * 4, run.s);
    if (e != cudaSuccess) return cuda_fail(e, "clear Y accumulator");
    if ((v = run(MOE_K_PLAN, "plan", [&] { return launch_plan(topk_idx, pg, status, run.s); }))) return v;
    auto e_lo = [&](int h) { return (int)((int64_t)h * c.E / P); };
    if ((v = run(MOE_K_HOP_PLAN, "hop plans", [&] {
           return launch_hop_plan_all(pg.expert_off, pg.row_route, hop_sets(c, L, w), P, c.E, L.cap, status, run.s);
         })))
      return v;
    // Stream order: hop plans, [gather(0)], then per hop [gate/up(h) down(h) gather(h+1) combine(h)].
    // Every hop has its own plan arrays and Op its own buffer, so gather(h+1) (into Xp, last read by
    // gate/up(h)) runs beside down(h) and gate/up(h+1) (into act, last read by down(h)) beside combine(h);
    // each waits for the kernel it overlaps at its end, except that a CTA-pair gate/up waits up front.
    // On load the gate/up GEMM gathers the hop's rows of X itself.
    if (!L.on_load) {
      const HopPtrs h0 = hop_ptrs(c, L, w, 0);
      if ((v = run(MOE_K_GATHER, "gather X",
                   [&] { return launch_gather_dev(X, Xp, h0.row_route, h0.rows, L.cap, c.H, c.k, run.s); })))
        return v;
    }
    for (int h = 0; h < P; ++h) {
      const HopPtrs hp = hop_ptrs(c, L, w, h);
      const int e0 = e_lo(h), e1 = e_lo(h + 1);
      const bool gather_next = !L.on_load && h + 1 < P;
      ChunkGemm g = hop_gemm(c, L, hp, h, status, reinterpret_cast<int*>(w + L.work_ctr));
      g.late_wait = h > 0 && !g.pair;
      if ((v = run(MOE_K_GEMM_GATEUP, "gemm gate/up", [&] { return gemm_gateup_fwd(g, Xp, Wg, Wu, act, run.s); })))
        return v;
      g.late_wait = false;
      g.trigger_early = gather_next;
      if ((v = run(MOE_K_GEMM_DOWN, "gemm down", [&] { return gemm_down(g, act, Wd, Op, run.s); }))) return v;
      g.trigger_early = false;
      if (gather_next) {
        const HopPtrs hn = hop_ptrs(c, L, w, h + 1);
        if ((v = run(MOE_K_GATHER, "gather X", [&] {
               return launch_gather_dev(X, Xp, hn.row_route, hn.rows, L.cap, c.H, c.k, run.s, true);
             })))
          return v;
      }
      if ((v = run(MOE_K_COMBINE, "combine", [&] {
             return launch_combine_hop(Op, gates, pg.row_of, topk_idx, hp.base, hp.rows, e0, e1, Yacc, c.N, c.H,
                                       c.k, run.s);
           })))
        return v;
    }
    if ((v = run(MOE_K_FINAL, "finalize Y",
                 [&] { return launch_to_bf16(Yacc, Y, (int64_t)c.N * c.H, run.s); })))
      return v;
  }
  moe_stats st = {};
  st.K = P;
  st.c_eff = 0;
  st.routed_rows = L.cap;
  st.routed_bytes_peak = (L.on_load ? 1LL : 2LL) * L.cap * c.H * 2;   // Op, and Xp unless gathered on load
  st.routed_bytes_bound = 2LL * L.cap * c.H * 2;
  st.inter_bytes_peak = (int64_t)L.cap * c.I * 2;
  st.inter_bytes_bound = 3LL * L.cap * c.I * 2;
  st.workspace_bytes = (int64_t)L.fwd_total;
  st.kernel_launches = run.launches;
  g_stats = st;
  return MOE_OK;
}

int moe_backward_hops(const moe_config* cfg, int32_t P, int32_t max_hop_rows, const uint16_t* X, const float* Wr,
                      const int32_t* topk_idx, const float* gates, const uint16_t* Wg, const uint16_t* Wu,
                      const uint16_t* Wd, const uint16_t* dY, uint16_t* dX, float* dWr, float* dWg, float* dWu,
                      float* dWd, float* dgates, void* ws, size_t ws_bytes, void* stream) {
  int v = validate_hops(cfg, P, max_hop_rows);
  if (v != MOE_OK) return v;
  const moe_config& c = *cfg;
  const HopLayout L = make_hop_layout(c, P, max_hop_rows);
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < L.bwd_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!ok_ptr(dWr) || !ok_ptr(dWg) || !ok_ptr(dWu) || !ok_ptr(dWd)) return MOE_ERR_INVALID_ARG;
  if (c.N > 0 && (!ok_ptr(X) || !ok_ptr(Wr) || !ok_ptr(topk_idx) || !ok_ptr(gates) || !ok_ptr(Wg) ||
                  !ok_ptr(Wu) || !ok_ptr(Wd) || !ok_ptr(dY) || !ok_ptr(dX)))
    return MOE_ERR_INVALID_ARG;
  if (dgates && !aligned16(dgates)) return MOE_ERR_INVALID_ARG;
  Launcher run{static_cast<cudaStream_t>(stream)};
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);
  const size_t IH = (size_t)c.I * c.H;
  if (c.N == 0) {
    cudaError_t e = cudaMemsetAsync(dWg, 0, c.E * IH * 4, run.s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWu, 0, c.E * IH * 4, run.s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWd, 0, c.E * IH * 4, run.s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWr, 0, (size_t)c.E * c.H * 4, run.s);
    if (e != cudaSuccess) return cuda_fail(e, "memset");
    return MOE_OK;
  }
  const PlanPtrs pg = global_plan(c, L, w);
  float* dXacc = reinterpret_cast<float*>(w + L.dxacc);
  float* dg_route = reinterpret_cast<float*>(w + L.dg_route);
  float* dlogit = reinterpret_cast<float*>(w + L.dlogit);
  uint16_t* Xp = L.on_load ? const_cast<uint16_t*>(X) : reinterpret_cast<uint16_t*>(w + L.b_xp);
  uint16_t* dYp = L.on_load ? const_cast<uint16_t*>(dY) : reinterpret_cast<uint16_t*>(w + L.b_dyp);
  uint16_t* dXp = reinterpret_cast<uint16_t*>(w + L.b_dxp);   // over Xp when materialised
  uint16_t* gate = reinterpret_cast<uint16_t*>(w + L.b_gate);
  uint16_t* up = reinterpret_cast<uint16_t*>(w + L.b_up);
  uint16_t* gact = reinterpret_cast<uint16_t*>(w + L.b_gact);
  float* dgp = reinterpret_cast<float*>(w + L.b_dgp);
  int* ft_zero = reinterpret_cast<int*>(w + L.ft_zero);
  cudaError_t e = cudaMemsetAsync(dXacc, 0, (size_t)c.N * c.H * 4, run.s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ft_zero, 0, (size_t)c.E * 4, run.s);
  if (e == cudaSuccess) e = cudaMemsetAsync(w + L.work_ctr, 0, (size_t)P * GEMM_CTR_SLOTS * 4, run.s);
  if (e != cudaSuccess) return cuda_fail(e, "clear accumulators");
  if ((v = run(MOE_K_PLAN, "plan", [&] { return launch_plan(topk_idx, pg, status, run.s); }))) return v;
  auto e_lo = [&](int h) { return (int)((int64_t)h * c.E / P); };
  if ((v = run(MOE_K_HOP_PLAN, "hop plans", [&] {
         return launch_hop_plan_all(pg.expert_off, pg.row_route, hop_sets(c, L, w), P, c.E, L.cap, status, run.s);
       })))
    return v;
  // Stream order per hop h (P-1 .. 0): [gather X(h) gather dY(h)] gate/up(h) dActU(h) dWd(h) dWg/dWu(h)
  // dX(h) unpermute(h), with dWg/dWu beside the tail of dWd.  Every other kernel waits for its predecessor
  // up front: with the next hop's gathers and recompute chained beside dX and unpermute (a late-waiting
  // CTA-pair recompute followed by a gather that fits beside it), the backward of the full-size many
  // (Zipf 1.2) workload did not finish, while the same kernels in stream order did.  On load the GEMMs
  // gather the hop's rows of X and dY themselves.
  for (int h = P - 1; h >= 0; --h) {
    const HopPtrs hp = hop_ptrs(c, L, w, h);
    const int e0 = e_lo(h), e1 = e_lo(h + 1);
    ChunkGemm g = hop_gemm(c, L, hp, h, status, reinterpret_cast<int*>(w + L.work_ctr));
    if (!L.on_load) {
      if ((v = run(MOE_K_GATHER, "gather X",
                   [&] { return launch_gather_dev(X, Xp, hp.row_route, hp.rows, L.cap, c.H, c.k, run.s); })))
        return v;
      if ((v = run(MOE_K_GATHER, "gather dY",
                   [&] { return launch_gather_dev(dY, dYp, hp.row_route, hp.rows, L.cap, c.H, c.k, run.s); })))
        return v;
    }
    if ((v = run(MOE_K_GEMM_GATEUP, "gemm gate/up recompute",
                 [&] { return gemm_gateup_bwd(g, Xp, Wg, Wu, gate, up, run.s); })))
      return v;
    if ((v = run(MOE_K_GEMM_DACT, "gemm dact", [&] { return gemm_dact(g, dYp, Wd, gates, gate, up, gact, dgp, run.s); })))
      return v;
    // dWg/dWu (dGate, dUp and Xp in; dWg, dWu out) runs beside the tail of dWd (dYp and gact in)
    g.trigger_early = true;
    if ((v = run(MOE_K_GEMM_DW, "gemm dWd", [&] { return gemm_dwd(g, dYp, gact, hp.first_touch, dWd, run.s); })))
      return v;
    g.trigger_early = false;
    g.late_wait = true;
    if ((v = run(MOE_K_GEMM_DW, "gemm dWg/dWu",
                 [&] { return gemm_dwgu(g, gate, up, Xp, hp.first_touch, dWg, dWu, run.s); })))
      return v;
    g.late_wait = false;
    if ((v = run(MOE_K_GEMM_DX, "gemm dX",
                 [&] { return gemm_dx(g, gate, up, Wg, Wu, nullptr, nullptr, dXp, run.s); })))
      return v;
    if ((v = run(MOE_K_UNPERMUTE, "unpermute", [&] {
           return launch_unpermute_hop(dXp, dgp, L.n_dact, pg.row_of, topk_idx, hp.base, hp.rows, e0, e1, dXacc,
                                       dg_route, c.N, c.H, c.k, run.s);
         })))
      return v;
  }
  if ((v = run(MOE_K_FINAL, "router backward", [&] {
         return launch_router_final(dXacc, dg_route, gates, topk_idx, Wr, dX, dgates, dlogit, c.N, c.H, c.k, c.E,
                                    run.s);
       })))
    return v;
  if ((v = run(MOE_K_ROUTER_DW, "router dW", [&] {
         return launch_router_dw(X, dlogit, pg.row_route, pg.tiles, pg.tile_count, L.Tg, pg.active,
                                 pg.active_count, ft_zero, reinterpret_cast<float*>(w + L.b_rdw), dWr, 0, c.E, c.H,
                                 c.k, run.s);
       })))
    return v;
  if ((v = run(MOE_K_ZERO, "zero untouched",
               [&] {
                 return launch_zero_untouched(reinterpret_cast<int*>(w + L.first_touch), dWg, dWu, dWd, dWr, c.E, c.H,
                                              c.I, run.s);
               })))
    return v;
  moe_stats st = {};
  st.K = P;
  st.routed_rows = L.cap;
  st.routed_bytes_peak = (L.on_load ? 1LL : 2LL) * L.cap * c.H * 2;   // Xp/dXp and dYp, or dXp alone on load
  st.routed_bytes_bound = 2LL * L.cap * c.H * 2;
  st.inter_bytes_peak = 3LL * L.cap * c.I * 2;
  st.inter_bytes_bound = 3LL * L.cap * c.I * 2;
  st.workspace_bytes = (int64_t)L.bwd_total;
  st.kernel_launches = run.launches;
  g_stats = st;
  return MOE_OK;
}

int moe_check_status(void* ws, void* stream) {
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int h[2] = {0, 0};
  e = cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  if (h[0] != 0) {
    char buf[96];
    snprintf(buf, sizeof(buf), "device status %d at site %d", h[0], h[1]);
    g_err = buf;
    e = cudaMemset(ws, 0, sizeof(h));
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
  }
  return h[0];
}

int moe_set_wait_limit_ns(int64_t ns) {
  g_limit_ns = ns > 0 ? ns : kDefaultLimitNs;
  return MOE_OK;
}

int moe_set_launch_chaining(int mode) {
  if (mode != MOE_CHAIN_NONE && mode != MOE_CHAIN_EARLY && mode != MOE_CHAIN_LATE) return MOE_ERR_INVALID_ARG;
  moe::g_chain_mode.store(mode);
  return MOE_OK;
}

int moe_set_dispatch(int mode) {
  if (mode != MOE_DISPATCH_GATHER && mode != MOE_DISPATCH_ON_LOAD) return MOE_ERR_INVALID_ARG;
  g_dispatch.store(mode);
  return MOE_OK;
}

int moe_set_gemm_form(int form) {
  if (form != MOE_GEMM_AUTO && form != MOE_GEMM_SINGLE && form != MOE_GEMM_PAIR) return MOE_ERR_INVALID_ARG;
  g_gemm_form = form;
  return MOE_OK;
}

int moe_last_stats(moe_stats* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = g_stats;
  return MOE_OK;
}

const char* moe_strerror(int code) {
  static thread_local std::string msg;
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (NULL or misaligned pointer, or negative size)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (H, I multiples of 64; E <= 1024; k <= min(E, 32))";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_CUDA: msg = "CUDA error: " + g_err; return msg.c_str();
    case MOE_ERR_TIMEOUT: msg = "device-side wait ran past its limit; " + g_err; return msg.c_str();
    case MOE_ERR_DEVICE_CHECK: msg = "device-side index check failed; " + g_err; return msg.c_str();
    case MOE_ERR_NOT_BUILT: return "the library was built without this diagnostic";
    default: return "unknown error code";
  }
}

int moe_profile_enable(int on) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  g_prof_on = on != 0;
  return MOE_OK;
}

int moe_profile_reset(void) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto& r : g_prof) {
    cudaEventSynchronize(r.b);
    g_free_events.push_back(r.a);
    g_free_events.push_back(r.b);
  }
  g_prof.clear();
  for (int i = 0; i < MOE_K_COUNT; ++i) {
    g_prof_launches[i] = 0;
    g_prof_ms[i] = 0.0;
  }
  return MOE_OK;
}

int moe_profile_read(int32_t* launches, double* total_ms, const char** names) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto& r : g_prof) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return cuda_fail(e, "event synchronize");
    float ms = 0.0f;
    e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) return cuda_fail(e, "event elapsed");
    g_prof_launches[r.kind] += 1;
    g_prof_ms[r.kind] += ms;
    g_free_events.push_back(r.a);
    g_free_events.push_back(r.b);
  }
  g_prof.clear();
  for (int i = 0; i < MOE_K_COUNT; ++i) {
    if (launches) launches[i] = g_prof_launches[i];
    if (total_ms) total_ms[i] = g_prof_ms[i];
    if (names) names[i] = kKernelNames[i];
  }
  return MOE_OK;
}

int moe_diag_gemm_wait_stats(uint64_t* counters, int reset) {
#ifdef MOE_GEMM_WAIT_STATS
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const size_t bytes = (size_t)MOE_GEMM_WAIT_CLASSES * MOE_GEMM_WAIT_FIELDS * sizeof(unsigned long long);
  unsigned long long* buf = g_wait_stats.load();
  cudaError_t e;
  if (buf == nullptr) {
    if ((e = cudaMalloc(&buf, bytes)) != cudaSuccess) return cuda_fail(e, "wait-stats buffer");
    if ((e = cudaMemset(buf, 0, bytes)) != cudaSuccess) return cuda_fail(e, "wait-stats buffer");
    g_wait_stats.store(buf);
  }
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "wait-stats sync");
  if (counters && (e = cudaMemcpy(counters, buf, bytes, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "wait-stats read");
  if (reset && (e = cudaMemset(buf, 0, bytes)) != cudaSuccess) return cuda_fail(e, "wait-stats reset");
  return MOE_OK;
#else
  (void)counters;
  (void)reset;
  return MOE_ERR_NOT_BUILT;
#endif
}

int moe_diag_wait_timeout(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream) {
  if (!ok_ptr(ws) || ws_bytes < sizeof(WsHeader) || limit_ns <= 0) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_diag_wait(static_cast<int*>(ws), limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diag wait");
  return MOE_OK;
}

}  // extern "C"
