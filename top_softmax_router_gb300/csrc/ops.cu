// Router, permutation and data-movement kernels of the MoE block.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ===========================================================================
// Router logits (RelayMoE summary 2.1; workload text: logits = X.W_r + bias).
// Each thread owns an 8 x 4 block of (token, expert) logits and walks h in
// increasing order with one fused multiply-add per step, starting from 0, then
// adds the bias once: the same fp32 chain for every (t, e), whatever the tile.
// ===========================================================================
constexpr int RT_T = 128, RT_E = 64, RT_H = 32;   // block tile: tokens x experts; h slice
constexpr int RT_PAD = 4;                          // shared-memory row padding (floats)

// Each thread owns 8 tokens (two groups of 4: ty*4.. and 64+ty*4..) x 4 experts (tx*4..) of the block's
// 128 x 64 tile, so one h step is three 16-byte shared-memory loads for 32 fused multiply-adds.
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ X,
                                                            const float* __restrict__ Wr,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int N, int H, int E) {
  __shared__ __align__(16) float xs[RT_H][RT_T + RT_PAD];
  __shared__ __align__(16) float ws[RT_H][RT_E + RT_PAD];
  const int t0 = blockIdx.x * RT_T, e0 = blockIdx.y * RT_E;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads
  float acc[8][4];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;

  // The next 32-wide slice of X and Wr is loaded into registers while the current one is multiplied out
  // of shared memory, so the global loads overlap the FMA chain.  X: thread -> (token tid % 128, h half
  // tid / 128: 16 values); Wr: thread -> (expert tid % 64, h quarter tid / 64: 8 values).  Consecutive
  // lanes take consecutive tokens / experts, so the transposed shared-memory stores are conflict-free.
  const int lt = threadIdx.x & (RT_T - 1), lh = (threadIdx.x >> 7) * 16;
  const int le = threadIdx.x & (RT_E - 1), lq = (threadIdx.x >> 6) * 8;
  const bool x_ok = t0 + lt < N, w_ok = e0 + le < E;
  const uint16_t* xrow = X + (int64_t)(t0 + lt) * H + lh;
  const float* wrow = Wr + (int64_t)(e0 + le) * H + lq;
  uint4 xa_n = make_uint4(0, 0, 0, 0), xb_n = xa_n;
  float4 wa_n = make_float4(0, 0, 0, 0), wb_n = wa_n;
  auto load_slice = [&](int h0) {
    if (x_ok) {
      xa_n = *reinterpret_cast<const uint4*>(xrow + h0);
      xb_n = *reinterpret_cast<const uint4*>(xrow + h0 + 8);
    }
    if (w_ok) {
      wa_n = *reinterpret_cast<const float4*>(wrow + h0);
      wb_n = *reinterpret_cast<const float4*>(wrow + h0 + 4);
    }
  };
  auto store_slice = [&]() {
    const uint32_t xv[8] = {xa_n.x, xa_n.y, xa_n.z, xa_n.w, xb_n.x, xb_n.y, xb_n.z, xb_n.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      xs[lh + 2 * i][lt] = bf16_lo(xv[i]);
      xs[lh + 2 * i + 1][lt] = bf16_hi(xv[i]);
    }
    ws[lq + 0][le] = wa_n.x; ws[lq + 1][le] = wa_n.y; ws[lq + 2][le] = wa_n.z; ws[lq + 3][le] = wa_n.w;
    ws[lq + 4][le] = wb_n.x; ws[lq + 5][le] = wb_n.y; ws[lq + 6][le] = wb_n.z; ws[lq + 7][le] = wb_n.w;
  };
  load_slice(0);
  store_slice();
  __syncthreads();
  for (int h0 = 0; h0 < H; h0 += RT_H) {
    const bool next = h0 + RT_H < H;
    if (next) load_slice(h0 + RT_H);
#pragma unroll 4
    for (int h = 0; h < RT_H; ++h) {
      const float4 xa = *reinterpret_cast<const float4*>(&xs[h][ty * 4]);
      const float4 xb = *reinterpret_cast<const float4*>(&xs[h][64 + ty * 4]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[h][tx * 4]);
      const float xr[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const float wr[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = __fmaf_rn(xr[a], wr[b], acc[a][b]);
    }
    __syncthreads();
    if (next) {
      store_slice();
      __syncthreads();
    }
  }
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int t = t0 + (a < 4 ? ty * 4 + a : 64 + ty * 4 + a - 4);
    if (t >= N) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + tx * 4 + b;
      if (e < E) logits[(int64_t)t * E + e] = bias ? __fadd_rn(acc[a][b], bias[e]) : acc[a][b];
    }
  }
}

cudaError_t launch_router_logits(const uint16_t* X, const float* Wr, const float* bias, float* logits, int N,
                                 int H, int E, cudaStream_t s) {
  dim3 grid((N + RT_T - 1) / RT_T, (E + RT_E - 1) / RT_E);
  router_logits_kernel<<<grid, 256, 0, s>>>(X, Wr, bias, logits, N, H, E);
  return cudaGetLastError();
}

// ===========================================================================
// Top-k + gates: one warp per token.  k rounds of a warp argmax (larger logit
// wins, equal logits go to the lower expert id); gates are the softmax of the
// selected logits, g_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), which equals
// "softmax over all experts, renormalised over the top-k".
// ===========================================================================
// PER = candidate slots per lane (a power of two >= ceil(E / 32)): lane holds experts lane, lane+32, ...
template <int PER>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits,
                                                          int32_t* __restrict__ idx, float* __restrict__ gates,
                                                          int N, int E, int k, int* status) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= N) return;
  const float* l = logits + (int64_t)t * E;
  float v[PER];
  uint32_t taken = 0;
  constexpr int per = PER;
#pragma unroll
  for (int q = 0; q < PER; ++q) {
    const int e = q * 32 + lane;
    v[q] = e < E ? l[e] : 0.0f;
  }
  float sel_l = 0.0f, l0 = 0.0f;
  int sel_e = 0;
  for (int j = 0; j < k; ++j) {
    float best = 0.0f;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int e = q * 32 + lane;
      if (q < per && e < E && !((taken >> q) & 1u)) {
        if (be == 0x7FFFFFFF || v[q] > best) { best = v[q]; be = e; }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      const bool take = (oe != 0x7FFFFFFF) &&
                        (be == 0x7FFFFFFF || ob > best || (ob == best && oe < be));
      if (take) { best = ob; be = oe; }
    }
    if (be == 0x7FFFFFFF) { report(status, MOE_ERR_DEVICE_CHECK, 201); be = 0; }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (j == 0) l0 = best;
    if (lane == j) { sel_l = best; sel_e = be; }
  }
  // gates over the k selected logits, summed in slot order
  const float ex = (lane < k) ? expf(sel_l - l0) : 0.0f;
  float sum = 0.0f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
  if (lane < k) {
    idx[(int64_t)t * k + lane] = sel_e;
    gates[(int64_t)t * k + lane] = ex / sum;
  }
}

cudaError_t launch_router_topk(const float* logits, int32_t* idx, float* gates, int N, int E, int k, int* status,
                               cudaStream_t s) {
  const dim3 grid((N + 7) / 8), block(256);
  const int per = (E + 31) / 32;
  if (per <= 1) return launch_pdl(router_topk_kernel<1>, grid, block, 0, s, logits, idx, gates, N, E, k, status);
  if (per <= 2) return launch_pdl(router_topk_kernel<2>, grid, block, 0, s, logits, idx, gates, N, E, k, status);
  if (per <= 4) return launch_pdl(router_topk_kernel<4>, grid, block, 0, s, logits, idx, gates, N, E, k, status);
  if (per <= 8) return launch_pdl(router_topk_kernel<8>, grid, block, 0, s, logits, idx, gates, N, E, k, status);
  if (per <= 16) return launch_pdl(router_topk_kernel<16>, grid, block, 0, s, logits, idx, gates, N, E, k, status);
  return launch_pdl(router_topk_kernel<32>, grid, block, 0, s, logits, idx, gates, N, E, k, status);
}

// ===========================================================================
// Chunk permutation: stable counting sort of chunk i's routes by expert
// (RelayMoE summary 2.1; "bounded-streaming" summary, Methodology 1: strided
// membership, chunk i holds tokens i, i+K, ...).  One 1024-thread block per
// chunk.  Each warp owns a contiguous run of the chunk's routes (in (local
// token, slot) order); pass 1 counts per (warp, expert), a scan turns the
// counts into per-(warp, expert) base rows, pass 2 hands out rows in order, so
// rows within an expert ascend by token.  Also writes the GEMM tile list
// (128-row tiles of one expert) and the list of experts with rows.
// ===========================================================================
constexpr int PLAN_THREADS = 1024;
constexpr int GEMM_TILE_M = 128;

__global__ void __launch_bounds__(PLAN_THREADS, 1) plan_kernel(const int32_t* __restrict__ topk_idx, PlanPtrs p,
                                                               int* status) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  extern __shared__ int sm[];
  int* base = sm;                       // [32][E]
  int* scratch = sm + 32 * p.E;         // 33
  const int i = blockIdx.x;
  const int K = p.K, k = p.k, E = p.E;
  const int n_i = (p.N - i + K - 1) / K;
  const int kc = n_i * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int x = threadIdx.x; x < 32 * E; x += PLAN_THREADS) base[x] = 0;
  __syncthreads();

  const int seg = (((kc + 31) / 32) + 31) / 32 * 32;  // routes per warp, multiple of 32
  const int q_begin = warp * seg;
  const int q_end = min(kc, q_begin + seg);
  bool bad = false;
  // pass 1: per-(warp, expert) counts
  for (int q0 = q_begin; q0 < q_end; q0 += 32) {
    const int q = q0 + lane;
    int e = -1;
    if (q < q_end) {
      const int l = q / k, j = q - l * k;
      const int64_t gid = (int64_t)(i + (int64_t)K * l) * k + j;
      e = topk_idx[gid];
      if (e < 0 || e >= E) { bad = true; e = 0; }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) base[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (bad) report(status, MOE_ERR_DEVICE_CHECK, 301);
  __syncthreads();

  // per-expert totals; per-warp exclusive prefix within each expert
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    for (int w = 0; w < 32; ++w) {
      const int c = base[w * E + e];
      base[w * E + e] = cnt;
      cnt += c;
    }
  }
  __syncthreads();
  int tot;
  const int off = block_exclusive_scan(e < E ? cnt : 0, scratch, &tot);
  const int ntile = (cnt + GEMM_TILE_M - 1) / GEMM_TILE_M;
  int tile_total;
  const int toff = block_exclusive_scan(e < E ? ntile : 0, scratch, &tile_total);
  int act_total;
  const int aoff = block_exclusive_scan((e < E && cnt > 0) ? 1 : 0, scratch, &act_total);
  const int npair = (cnt + 2 * GEMM_TILE_M - 1) / (2 * GEMM_TILE_M);
  int pair_total;
  const int poff = block_exclusive_scan(e < E ? npair : 0, scratch, &pair_total);
  if (e < E) {
    for (int w = 0; w < 32; ++w) base[w * E + e] += off;
    p.expert_off[(int64_t)i * (E + 1) + e] = off;
    for (int m = 0; m < ntile; ++m) {
      const int rows = min(GEMM_TILE_M, cnt - m * GEMM_TILE_M);
      p.tiles[(int64_t)i * p.T_max + toff + m] = make_int2(off + m * GEMM_TILE_M, e | (rows << 16));
    }
    for (int m = 0; m < npair; ++m) {
      const int rows = min(2 * GEMM_TILE_M, cnt - m * 2 * GEMM_TILE_M);
      p.tiles2[(int64_t)i * p.T2_max + poff + m] = make_int2(off + m * 2 * GEMM_TILE_M, e | (rows << 16));
    }
    if (cnt > 0) p.active[(int64_t)i * E + aoff] = e;
  }
  if (threadIdx.x == 0) {
    p.expert_off[(int64_t)i * (E + 1) + E] = kc;
    p.tile_count[i] = tile_total;
    p.tile2_count[i] = pair_total;
    p.active_count[i] = act_total;
  }
  __syncthreads();

  // pass 2: stable row assignment
  const uint32_t lt_mask = (1u << lane) - 1u;
  int* rr = p.row_route + (int64_t)i * p.kc_max;
  for (int q0 = q_begin; q0 < q_end; q0 += 32) {
    const int q = q0 + lane;
    int ex = -1;
    int64_t gid = 0;
    if (q < q_end) {
      const int l = q / k, j = q - l * k;
      gid = (int64_t)(i + (int64_t)K * l) * k + j;
      ex = topk_idx[gid];
      if (ex < 0 || ex >= E) ex = 0;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, ex);
    int row = 0;
    if (ex >= 0) row = base[warp * E + ex] + __popc(peers & lt_mask);
    __syncwarp();
    if (ex >= 0) {
      rr[row] = (int)gid;
      p.row_of[gid] = row;
      if (lane == __ffs(peers) - 1) base[warp * E + ex] += __popc(peers);
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// One chunk holding many routes (K = 1: the expert-partition schedule's global plan, or a
// single-chunk call) is planned by several blocks instead of one: each block takes a contiguous run of
// PB routes; (1) every block counts its routes per expert, (2) one block turns the counts into each
// block's first row per expert (experts in order, blocks in order within an expert) and writes the
// offsets and tile lists, (3) every block hands out its rows in route order.  The rows, offsets and
// lists are exactly those of plan_kernel: rows of an expert ascend by route, i.e. by token.
// ---------------------------------------------------------------------------
// Per-(warp, expert) counts of routes [q_begin, q_end) of chunk 0 of a one-chunk plan (route id = q).
__device__ __forceinline__ bool warp_counts(const int32_t* __restrict__ topk_idx, int q_begin, int q_end, int* base,
                                            int E, int warp, int lane) {
  bool bad = false;
  for (int q0 = q_begin; q0 < q_end; q0 += 32) {
    const int q = q0 + lane;
    int e = -1;
    if (q < q_end) {
      e = topk_idx[q];
      if (e < 0 || e >= E) { bad = true; e = 0; }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) base[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  return bad;
}

__global__ void __launch_bounds__(PLAN_THREADS, 1) plan_count_kernel(const int32_t* __restrict__ topk_idx, PlanPtrs p,
                                                                     int per_block, int* status) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  extern __shared__ int sm[];
  int* base = sm;   // [32][E]
  const int E = p.E, kc = p.N * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int x = threadIdx.x; x < 32 * E; x += PLAN_THREADS) base[x] = 0;
  __syncthreads();
  const int b0 = blockIdx.x * per_block, per_warp = per_block / 32;
  const bool bad = warp_counts(topk_idx, min(kc, b0 + warp * per_warp), min(kc, b0 + (warp + 1) * per_warp), base,
                               E, warp, lane);
  if (bad) report(status, MOE_ERR_DEVICE_CHECK, 302);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += PLAN_THREADS) {
    int c = 0;
    for (int w = 0; w < 32; ++w) c += base[w * E + e];
    p.block_counts[(int64_t)blockIdx.x * E + e] = c;
  }
}

__global__ void __launch_bounds__(PLAN_THREADS, 1) plan_lists_kernel(PlanPtrs p) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  __shared__ int scratch[33];
  const int E = p.E, kc = p.N * p.k, B = p.count_blocks;
  const int e = threadIdx.x;   // E <= 1024 = PLAN_THREADS
  int cnt = 0;
  if (e < E) {
    for (int b = 0; b < B; ++b) {
      const int c = p.block_counts[(int64_t)b * E + e];
      p.block_counts[(int64_t)b * E + e] = cnt;   // rows of expert e in blocks before b
      cnt += c;
    }
  }
  int tot;
  const int off = block_exclusive_scan(e < E ? cnt : 0, scratch, &tot);
  const int ntile = (cnt + GEMM_TILE_M - 1) / GEMM_TILE_M;
  int tile_total;
  const int toff = block_exclusive_scan(e < E ? ntile : 0, scratch, &tile_total);
  int act_total;
  const int aoff = block_exclusive_scan((e < E && cnt > 0) ? 1 : 0, scratch, &act_total);
  const int npair = (cnt + 2 * GEMM_TILE_M - 1) / (2 * GEMM_TILE_M);
  int pair_total;
  const int poff = block_exclusive_scan(e < E ? npair : 0, scratch, &pair_total);
  if (e < E) {
    for (int b = 0; b < B; ++b) p.block_counts[(int64_t)b * E + e] += off;
    p.expert_off[e] = off;
    for (int m = 0; m < ntile; ++m) {
      const int rows = min(GEMM_TILE_M, cnt - m * GEMM_TILE_M);
      p.tiles[toff + m] = make_int2(off + m * GEMM_TILE_M, e | (rows << 16));
    }
    for (int m = 0; m < npair; ++m) {
      const int rows = min(2 * GEMM_TILE_M, cnt - m * 2 * GEMM_TILE_M);
      p.tiles2[poff + m] = make_int2(off + m * 2 * GEMM_TILE_M, e | (rows << 16));
    }
    if (cnt > 0) p.active[aoff] = e;
  }
  if (threadIdx.x == 0) {
    p.expert_off[E] = kc;
    p.tile_count[0] = tile_total;
    p.tile2_count[0] = pair_total;
    p.active_count[0] = act_total;
  }
}

__global__ void __launch_bounds__(PLAN_THREADS, 1) plan_scatter_kernel(const int32_t* __restrict__ topk_idx, PlanPtrs p,
                                                                       int per_block) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  extern __shared__ int sm[];
  int* base = sm;   // [32][E]
  const int E = p.E, kc = p.N * p.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int x = threadIdx.x; x < 32 * E; x += PLAN_THREADS) base[x] = 0;
  __syncthreads();
  const int b0 = blockIdx.x * per_block, per_warp = per_block / 32;
  const int q_begin = min(kc, b0 + warp * per_warp), q_end = min(kc, b0 + (warp + 1) * per_warp);
  warp_counts(topk_idx, q_begin, q_end, base, E, warp, lane);
  __syncthreads();
  // per-warp first rows: the block's first row for the expert, then the earlier warps' counts
  for (int e = threadIdx.x; e < E; e += PLAN_THREADS) {
    int r = p.block_counts[(int64_t)blockIdx.x * E + e];
    for (int w = 0; w < 32; ++w) {
      const int c = base[w * E + e];
      base[w * E + e] = r;
      r += c;
    }
  }
  __syncthreads();
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int q0 = q_begin; q0 < q_end; q0 += 32) {
    const int q = q0 + lane;
    int ex = -1;
    if (q < q_end) {
      ex = topk_idx[q];
      if (ex < 0 || ex >= E) ex = 0;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, ex);
    int row = 0;
    if (ex >= 0) row = base[warp * E + ex] + __popc(peers & lt_mask);
    __syncwarp();
    if (ex >= 0) {
      p.row_route[row] = q;
      p.row_of[q] = row;
      if (lane == __ffs(peers) - 1) base[warp * E + ex] += __popc(peers);
    }
    __syncwarp();
  }
}

cudaError_t launch_plan(const int32_t* topk_idx, const PlanPtrs& p, int* status, cudaStream_t s) {
  const size_t smem = (size_t)(32 * p.E + 33) * sizeof(int);
  const int64_t kc = (int64_t)p.N * p.k;
  if (p.K == 1 && p.count_blocks > 1) {
    const int per_block = (int)plan_per_block(kc);   // a multiple of 1024; count_blocks = ceil(kc / per_block)
    cudaError_t err =
        cudaFuncSetAttribute(plan_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(plan_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(plan_count_kernel, dim3(p.count_blocks), dim3(PLAN_THREADS), smem, s, topk_idx, p, per_block,
                     status);
    if (err == cudaSuccess) err = launch_pdl(plan_lists_kernel, dim3(1), dim3(PLAN_THREADS), 0, s, p);
    if (err == cudaSuccess)
      err = launch_pdl(plan_scatter_kernel, dim3(p.count_blocks), dim3(PLAN_THREADS), smem, s, topk_idx, p, per_block);
    return err;
  }
  cudaError_t err = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(plan_kernel, dim3(p.K), dim3(PLAN_THREADS), smem, s, topk_idx, p, status);
}

// first_touch[e] = largest chunk index in which expert e has rows (the first
// one the backward pass visits), or -1 if it has none.
__global__ void first_touch_kernel(PlanPtrs p) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= p.E) return;
  int f = -1;
  for (int i = p.K - 1; i >= 0; --i) {
    const int* o = p.expert_off + (int64_t)i * (p.E + 1);
    if (o[e + 1] > o[e]) { f = i; break; }
  }
  p.first_touch[e] = f;
}

cudaError_t launch_first_touch(const PlanPtrs& p, cudaStream_t s) {
  return launch_pdl(first_touch_kernel, dim3((p.E + 255) / 256), dim3(256), 0, s, p);
}

// ===========================================================================
// Dispatch gather: dst[r, :] = src[token(r), :]  (expand and permute,
// RelayMoE summary 2.1).  One warp per row, 16-byte vectors.
// ===========================================================================
__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                                     const int* __restrict__ row_route, int rows, int H, int k,
                                                     int late) {
  // one warp per row; each lane moves 16-byte vectors, all loads of a group issued before the stores
  // (measured against two and four rows per warp and a persistent grid: this form is the fastest)
  if (!late) pdl_wait();   // launched with programmatic serialization: nothing global before this
  pdl_trigger();           // the GEMM that follows may set itself up while the last rows are copied
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r < rows) {
    const int t = row_route[r] / k;
    const uint4* s = reinterpret_cast<const uint4*>(src + (int64_t)t * H);
    uint4* d = reinterpret_cast<uint4*>(dst + (int64_t)r * H);
    const int nv = H / 8;
    int c = lane;
    for (; c + 32 * 7 < nv; c += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(s + c + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) d[c + 32 * u] = v[u];
    }
    for (; c < nv; c += 32) d[c] = __ldg(s + c);
  }
  // a late gather ran beside the kernel before it: it completes only after that kernel has
  if (late && blockIdx.x == 0) pdl_wait();
}

cudaError_t launch_gather(const uint16_t* src, uint16_t* dst, const int* row_route, int rows, int H, int k,
                          cudaStream_t s, bool late) {
  if (rows <= 0) return cudaSuccess;
  return launch_pdl(gather_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, src, dst, row_route, rows, H, k,
                    late && launch_chain_mode() == MOE_CHAIN_LATE ? 1 : 0);
}

// ===========================================================================
// Combine: Y[t] = bf16( sum_{j=0..k-1} g[t,j] * Op[row_of(t,j)] ), one fp32
// fused multiply-add per slot in slot order (RelayMoE summary 2.1: outputs
// returned and recombined).  One warp per (token, 512 columns).
// ===========================================================================
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ Op, const float* __restrict__ gates,
                                                      const int* __restrict__ row_of, uint16_t* __restrict__ Y,
                                                      int chunk, int K, int n_i, int H, int k) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  // one warp per (token, two adjacent 256-element spans); every lane issues the k row loads of both
  // spans back to back
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = H / 8;
  const int pairs = (nv + 63) / 64;
  const int gw = blockIdx.x * 8 + warp;
  const int l = gw / pairs, q = gw - l * pairs;
  if (l >= n_i) return;
  const int64_t t = chunk + (int64_t)K * l;
  const int my_row = lane < k ? row_of[t * k + lane] : 0;
  const float my_g = lane < k ? gates[t * k + lane] : 0.0f;
  const int c0 = q * 64 + lane, c1 = c0 + 32;
  const bool live0 = c0 < nv, live1 = c1 < nv;
  float a0[8], a1[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) a0[x] = a1[x] = 0.0f;
#pragma unroll 8
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, my_row, j);
    const float g = __shfl_sync(0xffffffffu, my_g, j);
    const uint4* base = reinterpret_cast<const uint4*>(Op + (int64_t)row * H);
    if (live0) {
      const uint4 v = __ldg(base + c0);
      a0[0] = __fmaf_rn(g, bf16_lo(v.x), a0[0]); a0[1] = __fmaf_rn(g, bf16_hi(v.x), a0[1]);
      a0[2] = __fmaf_rn(g, bf16_lo(v.y), a0[2]); a0[3] = __fmaf_rn(g, bf16_hi(v.y), a0[3]);
      a0[4] = __fmaf_rn(g, bf16_lo(v.z), a0[4]); a0[5] = __fmaf_rn(g, bf16_hi(v.z), a0[5]);
      a0[6] = __fmaf_rn(g, bf16_lo(v.w), a0[6]); a0[7] = __fmaf_rn(g, bf16_hi(v.w), a0[7]);
    }
    if (live1) {
      const uint4 v = __ldg(base + c1);
      a1[0] = __fmaf_rn(g, bf16_lo(v.x), a1[0]); a1[1] = __fmaf_rn(g, bf16_hi(v.x), a1[1]);
      a1[2] = __fmaf_rn(g, bf16_lo(v.y), a1[2]); a1[3] = __fmaf_rn(g, bf16_hi(v.y), a1[3]);
      a1[4] = __fmaf_rn(g, bf16_lo(v.z), a1[4]); a1[5] = __fmaf_rn(g, bf16_hi(v.z), a1[5]);
      a1[6] = __fmaf_rn(g, bf16_lo(v.w), a1[6]); a1[7] = __fmaf_rn(g, bf16_hi(v.w), a1[7]);
    }
  }
  uint4* y = reinterpret_cast<uint4*>(Y + t * H);
  if (live0) y[c0] = make_uint4(pack_bf16(a0[0], a0[1]), pack_bf16(a0[2], a0[3]), pack_bf16(a0[4], a0[5]),
                                pack_bf16(a0[6], a0[7]));
  if (live1) y[c1] = make_uint4(pack_bf16(a1[0], a1[1]), pack_bf16(a1[2], a1[3]), pack_bf16(a1[4], a1[5]),
                                pack_bf16(a1[6], a1[7]));
}

cudaError_t launch_combine(const uint16_t* Op, const float* gates, const int* row_of, uint16_t* Y, int chunk,
                           int K, int n_i, int H, int k, cudaStream_t s) {
  if (n_i <= 0) return cudaSuccess;
  const int64_t warps = (int64_t)n_i * ((H / 8 + 63) / 64);
  return launch_pdl(combine_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, Op, gates, row_of, Y, chunk, K, n_i, H, k);
}

// ===========================================================================
// Router backward of a chunk (per route), then the unpermute:
//   dg_j  = sum over the dActU GEMM's column tiles of the partial sums (tile order)
//   dl_j  = g_j (dg_j - sum_i g_i dg_i)       (softmax restricted to the selected set)
//   the router-path term dl_j Wr[e_j] is added to dXp[row_j] by the dX GEMM's epilogue (fp32), so
//   dX[t] = bf16( sum_j dXp[row_of(t,j)] )   (fp32, slot order)
// ===========================================================================
// One warp per token of the chunk; lane j < k holds slot j.
__global__ void __launch_bounds__(256) route_grad_kernel(const float* __restrict__ dgp, int dgp_tiles,
                                                         const float* __restrict__ gates,
                                                         const int* __restrict__ row_of, float* __restrict__ dgates,
                                                         float* __restrict__ dlogit, float* __restrict__ dl_row,
                                                         int chunk, int K, int n_i, int k) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int l = blockIdx.x * 8 + warp;
  if (l >= n_i) return;
  const int64_t t = chunk + (int64_t)K * l;
  int my_row = 0;
  float my_g = 0.0f, my_dg = 0.0f;
  if (lane < k) {
    my_row = row_of[t * k + lane];
    my_g = gates[t * k + lane];
    const float* d = dgp + (int64_t)my_row * dgp_tiles;
    for (int qq = 0; qq < dgp_tiles; ++qq) my_dg += d[qq];
  }
  float s = 0.0f;
  for (int j = 0; j < k; ++j) {
    const float gj = __shfl_sync(0xffffffffu, my_g, j);
    const float dj = __shfl_sync(0xffffffffu, my_dg, j);
    s = __fmaf_rn(gj, dj, s);
  }
  const float my_dl = my_g * (my_dg - s);
  if (lane < k) {
    if (dgates) dgates[t * k + lane] = my_dg;
    dlogit[t * k + lane] = my_dl;
    dl_row[my_row] = my_dl;
  }
}

cudaError_t launch_route_grad(const float* dgp, int dgp_tiles, const float* gates, const int* row_of, float* dgates,
                              float* dlogit, float* dl_row, int chunk, int K, int n_i, int k, cudaStream_t s) {
  if (n_i <= 0) return cudaSuccess;
  return launch_pdl(route_grad_kernel, dim3((unsigned)((n_i + 7) / 8)), dim3(256), 0, s, dgp, dgp_tiles, gates,
                    row_of, dgates, dlogit, dl_row, chunk, K, n_i, k);
}

// One warp per (token, two adjacent 256-element spans); every lane issues the k row loads of both spans
// back to back.
__global__ void __launch_bounds__(256) unpermute_kernel(const uint16_t* __restrict__ dXp,
                                                        const int* __restrict__ row_of, uint16_t* __restrict__ dX,
                                                        int chunk, int K, int n_i, int H, int k) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = H / 8;
  const int pairs = (nv + 63) / 64;
  const int gw = blockIdx.x * 8 + warp;
  const int l = gw / pairs, q = gw - l * pairs;
  if (l >= n_i) return;
  const int64_t t = chunk + (int64_t)K * l;
  const int my_row = lane < k ? row_of[t * k + lane] : 0;
  const int c0 = q * 64 + lane, c1 = c0 + 32;
  const bool live0 = c0 < nv, live1 = c1 < nv;
  float a0[8], a1[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) a0[x] = a1[x] = 0.0f;
#pragma unroll 8
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, my_row, j);
    const uint4* base = reinterpret_cast<const uint4*>(dXp + (int64_t)row * H);
    if (live0) {
      const uint4 v = __ldg(base + c0);
      a0[0] += bf16_lo(v.x); a0[1] += bf16_hi(v.x); a0[2] += bf16_lo(v.y); a0[3] += bf16_hi(v.y);
      a0[4] += bf16_lo(v.z); a0[5] += bf16_hi(v.z); a0[6] += bf16_lo(v.w); a0[7] += bf16_hi(v.w);
    }
    if (live1) {
      const uint4 v = __ldg(base + c1);
      a1[0] += bf16_lo(v.x); a1[1] += bf16_hi(v.x); a1[2] += bf16_lo(v.y); a1[3] += bf16_hi(v.y);
      a1[4] += bf16_lo(v.z); a1[5] += bf16_hi(v.z); a1[6] += bf16_lo(v.w); a1[7] += bf16_hi(v.w);
    }
  }
  uint4* d = reinterpret_cast<uint4*>(dX + t * H);
  if (live0) d[c0] = make_uint4(pack_bf16(a0[0], a0[1]), pack_bf16(a0[2], a0[3]), pack_bf16(a0[4], a0[5]),
                                pack_bf16(a0[6], a0[7]));
  if (live1) d[c1] = make_uint4(pack_bf16(a1[0], a1[1]), pack_bf16(a1[2], a1[3]), pack_bf16(a1[4], a1[5]),
                                pack_bf16(a1[6], a1[7]));
}

cudaError_t launch_unpermute(const uint16_t* dXp, const int* row_of, uint16_t* dX, int chunk, int K, int n_i, int H,
                             int k, cudaStream_t s) {
  if (n_i <= 0) return cudaSuccess;
  const int64_t warps = (int64_t)n_i * ((H / 8 + 63) / 64);
  return launch_pdl(unpermute_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, dXp, row_of, dX, chunk, K,
                    n_i, H, k);
}

// ===========================================================================
// Router weight gradient for one chunk: dWr[e, h] (+)= sum over the chunk's
// rows of expert e, in row order, of dlogit(route) * X[token, h].
// ===========================================================================
// Two passes over the chunk's 128-row tiles, so a hot expert's rows are spread over many blocks:
// (1) block (tile, 256-column slab): warp w adds rows 16w .. 16w+15 of the tile in order, the 8 warp
//     sums are added in warp order, and the tile's partial sum goes to partial[tile][h];
// (2) block (expert, 256-column slab): the expert's tiles (contiguous in the tile list, found by a
//     binary search on the expert ids) are added in list order onto the stored gradient (or onto 0 on
//     the expert's first chunk).  A fixed order throughout, so the result is reproducible run to run.
__global__ void __launch_bounds__(256) router_dw_tiles_kernel(const uint16_t* __restrict__ X,
                                                              const float* __restrict__ dlogit,
                                                              const int* __restrict__ row_route,
                                                              const int2* __restrict__ tiles,
                                                              const int* __restrict__ tile_count,
                                                              float* __restrict__ partial, int H, int k) {
  __shared__ float part[8][256];
  __shared__ int s_tok[128];
  __shared__ float s_dl[128];
  if ((int)blockIdx.x >= *tile_count) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int2 tl = tiles[blockIdx.x];
  const int row0 = tl.x, rows = tl.y >> 16;
  if ((int)threadIdx.x < rows) {
    const int q = row_route[row0 + threadIdx.x];
    s_tok[threadIdx.x] = q / k;
    s_dl[threadIdx.x] = dlogit[q];
  }
  __syncthreads();
  const int h0 = blockIdx.y * 256 + lane * 8;
  float acc[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) acc[x] = 0.0f;
  if (h0 < H) {
    const int a = warp * 16, b = min(rows, a + 16);
#pragma unroll 8
    for (int j = a; j < b; ++j) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)s_tok[j] * H + h0));
      const float dl = s_dl[j];
      acc[0] = __fmaf_rn(dl, bf16_lo(v.x), acc[0]); acc[1] = __fmaf_rn(dl, bf16_hi(v.x), acc[1]);
      acc[2] = __fmaf_rn(dl, bf16_lo(v.y), acc[2]); acc[3] = __fmaf_rn(dl, bf16_hi(v.y), acc[3]);
      acc[4] = __fmaf_rn(dl, bf16_lo(v.z), acc[4]); acc[5] = __fmaf_rn(dl, bf16_hi(v.z), acc[5]);
      acc[6] = __fmaf_rn(dl, bf16_lo(v.w), acc[6]); acc[7] = __fmaf_rn(dl, bf16_hi(v.w), acc[7]);
    }
  }
#pragma unroll
  for (int x = 0; x < 8; ++x) part[warp][lane * 8 + x] = acc[x];
  __syncthreads();
  const int col = warp * 32 + lane;
  const int h = blockIdx.y * 256 + col;
  if (h < H) {
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += part[w][col];
    partial[(int64_t)blockIdx.x * H + h] = sum;
  }
}

__global__ void __launch_bounds__(256) router_dw_sum_kernel(const float* __restrict__ partial,
                                                            const int2* __restrict__ tiles,
                                                            const int* __restrict__ tile_count,
                                                            const int* __restrict__ active,
                                                            const int* __restrict__ active_count,
                                                            const int* __restrict__ first_touch,
                                                            float* __restrict__ dWr, int chunk, int H) {
  if ((int)blockIdx.x >= *active_count) return;
  const int e = active[blockIdx.x];
  const int T = *tile_count;
  // first tile of expert e: tiles are in ascending expert order
  int lo = 0, hi = T;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((tiles[mid].y & 0xFFFF) < e) lo = mid + 1;
    else hi = mid;
  }
  const int h = blockIdx.y * 256 + threadIdx.x;
  if (h >= H) return;
  float tot = (first_touch[e] == chunk) ? 0.0f : dWr[(int64_t)e * H + h];
  float sum = 0.0f;
  for (int t = lo; t < T && (tiles[t].y & 0xFFFF) == e; ++t) sum += partial[(int64_t)t * H + h];
  dWr[(int64_t)e * H + h] = tot + sum;
}

cudaError_t launch_router_dw(const uint16_t* X, const float* dlogit, const int* row_route, const int2* tiles,
                             const int* tile_count, int max_tiles, const int* active, const int* active_count,
                             const int* first_touch, float* partial, float* dWr, int chunk, int E, int H, int k,
                             cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  const unsigned slabs = (unsigned)((H + 255) / 256);
  router_dw_tiles_kernel<<<dim3((unsigned)max_tiles, slabs), 256, 0, s>>>(X, dlogit, row_route, tiles, tile_count,
                                                                          partial, H, k);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  router_dw_sum_kernel<<<dim3((unsigned)E, slabs), 256, 0, s>>>(partial, tiles, tile_count, active, active_count,
                                                                first_touch, dWr, chunk, H);
  return cudaGetLastError();
}

// Zero the gradients of experts that no token selected.
__global__ void zero_untouched_kernel(const int* __restrict__ first_touch, float* dWg, float* dWu, float* dWd,
                                      float* dWr, int64_t IH, int H) {
  const int e = blockIdx.y;
  if (first_touch[e] >= 0) return;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t x = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; x < IH; x += stride) {
    const float4 z = make_float4(0, 0, 0, 0);
    *reinterpret_cast<float4*>(dWg + e * IH + x) = z;
    *reinterpret_cast<float4*>(dWu + e * IH + x) = z;
    *reinterpret_cast<float4*>(dWd + e * IH + x) = z;
  }
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < H; x += (int64_t)gridDim.x * blockDim.x)
    dWr[(int64_t)e * H + x] = 0.0f;
}

cudaError_t launch_zero_untouched(const int* first_touch, float* dWg, float* dWu, float* dWd, float* dWr, int E,
                                  int H, int I, cudaStream_t s) {
  dim3 grid(64, E);
  zero_untouched_kernel<<<grid, 256, 0, s>>>(first_touch, dWg, dWu, dWd, dWr, (int64_t)I * H, H);
  return cudaGetLastError();
}

// ===========================================================================
// Diagnostic: a bounded wait on a barrier nothing signals.
// ===========================================================================
__global__ void diag_wait_kernel(int* status, int64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int ab;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    ab = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0, &ab, limit_ns, status, 900);
}

cudaError_t launch_diag_wait(int* status, int64_t limit_ns, cudaStream_t s) {
  diag_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
