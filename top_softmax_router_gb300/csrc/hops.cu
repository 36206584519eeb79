// Kernels of the expert-partition ("hop") schedule of the MoE block.
//
// RelayMoE summary, sections 3.1 and 3.3: instead of chunking the tokens, the
// computation walks over partitions of the experts ("hops"); each hop runs all
// routes to its experts, then releases its intermediates before the next hop.
// On one device the ring becomes a loop over expert ranges [e0, e1).  Each
// expert's weights are read once per pass and its weight gradient is written
// once (no per-chunk read-modify-write); the price is a routed working set set
// by the largest hop, which depends on the router (section 3.3).
//
// The hop's rows are a contiguous range of the global expert-sorted
// permutation (the chunk plan with one chunk), rebased to start at 0.  Per-token
// outputs accumulate in fp32 across hops (hop order, then slot order).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------
// Hop plan: one 1024-thread block per hop, all hops in one launch.  Rebases each hop's slice of the
// global plan into that hop's arrays.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024, 1) hop_plan_kernel(const int* __restrict__ expert_off_g,
                                                           const int* __restrict__ row_route_g, HopSets S, int P,
                                                           int E, int cap, int* status) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  __shared__ int scratch[33];
  const int h = blockIdx.x;
  const HopPtrs hp = hop_set(S, h);
  const int e0 = (int)((int64_t)h * E / P), e1 = (int)((int64_t)(h + 1) * E / P);
  const int base = expert_off_g[e0];
  int rows = expert_off_g[e1] - base;
  if (rows > cap) {                     // the hop does not fit the workspace: run nothing, report
    if (threadIdx.x == 0) report(status, MOE_ERR_DEVICE_CHECK, 601);
    rows = -1;
  }
  const int el = threadIdx.x;            // expert e0 + el
  const int e = e0 + el;
  const bool mine = e < e1;
  const int cnt = (mine && rows >= 0) ? expert_off_g[e + 1] - expert_off_g[e] : 0;
  const int ntile = (cnt + 127) / 128;
  const int npair = (cnt + 255) / 256;
  int tile_total, act_total, pair_total;
  const int toff = block_exclusive_scan(ntile, scratch, &tile_total);
  const int aoff = block_exclusive_scan(cnt > 0 ? 1 : 0, scratch, &act_total);
  const int poff = block_exclusive_scan(npair, scratch, &pair_total);
  if (mine) {
    const int off = rows >= 0 ? expert_off_g[e] - base : 0;
    hp.expert_off[e] = off;
    for (int m = 0; m < ntile; ++m)
      hp.tiles[toff + m] = make_int2(off + m * 128, e | (min(128, cnt - m * 128) << 16));
    for (int m = 0; m < npair; ++m)
      hp.tiles2[poff + m] = make_int2(off + m * 256, e | (min(256, cnt - m * 256) << 16));
    if (cnt > 0) hp.active[aoff] = e;
    hp.first_touch[e] = cnt > 0 ? h : -1;
  }
  if (threadIdx.x == 0) {
    hp.expert_off[e1] = rows >= 0 ? rows : 0;
    *hp.tile_count = tile_total;
    *hp.tile2_count = pair_total;
    *hp.active_count = act_total;
    *hp.base = base;
    *hp.rows = rows >= 0 ? rows : 0;
  }
  for (int r = threadIdx.x; r < rows; r += blockDim.x) hp.row_route[r] = row_route_g[base + r];
}

cudaError_t launch_hop_plan_all(const int* expert_off_g, const int* row_route_g, const HopSets& S, int P, int E,
                                int cap, int* status, cudaStream_t s) {
  return launch_pdl(hop_plan_kernel, dim3((unsigned)P), dim3(1024), 0, s, expert_off_g, row_route_g, S, P, E, cap,
                    status);
}

// ---------------------------------------------------------------------------
// Gather with the row count on the device: dst[r] = src[token(r)], r < *rows.  The grid is sized for
// the largest possible hop, so it is a persistent grid (8 blocks per SM) whose warps stride over the
// rows rather than one block per 8 rows, most of which would find nothing to do.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_dev_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                                         const int* __restrict__ row_route,
                                                         const int* __restrict__ rows_dev, int H, int k,
                                                         int late) {
  if (!late) pdl_wait();   // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = *rows_dev;
  const int nv = H / 8;
  for (int r = blockIdx.x * 8 + warp; r < rows; r += gridDim.x * 8) {
    const int t = row_route[r] / k;
    const uint4* sp = reinterpret_cast<const uint4*>(src + (int64_t)t * H);
    uint4* d = reinterpret_cast<uint4*>(dst + (int64_t)r * H);
    int c = lane;
    for (; c + 32 * 7 < nv; c += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(sp + c + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) d[c + 32 * u] = v[u];
    }
    for (; c < nv; c += 32) d[c] = __ldg(sp + c);
  }
  // a late gather ran beside the kernel before it: it completes only after that kernel has
  if (late && blockIdx.x == 0) pdl_wait();
}

cudaError_t launch_gather_dev(const uint16_t* src, uint16_t* dst, const int* row_route, const int* rows_dev, int cap,
                              int H, int k, cudaStream_t s, bool late) {
  if (cap <= 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>((cap + 7) / 8, (int64_t)device_sm_count() * 8);
  return launch_pdl(gather_dev_kernel, dim3(blocks), dim3(256), 0, s, src, dst, row_route, rows_dev, H, k,
                    late && launch_chain_mode() == MOE_CHAIN_LATE ? 1 : 0);
}

// ---------------------------------------------------------------------------
// Per-token slots of the current hop, shared by the two accumulation kernels.
// Lane j < k holds slot j; `in` says whether its expert lies in [e0, e1).
// ---------------------------------------------------------------------------
struct HopSlot {
  int row;     // row in the hop's buffers (global row minus the hop base)
  int e;
  float g;
  bool in;
};

__device__ __forceinline__ HopSlot hop_slot(const int* row_of_g, const int32_t* topk_idx, const float* gates,
                                            int64_t t, int k, int lane, int base, int rows, int e0, int e1) {
  HopSlot s{0, 0, 0.0f, false};
  if (lane < k) {
    s.e = topk_idx[t * k + lane];
    s.in = s.e >= e0 && s.e < e1;
    if (s.in) {
      s.row = row_of_g[t * k + lane] - base;
      s.in = s.row >= 0 && s.row < rows;   // a hop that did not fit the workspace has rows == 0
    }
    if (gates) s.g = gates[t * k + lane];
  }
  return s;
}

// Yacc[t] += sum over the token's slots in this hop, in slot order, of g_j * Op[row_j]   (fp32)
__global__ void __launch_bounds__(256) combine_hop_kernel(const uint16_t* __restrict__ Op, const float* __restrict__ gates,
                                                          const int* __restrict__ row_of_g,
                                                          const int32_t* __restrict__ topk_idx,
                                                          const int* __restrict__ hop_base,
                                                          const int* __restrict__ hop_rows, int e0, int e1,
                                                          float* __restrict__ Yacc, int N, int H, int k) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = H / 8;
  const int spans = (nv + 31) / 32;
  const int gw = blockIdx.x * 8 + warp;
  const int t = gw / spans, sp = gw - t * spans;
  if (t >= N) return;
  const HopSlot s = hop_slot(row_of_g, topk_idx, gates, t, k, lane, *hop_base, *hop_rows, e0, e1);
  const uint32_t in_mask = __ballot_sync(0xffffffffu, s.in);
  if (in_mask == 0) return;                        // uniform across the warp
  const int c = sp * 32 + lane;
  const bool live = c < nv;
  float4* acc_p = reinterpret_cast<float4*>(Yacc + (int64_t)t * H) + 2 * c;
  float acc[8];
  if (live) {
    const float4 a = acc_p[0], b = acc_p[1];
    acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
  }
  for (int j = 0; j < k; ++j) {
    if (!((in_mask >> j) & 1u)) continue;
    const int row = __shfl_sync(0xffffffffu, s.row, j);
    const float g = __shfl_sync(0xffffffffu, s.g, j);
    if (!live) continue;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(Op + (int64_t)row * H) + c);
    acc[0] = __fmaf_rn(g, bf16_lo(v.x), acc[0]); acc[1] = __fmaf_rn(g, bf16_hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(g, bf16_lo(v.y), acc[2]); acc[3] = __fmaf_rn(g, bf16_hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(g, bf16_lo(v.z), acc[4]); acc[5] = __fmaf_rn(g, bf16_hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(g, bf16_lo(v.w), acc[6]); acc[7] = __fmaf_rn(g, bf16_hi(v.w), acc[7]);
  }
  if (!live) return;
  acc_p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  acc_p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

cudaError_t launch_combine_hop(const uint16_t* Op, const float* gates, const int* row_of_g, const int32_t* topk_idx,
                               const int* hop_base, const int* hop_rows, int e0, int e1, float* Yacc, int N, int H,
                               int k, cudaStream_t s) {
  const int64_t warps = (int64_t)N * ((H / 8 + 31) / 32);
  return launch_pdl(combine_hop_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, Op, gates, row_of_g, topk_idx, hop_base, hop_rows, e0, e1, Yacc, N, H, k);
}

// out[i] = bf16(in[i])  (n a multiple of 8)
__global__ void __launch_bounds__(256) to_bf16_kernel(const float* __restrict__ in, uint16_t* __restrict__ out,
                                                      int64_t n8) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(in)[2 * i], b = reinterpret_cast<const float4*>(in)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16(a.x, a.y); o.y = pack_bf16(a.z, a.w); o.z = pack_bf16(b.x, b.y); o.w = pack_bf16(b.z, b.w);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
}

cudaError_t launch_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t n8 = n / 8;
  const int blocks = (int)std::min<int64_t>((n8 + 255) / 256, 152 * 16);
  return launch_pdl(to_bf16_kernel, dim3(blocks), dim3(256), 0, s, in, out, n8);
}

// Backward, per hop: dXacc[t] += sum over the token's slots in this hop of dXp[row_j] (fp32, slot
// order); dg[t,j] = sum of the dActU tile partials of row_j (index order), written by span 0.
__global__ void __launch_bounds__(256) unpermute_hop_kernel(const uint16_t* __restrict__ dXp,
                                                            const float* __restrict__ dgp, int dgp_tiles,
                                                            const int* __restrict__ row_of_g,
                                                            const int32_t* __restrict__ topk_idx,
                                                            const int* __restrict__ hop_base,
                                                            const int* __restrict__ hop_rows, int e0, int e1,
                                                            float* __restrict__ dXacc, float* __restrict__ dg_route,
                                                            int N, int H, int k) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = H / 8;
  const int spans = (nv + 31) / 32;
  const int gw = blockIdx.x * 8 + warp;
  const int t = gw / spans, sp = gw - t * spans;
  if (t >= N) return;
  const HopSlot s = hop_slot(row_of_g, topk_idx, nullptr, t, k, lane, *hop_base, *hop_rows, e0, e1);
  const uint32_t in_mask = __ballot_sync(0xffffffffu, s.in);
  if (in_mask == 0) return;
  if (sp == 0 && s.in) {
    const float* d = dgp + (int64_t)s.row * dgp_tiles;
    float dg = 0.0f;
    for (int q = 0; q < dgp_tiles; ++q) dg += d[q];
    dg_route[(int64_t)t * k + lane] = dg;
  }
  const int c = sp * 32 + lane;
  const bool live = c < nv;
  float4* acc_p = reinterpret_cast<float4*>(dXacc + (int64_t)t * H) + 2 * c;
  float acc[8];
  if (live) {
    const float4 a = acc_p[0], b = acc_p[1];
    acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
  }
  for (int j = 0; j < k; ++j) {
    if (!((in_mask >> j) & 1u)) continue;
    const int row = __shfl_sync(0xffffffffu, s.row, j);
    if (!live) continue;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(dXp + (int64_t)row * H) + c);
    acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x); acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
    acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z); acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
  }
  if (!live) return;
  acc_p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  acc_p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

cudaError_t launch_unpermute_hop(const uint16_t* dXp, const float* dgp, int dgp_tiles, const int* row_of_g,
                                 const int32_t* topk_idx, const int* hop_base, const int* hop_rows, int e0, int e1,
                                 float* dXacc, float* dg_route, int N, int H, int k, cudaStream_t s) {
  const int64_t warps = (int64_t)N * ((H / 8 + 31) / 32);
  return launch_pdl(unpermute_hop_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, dXp, dgp, dgp_tiles, row_of_g, topk_idx, hop_base, hop_rows, e0, e1, dXacc, dg_route, N, H, k);
}

// After the last hop: dl_j = g_j (dg_j - sum_i g_i dg_i); dX[t] = bf16(dXacc[t] + sum_j dl_j Wr[e_j]).
__global__ void __launch_bounds__(256) router_final_kernel(const float* __restrict__ dXacc,
                                                           const float* __restrict__ dg_route,
                                                           const float* __restrict__ gates,
                                                           const int32_t* __restrict__ topk_idx,
                                                           const float* __restrict__ Wr, uint16_t* __restrict__ dX,
                                                           float* __restrict__ dgates, float* __restrict__ dlogit,
                                                           int N, int H, int k, int E) {
  pdl_wait();      // launched with programmatic serialization: nothing global before this
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nv = H / 8;
  const int spans = (nv + 31) / 32;
  const int gw = blockIdx.x * 8 + warp;
  const int t = gw / spans, sp = gw - t * spans;
  if (t >= N) return;
  int my_e = 0;
  float my_g = 0.0f, my_dg = 0.0f;
  if (lane < k) {
    my_e = topk_idx[(int64_t)t * k + lane];
    if (my_e < 0 || my_e >= E) my_e = 0;
    my_g = gates[(int64_t)t * k + lane];
    my_dg = dg_route[(int64_t)t * k + lane];
  }
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s = __fmaf_rn(__shfl_sync(0xffffffffu, my_g, j), __shfl_sync(0xffffffffu, my_dg, j), s);
  const float my_dl = my_g * (my_dg - s);
  if (lane < k && sp == 0) {
    if (dgates) dgates[(int64_t)t * k + lane] = my_dg;
    dlogit[(int64_t)t * k + lane] = my_dl;
  }
  const int c = sp * 32 + lane;
  const bool live = c < nv;
  float acc[8];
  if (live) {
    const float4* a_p = reinterpret_cast<const float4*>(dXacc + (int64_t)t * H) + 2 * c;
    const float4 a = a_p[0], b = a_p[1];
    acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
  }
  for (int j = 0; j < k; ++j) {
    const int e = __shfl_sync(0xffffffffu, my_e, j);
    const float dl = __shfl_sync(0xffffffffu, my_dl, j);
    if (!live) continue;
    const float4* w = reinterpret_cast<const float4*>(Wr + (int64_t)e * H) + 2 * c;
    const float4 a = __ldg(w), b = __ldg(w + 1);
    acc[0] = __fmaf_rn(dl, a.x, acc[0]); acc[1] = __fmaf_rn(dl, a.y, acc[1]);
    acc[2] = __fmaf_rn(dl, a.z, acc[2]); acc[3] = __fmaf_rn(dl, a.w, acc[3]);
    acc[4] = __fmaf_rn(dl, b.x, acc[4]); acc[5] = __fmaf_rn(dl, b.y, acc[5]);
    acc[6] = __fmaf_rn(dl, b.z, acc[6]); acc[7] = __fmaf_rn(dl, b.w, acc[7]);
  }
  if (!live) return;
  uint4 o;
  o.x = pack_bf16(acc[0], acc[1]); o.y = pack_bf16(acc[2], acc[3]);
  o.z = pack_bf16(acc[4], acc[5]); o.w = pack_bf16(acc[6], acc[7]);
  reinterpret_cast<uint4*>(dX + (int64_t)t * H)[c] = o;
}

cudaError_t launch_router_final(const float* dXacc, const float* dg_route, const float* gates, const int32_t* topk_idx,
                                const float* Wr, uint16_t* dX, float* dgates, float* dlogit, int N, int H, int k,
                                int E, cudaStream_t s) {
  const int64_t warps = (int64_t)N * ((H / 8 + 31) / 32);
  return launch_pdl(router_final_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, dXacc, dg_route, gates, topk_idx, Wr, dX, dgates, dlogit, N, H, k, E);
}

}  // namespace moe
