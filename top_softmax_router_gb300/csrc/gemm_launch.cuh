// Host-side launch helper for grouped_gemm_kernel.
#pragma once

#include "gemm2sm_kernel.cuh"
#include "gemm_kernel.cuh"
#include "kernels.h"

// Row-tile GEMMs (gate/up, down, dX, dActU) run on CTA pairs (2-SM MMA, 256-row tiles) when
// ChunkGemm::pair is set, else on single CTAs (128-row tiles).

namespace moe {

template <int EPI, bool A_MN, bool B_MN, bool SEGK, int BN, bool DUAL_B, bool TWO_PHASE, int GATH = 0>
cudaError_t launch_grouped_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                                const CUtensorMap& b1, const GemmParams& p, int num_sms, cudaStream_t s,
                                const CUtensorMap* o0 = nullptr, const CUtensorMap* o1 = nullptr) {
  auto kern = grouped_gemm_kernel<EPI, A_MN, B_MN, SEGK, BN, DUAL_B, TWO_PHASE, GATH>;
  const int smem = GemmSmem<BN, EPI>::TOTAL;
  GemmParams q = p;
  if (!SEGK) q.nk_total = TWO_PHASE ? 2 * p.nk : p.nk;
  if (launch_chain_mode() < MOE_CHAIN_LATE) q.pdl_late = q.trigger_early = 0;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // Programmatic dependent launch: the kernel's set-up (barriers, TMEM, descriptor prefetch) may overlap
  // the tail of the kernel before it; it waits for that kernel before touching global memory.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_sms);
  cfg.blockDim = dim3(gemm_threads(EPI));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_chain_mode() >= MOE_CHAIN_EARLY ? 1 : 0;
  err = cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, o0 ? *o0 : a0, o1 ? *o1 : a0, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

inline GemmParams base_params(const ChunkGemm& c, int ctr_slot) {
  GemmParams p = {};
  p.work_ctr = c.work_ctr ? c.work_ctr + ctr_slot : nullptr;
  p.tiles = c.tiles;
  p.tile_count = c.tile_count;
  p.tiles2 = c.tiles2;
  p.tile2_count = c.tile2_count;
  p.active = c.active;
  p.active_count = c.active_count;
  p.expert_off = c.expert_off;
  p.row_route = c.row_route;
  p.route_k = c.k;
  p.chunk = c.chunk;
  p.status = c.status;
  p.limit_ns = c.limit_ns;
  p.n_problems = 1;
  p.pdl_late = c.late_wait ? 1 : 0;
  p.trigger_early = c.trigger_early ? 1 : 0;
  p.wait_stats = gemm_wait_stats_buffer();
  return p;
}

}  // namespace moe
