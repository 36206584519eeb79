// Row-tile grouped GEMM on CTA pairs: the 2-SM form of the 5th-generation tensor-core MMA.
//
// Same computation and epilogues as the row-tile kernels of gemm_kernel.cuh (gate/up + SwiGLU,
// down projection, dX, dActU), on tiles of 256 rows of one expert.  A cluster of two CTAs works on
// one tile: CTA r loads its 128 rows of the activation operand and half of the 256-wide weight
// tile (128 weight rows, or two of the four 64-wide MN atoms); the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which reads both CTAs' shared memory and
// leaves rows 0..127 of the accumulator in its own TMEM and rows 128..255 in its peer's.  Each CTA
// keeps only 32 KB per pipeline stage (16 KB rows + 16 KB weights), half the weight bytes of the
// one-CTA form, so six stages fit and the mainloop tolerates more latency.
//
// Synchronisation: both producers' TMA loads complete on the even CTA's full barrier (which the
// even producer arms for both CTAs' bytes); the even CTA's commits arrive on both CTAs' empty and
// accumulator-full barriers (multicast); both CTAs' epilogue warps release the accumulator on the
// even CTA's accumulator-empty barrier.  Every wait is bounded (wait_bounded).
#pragma once

#include "gemm_kernel.cuh"

namespace moe {

struct PairSmem {
  static constexpr int A_BYTES = 128 * GEMM_BK * 2;      // 16 KB: this CTA's rows
  static constexpr int B_BYTES = 128 * GEMM_BK * 2;      // 16 KB: this CTA's half of the weight tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = BAR_OFF + 256 + 1024;
  static constexpr int TMEM_COLS = 512;                  // two 256-column accumulators
};

// Work item of a pair tile: (256-row tile, N tile).
__device__ __forceinline__ Work decode_pair(const GemmParams& p, int w) {
  Work r;
  const int t = w / p.n_tiles;
  r.nt = w - t * p.n_tiles;
  const int2 tl = p.tiles2[t];
  r.row0 = tl.x;
  r.e = tl.y & 0xFFFF;
  r.rows = tl.y >> 16;
  r.mt = 0;
  r.prob = 0;
  r.nkb = p.nk_total;
  return r;
}

// GATH = 1: each CTA gathers its 128 A rows straight from the token-major source (map ta0 of
// make_map_gather) by the rows' tokens, four rows per tile::gather4, as the one-CTA kernel does.
template <int EPI, bool B_MN, bool DUAL_B, bool TWO_PHASE, int GATH = 0>
__global__ void __launch_bounds__(gemm_threads(EPI), 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap ta1,
                             const __grid_constant__ CUtensorMap tb0, const __grid_constant__ CUtensorMap tb1,
                             const GemmParams p) {
  using S = PairSmem;
  constexpr int BN = 256;
  constexpr int NE = gemm_epi_warps(EPI);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::BAR_OFF + 8 * (2 * S::STAGES + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int clusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * NE);          // both CTAs' epilogue warps
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&ta0);
    tma_prefetch_desc(&tb0);
    if (TWO_PHASE) tma_prefetch_desc(&ta1);
    if (DUAL_B || TWO_PHASE) tma_prefetch_desc(&tb1);
  }
  if (warp == 1) {
    tc_alloc_pair(smem_u32(tmem_slot), S::TMEM_COLS);
    tc_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();                                // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (!p.pdl_late) pdl_wait();                   // no global memory access before this point
  if (p.trigger_early) pdl_trigger();

  const int total = (*p.tile2_count) * p.n_tiles;

  if (warp == 0 && GATH != 0) {
    // ------------------------------------------------------------ producer, gather-on-load (both CTAs)
    static_assert(GATH == 0 || !TWO_PHASE, "gathered operands have one K phase");
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    long long ws_stage = 0;
    for (int w = cluster; w < total && ok; w += clusters) {
      const Work wk = decode_pair(p, w);
      int tok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 128 * (int)rank + 4 * lane + j;   // this lane's rows of the 256-row tile
        tok[j] = gather_token(p, wk.row0 + (r < wk.rows ? r : 0));
      }
      for (int kb = 0; kb < wk.nkb; ++kb) {
        int good = 1;
        const long long ws0 = ws_clock();
        if (lane == 0) good = wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.limit_ns, p.status, 111);
        ws_stage += ws_clock() - ws0;
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        if (leader && lane == 0) mbar_expect_tx(full_bar(stage), 2 * S::STAGE_BYTES);
        __syncwarp();
        const uint32_t fb = mapa_shared(full_bar(stage), 0);
        const uint32_t sa = sbase + stage * S::STAGE_BYTES;
        const uint32_t sb = sa + S::A_BYTES;
        const int k0 = kb * GEMM_BK;
        tma_gather4_pair(sa + 512 * lane, &ta0, fb, k0, tok[0], tok[1], tok[2], tok[3]);
        if (lane == 0) {
          if constexpr (DUAL_B) {
            tma_load_3d_pair(sb, rank ? &tb1 : &tb0, fb, k0, wk.nt * 128, wk.e);       // gate | up half
          } else if constexpr (!B_MN) {
            tma_load_3d_pair(sb, &tb0, fb, k0, wk.nt * BN + 128 * (int)rank, wk.e);
          } else {
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_load_3d_pair(sb + b * 8192, &tb0, fb, wk.nt * BN + 64 * (2 * (int)rank + b), k0, wk.e);
          }
        }
        if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (lane == 0) {
      pdl_trigger();   // every load of this CTA is issued: the next kernel may be scheduled
      if (p.wait_stats && leader)
        atomicAdd(p.wait_stats + ws_class(1, EPI, TWO_PHASE) * WS_FIELDS + WS_STAGE, (unsigned long long)ws_stage);
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      long long ws_stage = 0;
      for (int w = cluster; w < total && ok; w += clusters) {
        const Work wk = decode_pair(p, w);
        const int my_row0 = wk.row0 + 128 * (int)rank;
        for (int kb = 0; kb < wk.nkb; ++kb) {
          const long long ws0 = ws_clock();
          const bool free_stage = wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.limit_ns, p.status, 111);
          ws_stage += ws_clock() - ws0;
          if (!free_stage) {
            ok = false;
            break;
          }
          if (leader) mbar_expect_tx(full_bar(stage), 2 * S::STAGE_BYTES);
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t sa = sbase + stage * S::STAGE_BYTES;
          const uint32_t sb = sa + S::A_BYTES;
          const int ph = TWO_PHASE ? (kb >= p.nk ? 1 : 0) : 0;
          const int k0 = (kb - ph * p.nk) * GEMM_BK;
          tma_load_2d_pair(sa, ph ? &ta1 : &ta0, fb, k0, my_row0);
          if constexpr (DUAL_B) {
            tma_load_3d_pair(sb, rank ? &tb1 : &tb0, fb, k0, wk.nt * 128, wk.e);       // gate | up half
          } else if constexpr (!B_MN) {
            tma_load_3d_pair(sb, ph ? &tb1 : &tb0, fb, k0, wk.nt * BN + 128 * (int)rank, wk.e);
          } else {
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_load_3d_pair(sb + b * 8192, ph ? &tb1 : &tb0, fb, wk.nt * BN + 64 * (2 * (int)rank + b), k0, wk.e);
          }
          if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      pdl_trigger();   // every load of this CTA is issued: the next kernel may be scheduled
      if (p.wait_stats && leader)
        atomicAdd(p.wait_stats + ws_class(1, EPI, TWO_PHASE) * WS_FIELDS + WS_STAGE, (unsigned long long)ws_stage);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA only)
    if (leader) {
      constexpr uint32_t idesc = instr_desc_bf16(256, BN, false, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      const long long ws_start = ws_clock();
      long long ws_operands = 0, ws_accum = 0, ws_kblocks = 0;
      for (int w = cluster; w < total && ok; w += clusters, ++it) {
        const Work wk = decode_pair(p, w);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        int good = 1;
        const long long ws0 = ws_clock();
        if (lane == 0) good = wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.limit_ns, p.status, 112);
        ws_accum += ws_clock() - ws0;
        ws_kblocks += wk.nkb;
        if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tacc = tmem_base + acc * BN;
        for (int kb = 0; kb < wk.nkb; ++kb) {
          const long long ws1 = ws_clock();
          if (lane == 0) good = wait_bounded(full_bar(stage), phase, abort_flag, p.limit_ns, p.status, 113);
          ws_operands += ws_clock() - ws1;
          if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = sbase + stage * S::STAGE_BYTES;
          const uint32_t sb = sa + S::A_BYTES;
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < GEMM_BK / 16; ++kk) {
              const uint64_t ad = smem_desc_sw128(sa + kk * 32, 0, 1024);
              const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                       : smem_desc_sw128(sb + kk * 32, 0, 1024);
              tc_mma_pair(tacc, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit_pair(empty_bar(stage), 0x3);
          }
          __syncwarp();
          if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) tc_commit_pair(tfull_bar(acc), 0x3);
        __syncwarp();
      }
      if (lane == 0) {
        tc_commit_pair(drain_bar, 0x1);
        volatile int no_abort = 0;
        wait_bounded(drain_bar, 0, &no_abort, p.limit_ns, nullptr, 0);
        if (p.wait_stats) {
          unsigned long long* c = p.wait_stats + ws_class(1, EPI, TWO_PHASE) * WS_FIELDS;
          atomicAdd(c + WS_CTAS, 1ull);
          atomicAdd(c + WS_LIFE, (unsigned long long)(ws_clock() - ws_start));
          atomicAdd(c + WS_OPERANDS, (unsigned long long)ws_operands);
          atomicAdd(c + WS_ACCUM, (unsigned long long)ws_accum);
          atomicAdd(c + WS_KBLOCKS, (unsigned long long)ws_kblocks);
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int it = 0;
    for (int w = cluster; w < total; w += clusters, ++it) {
      const Work wk = decode_pair(p, w);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      int good = 1;
      if (lane == 0) good = wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.limit_ns, p.status, 114);
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
      tc_fence_after();
      const int my_rows = max(0, min(128, wk.rows - 128 * (int)rank));
      epilogue_rows<EPI, BN>(p, wk.row0 + 128 * (int)rank, my_rows, wk.nt, wk.e, tmem_base + lane_off + acc * BN,
                             r, half);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar(acc));
        else mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      }
    }
  }

  tc_fence_before();
  cluster_sync();                                // no CTA leaves while its peer may still signal it
  tc_fence_after();
  if (warp == 1) tc_dealloc_pair(tmem_base, S::TMEM_COLS);
  if (p.pdl_late) pdl_wait();
}

template <int EPI, bool B_MN, bool DUAL_B, bool TWO_PHASE, int GATH = 0>
cudaError_t launch_pair_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                             const CUtensorMap& b1, const GemmParams& p, int num_sms, cudaStream_t s) {
  auto kern = grouped_gemm_pair_kernel<EPI, B_MN, DUAL_B, TWO_PHASE, GATH>;
  GemmParams q = p;
  q.nk_total = TWO_PHASE ? 2 * p.nk : p.nk;
  if (launch_chain_mode() < MOE_CHAIN_LATE) q.pdl_late = q.trigger_early = 0;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PairSmem::TOTAL);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_sms & ~1));
  cfg.blockDim = dim3(gemm_threads(EPI));
  cfg.dynamicSmemBytes = PairSmem::TOTAL;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = launch_chain_mode() >= MOE_CHAIN_EARLY ? 2 : 1;   // the cluster attribute comes first
  err = cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, q);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace moe
