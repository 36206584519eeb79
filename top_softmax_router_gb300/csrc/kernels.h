// Internal launch interface between the ABI layer (moe_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Per-call chunk plan arrays, all in the workspace (device pointers).
struct PlanPtrs {
  int* expert_off;    // [K][E+1]
  int* row_route;     // [K][kc_max]
  int* row_of;        // [N*k]
  int2* tiles;        // [K][T_max]
  int* tile_count;    // [K]
  int* active;        // [K][E]
  int* active_count;  // [K]
  int* first_touch;   // [E]
  int N, E, k, K, c_eff, kc_max, T_max;
};

// router
cudaError_t launch_router_logits(const uint16_t* X, const float* Wr, const float* bias, float* logits, int N,
                                 int H, int E, cudaStream_t s);
cudaError_t launch_router_topk(const float* logits, int32_t* idx, float* gates, int N, int E, int k, int* status,
                               cudaStream_t s);
// permutation
cudaError_t launch_plan(const int32_t* topk_idx, const PlanPtrs& p, int* status, cudaStream_t s);
cudaError_t launch_first_touch(const PlanPtrs& p, cudaStream_t s);
// data movement
cudaError_t launch_gather(const uint16_t* src, uint16_t* dst, const int* row_route, int rows, int H, int k,
                          cudaStream_t s);
cudaError_t launch_combine(const uint16_t* Op, const float* gates, const int* row_of, uint16_t* Y, int chunk,
                           int K, int n_i, int H, int k, cudaStream_t s);
cudaError_t launch_unpermute(const uint16_t* dXp, const float* dgp, int dgp_tiles, const float* gates,
                             const int* row_of, const int32_t* topk_idx, const float* Wr, uint16_t* dX,
                             float* dgates, float* dlogit, int chunk, int K, int n_i, int H, int k, int E,
                             cudaStream_t s);
cudaError_t launch_router_dw(const uint16_t* X, const float* dlogit, const int* row_route, const int* active,
                             const int* active_count, const int* expert_off, const int* first_touch, float* dWr,
                             int chunk, int E, int H, int k, cudaStream_t s);
cudaError_t launch_zero_untouched(const int* first_touch, float* dWg, float* dWu, float* dWd, float* dWr, int E,
                                  int H, int I, cudaStream_t s);
cudaError_t launch_diag_wait(int* status, int64_t limit_ns, cudaStream_t s);

// grouped GEMMs (gemm_fwd.cu / gemm_bwd.cu).  `rows` = permuted rows of the chunk.
struct ChunkGemm {
  const int2* tiles;
  const int* tile_count;
  const int* active;
  const int* active_count;
  const int* expert_off;
  const int* row_route;
  int rows;
  int chunk;
  int E, H, I;
  int num_sms;
  int* status;
  int64_t limit_ns;
};
// act = silu(Xp Wg^T) * (Xp Wu^T)
cudaError_t gemm_gateup_fwd(const ChunkGemm& c, const uint16_t* Xp, const uint16_t* Wg, const uint16_t* Wu,
                            uint16_t* act, cudaStream_t s);
// Op = act Wd^T
cudaError_t gemm_down(const ChunkGemm& c, const uint16_t* act, const uint16_t* Wd, uint16_t* Op, cudaStream_t s);
// gate = Xp Wg^T, up = Xp Wu^T (bf16)
cudaError_t gemm_gateup_bwd(const ChunkGemm& c, const uint16_t* Xp, const uint16_t* Wg, const uint16_t* Wu,
                            uint16_t* gate, uint16_t* up, cudaStream_t s);
// dActU = dYp Wd, fused SwiGLU backward epilogue (gate -> dGate, up -> dUp in place; gact; dgp)
cudaError_t gemm_dact(const ChunkGemm& c, const uint16_t* dYp, const uint16_t* Wd, const float* gates,
                      uint16_t* gate, uint16_t* up, uint16_t* gact, float* dgp, cudaStream_t s);
// dWd_e (+)= dYp_e^T gact_e
cudaError_t gemm_dwd(const ChunkGemm& c, const uint16_t* dYp, const uint16_t* gact, const int* first_touch,
                     float* dWd, cudaStream_t s);
// dWg_e (+)= dGate_e^T Xp_e ; dWu_e (+)= dUp_e^T Xp_e
cudaError_t gemm_dwgu(const ChunkGemm& c, const uint16_t* dGate, const uint16_t* dUp, const uint16_t* Xp,
                      const int* first_touch, float* dWg, float* dWu, cudaStream_t s);
// dXp = dGate Wg_e + dUp Wu_e
cudaError_t gemm_dx(const ChunkGemm& c, const uint16_t* dGate, const uint16_t* dUp, const uint16_t* Wg,
                    const uint16_t* Wu, uint16_t* dXp, cudaStream_t s);

constexpr int DACT_BN = 256;   // N tile of the dActU GEMM
constexpr int DACT_SPLIT = 2;  // epilogue warps per TMEM lane quarter in the dActU GEMM
// dgate partial sums per row: DACT_SPLIT per 256-column tile, summed in index order
inline int dgate_partials(int I) { return (I + DACT_BN - 1) / DACT_BN * DACT_SPLIT; }

// tensor maps (tma.cu)
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows);
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
                 uint32_t box_inner, uint32_t box_rows);
bool make_map_3d_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
                     uint32_t box_inner, uint32_t box_rows);

}  // namespace moe
