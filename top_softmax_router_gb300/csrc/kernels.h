// Internal launch interface between the ABI layer (moe_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <functional>

namespace moe {

// Per-call chunk plan arrays, all in the workspace (device pointers).
struct PlanPtrs {
  int* expert_off;    // [K][E+1]
  int* row_route;     // [K][kc_max]
  int* row_of;        // [N*k]
  int2* tiles;        // [K][T_max]    128-row tiles of one expert
  int* tile_count;    // [K]
  int2* tiles2;       // [K][T2_max]   256-row tiles of one expert (CTA-pair GEMMs)
  int* tile2_count;   // [K]
  int* active;        // [K][E]
  int* active_count;  // [K]
  int* first_touch;   // [E]
  int* block_counts;  // [count_blocks][E] scratch of the multi-block plan (K = 1), or NULL
  int count_blocks;   // blocks of the multi-block plan (0 or 1: one block per chunk)
  int N, E, k, K, c_eff, kc_max, T_max, T2_max;
};
// The multi-block plan of one chunk of kc routes: blocks of plan_per_block(kc) routes (a multiple of
// 1024, so each of a block's 32 warps takes a multiple of 32), at most 1024 blocks; none below 8192
// routes (one block plans the chunk).
inline int64_t plan_per_block(int64_t kc) {
  const int64_t b = (kc + 1023) / 1024 < 1024 ? (kc + 1023) / 1024 : 1024;
  return ((kc + b - 1) / b + 1023) / 1024 * 1024;
}
inline int plan_count_blocks(int64_t kc) {
  if (kc < 8192) return 0;
  return (int)((kc + plan_per_block(kc) - 1) / plan_per_block(kc));
}

// router
cudaError_t launch_router_logits(const uint16_t* X, const float* Wr, const float* bias, float* logits, int N,
                                 int H, int E, cudaStream_t s);
cudaError_t launch_router_topk(const float* logits, int32_t* idx, float* gates, int N, int E, int k, int* status,
                               cudaStream_t s);
// permutation
cudaError_t launch_plan(const int32_t* topk_idx, const PlanPtrs& p, int* status, cudaStream_t s);
cudaError_t launch_first_touch(const PlanPtrs& p, cudaStream_t s);
// data movement
// Dispatch gather into a permuted buffer (MOE_DISPATCH_GATHER; with MOE_DISPATCH_ON_LOAD the GEMMs gather
// their rows themselves and these kernels do not run).
// late: the gather overlaps the kernel before it in the stream (which must neither read nor write dst, and
// whose own predecessors must have finished with dst); one block waits for that kernel before the
// gather completes, so whatever follows in the stream sees both complete.
cudaError_t launch_gather(const uint16_t* src, uint16_t* dst, const int* row_route, int rows, int H, int k,
                          cudaStream_t s, bool late = false);
cudaError_t launch_combine(const uint16_t* Op, const float* gates, const int* row_of, uint16_t* Y, int chunk,
                           int K, int n_i, int H, int k, cudaStream_t s);
// Router backward of chunk `chunk`, per route: dg = the dActU partials of its row summed in index order;
// dl = g (dg - sum over the token's slots of g dg); writes dgates (optional), dlogit and dl_row[row].
cudaError_t launch_route_grad(const float* dgp, int dgp_tiles, const float* gates, const int* row_of, float* dgates,
                              float* dlogit, float* dl_row, int chunk, int K, int n_i, int k, cudaStream_t s);
// dX[t] = bf16(sum over the token's slots, in slot order, of dXp[row_of(t, j)]) (fp32)
cudaError_t launch_unpermute(const uint16_t* dXp, const int* row_of, uint16_t* dX, int chunk, int K, int n_i, int H,
                             int k, cudaStream_t s);
// Router weight gradient of one chunk over its tile list (at most max_tiles entries); partial is
// scratch of max_tiles * H floats.
cudaError_t launch_router_dw(const uint16_t* X, const float* dlogit, const int* row_route, const int2* tiles,
                             const int* tile_count, int max_tiles, const int* active, const int* active_count,
                             const int* first_touch, float* partial, float* dWr, int chunk, int E, int H, int k,
                             cudaStream_t s);
cudaError_t launch_zero_untouched(const int* first_touch, float* dWg, float* dWu, float* dWd, float* dWr, int E,
                                  int H, int I, cudaStream_t s);
cudaError_t launch_diag_wait(int* status, int64_t limit_ns, cudaStream_t s);

// grouped GEMMs (gemm_fwd.cu / gemm_bwd.cu).  `rows` = permuted rows of the chunk.
struct ChunkGemm {
  const int2* tiles;
  const int* tile_count;
  const int2* tiles2;
  const int* tile2_count;
  const int* active;
  const int* active_count;
  const int* expert_off;
  const int* row_route;   // permuted row -> route id t*k + j (the gathered operands read token t)
  int rows;
  int chunk;
  int N, k;               // tokens and routes per token of the token-major sources (X, dY)
  bool on_load;           // the operands below named Xp / dYp are gathered on load from X / dY (GATH
                          // kernels); otherwise they are permuted buffers [rows, H] filled by a gather kernel
  int E, H, I;
  bool pair;          // run the row-tile GEMMs on CTA pairs (2-SM MMA, 256-row tiles)
  int* work_ctr;      // GEMM_CTR_SLOTS zeroed work counters of this chunk (or hop); NULL = static schedule
  // Launch chaining (programmatic dependent launch; see GemmParams::pdl_late / trigger_early)
  bool late_wait;     // the GEMM overlaps the kernel before it in the stream and waits for it at its end
  bool trigger_early; // release the next kernel in the stream right after this one's dependency wait
  int num_sms;
  int* status;
  int64_t limit_ns;
};
// Wait-accounting counters of a diagnostic build (moe_diag_gemm_wait_stats), or NULL.
unsigned long long* gemm_wait_stats_buffer();
// Work-counter slot of each GEMM within a chunk (or hop).
enum : int {
  GEMM_CTR_GATEUP_FWD = 0, GEMM_CTR_DOWN, GEMM_CTR_GATEUP_BWD, GEMM_CTR_DACT, GEMM_CTR_DWD, GEMM_CTR_DWGU,
  GEMM_CTR_DX, GEMM_CTR_SLOTS = 8
};
// Xp and dYp below are the chunk's (or hop's) permuted rows of X and dY: row r is row token(r) of X [N, H]
// or dY [N, H].  With ChunkGemm::on_load the pointer passed for them is X or dY itself and the GEMM
// gathers those rows on load; otherwise it is the permuted buffer [rows, H] a gather kernel filled.
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
// dXp = dGate Wg_e + dUp Wu_e, plus, when dl is not NULL, each row's router-path term dl[r] Wr[e] (fp32, before
// the bf16 store)
cudaError_t gemm_dx(const ChunkGemm& c, const uint16_t* dGate, const uint16_t* dUp, const uint16_t* Wg,
                    const uint16_t* Wu, const float* dl, const float* Wr, uint16_t* dXp, cudaStream_t s);

constexpr int DACT_BN = 256;   // N tile of the dActU GEMM
constexpr int DACT_SPLIT = 2;  // epilogue warps per TMEM lane quarter in the dActU GEMM
// dgate partial sums per row: DACT_SPLIT per 256-column tile, summed in index order
inline int dgate_partials(int I) { return (I + DACT_BN - 1) / DACT_BN * DACT_SPLIT; }

// expert-partition ("hop") schedule (hops.cu).  Arrays of the current hop, in the workspace.
struct HopPtrs {
  int2* tiles;         // [cap/128 + E] tile list, rows rebased to the hop
  int* tile_count;     // [1]
  int2* tiles2;        // [cap/256 + E] 256-row tile list
  int* tile2_count;    // [1]
  int* active;         // [E] experts of the hop with rows
  int* active_count;   // [1]
  int* expert_off;     // [E+1] rebased offsets (entries e0..e1 meaningful)
  int* first_touch;    // [E] hop index of expert e, or -1 (shared by all hops; written by the hop plan)
  int* row_route;      // [cap] route id of each hop row
  int* base;           // [1] first global row of the hop
  int* rows;           // [1] rows of the hop (0 if it did not fit)
};
// The plan arrays of all P hops: hop h's arrays start h strides after hop 0's (the one-element arrays
// tile_count .. rows have stride 1; first_touch is shared).
struct HopSets {
  HopPtrs h0;
  int64_t s_tiles, s_tiles2, s_active, s_expert_off, s_row_route;
};
__host__ __device__ inline HopPtrs hop_set(const HopSets& S, int h) {
  HopPtrs p = S.h0;
  p.tiles += h * S.s_tiles;
  p.tile_count += h;
  p.tiles2 += h * S.s_tiles2;
  p.tile2_count += h;
  p.active += h * S.s_active;
  p.active_count += h;
  p.expert_off += h * S.s_expert_off;
  p.row_route += h * S.s_row_route;
  p.base += h;
  p.rows += h;
  return p;
}
// Plans every hop at once (one block per hop): hop h holds experts [h E / P, (h+1) E / P).
cudaError_t launch_hop_plan_all(const int* expert_off_g, const int* row_route_g, const HopSets& S, int P, int E,
                                int cap, int* status, cudaStream_t s);
// late: as for launch_gather
cudaError_t launch_gather_dev(const uint16_t* src, uint16_t* dst, const int* row_route, const int* rows_dev, int cap,
                              int H, int k, cudaStream_t s, bool late = false);
cudaError_t launch_combine_hop(const uint16_t* Op, const float* gates, const int* row_of_g, const int32_t* topk_idx,
                               const int* hop_base, const int* hop_rows, int e0, int e1, float* Yacc, int N, int H,
                               int k, cudaStream_t s);
cudaError_t launch_to_bf16(const float* in, uint16_t* out, int64_t n, cudaStream_t s);
cudaError_t launch_unpermute_hop(const uint16_t* dXp, const float* dgp, int dgp_tiles, const int* row_of_g,
                                 const int32_t* topk_idx, const int* hop_base, const int* hop_rows, int e0, int e1,
                                 float* dXacc, float* dg_route, int N, int H, int k, cudaStream_t s);
cudaError_t launch_router_final(const float* dXacc, const float* dg_route, const float* gates, const int32_t* topk_idx,
                                const float* Wr, uint16_t* dX, float* dgates, float* dlogit, int N, int H, int k,
                                int E, cudaStream_t s);

// tensor maps (tma.cu)
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows);
// bf16 rows of `inner` valid elements, `row_stride` elements apart
bool make_map_2d_strided(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                         uint32_t box_inner, uint32_t box_rows);
// Row gathers (tile::gather4): bf16 [rows][inner], box of 64 elements x 1 row, 128-byte swizzle.
bool make_map_gather(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows);
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
                 uint32_t box_inner, uint32_t box_rows);
bool make_map_3d_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t depth,
                     uint32_t box_inner, uint32_t box_rows);

// helpers of the ABI layer (moe_api.cu) shared with the optimizer step (adamw.cu)
int record_cuda_error(cudaError_t e, const char* what);  // keeps the message for moe_strerror; MOE_ERR_CUDA
int device_sm_count();                                    // SMs of the current device
int64_t wait_limit_ns();                                  // moe_set_wait_limit_ns's value
// Runs one launch on `s`, bracketed by profiling events of class `kind` when profiling is on.
int timed_launch(int kind, const char* what, cudaStream_t s, const std::function<cudaError_t()>& f);

// fused AdamW update (adamw.cu)
struct AdamConst {
  float decay;         // 1 - lr * weight_decay
  float beta1, omb1;   // beta1, 1 - beta1
  float beta2, omb2;   // beta2, 1 - beta2
  float step_size;     // lr / (1 - beta1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
  float eps;
};

}  // namespace moe
