// Weight-gradient grouped GEMMs: the contraction runs over each expert's rows
// in the chunk; results are stored on the expert's first chunk (in backward
// order) and added on later chunks, in a fixed chunk order.
#include "gemm_launch.cuh"

namespace moe {

// dWd_e[h, i] (+)= sum_r dYp[r, h] * gact[r, i].  A = dYp (MN-major over H; on_load, gathered from dY),
// B = gact (MN-major over I).
cudaError_t gemm_dwd(const ChunkGemm& c, const uint16_t* dYp, const uint16_t* gact, const int* first_touch,
                     float* dWd, cudaStream_t s) {
  CUtensorMap a, b, o;
  if (!(c.on_load ? make_map_gather(&a, dYp, c.H, c.N) : make_map_2d(&a, dYp, c.H, c.rows, 64, 64)) ||
      !make_map_2d(&b, gact, c.I, c.rows, 64, 64) ||
      !make_map_3d_f32(&o, dWd, c.I, c.H, c.E, 32, 32))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_DWD);
  p.m_tiles = (c.H + GEMM_BM - 1) / GEMM_BM;
  p.n_tiles = (c.I + 255) / 256;
  p.M = c.H;
  p.N = c.I;
  p.ldo = c.I;
  p.out0 = dWd;
  p.out1 = dWd;
  p.first_touch = first_touch;
  p.out_estride = (int64_t)c.H * c.I;
  if (c.on_load)
    return launch_grouped_gemm<EPI_DW, true, true, true, 256, false, false, 1>(a, a, b, b, p, c.num_sms, s, &o, &o);
  return launch_grouped_gemm<EPI_DW, true, true, true, 256, false, false>(a, a, b, b, p, c.num_sms, s, &o, &o);
}

// dWg_e[i, h] (+)= sum_r dGate[r, i] * Xp[r, h] and the same for dWu with dUp, in one launch; Xp is the B
// operand, MN-major over H (on_load, gathered from X).
cudaError_t gemm_dwgu(const ChunkGemm& c, const uint16_t* dGate, const uint16_t* dUp, const uint16_t* Xp,
                      const int* first_touch, float* dWg, float* dWu, cudaStream_t s) {
  CUtensorMap a0, a1, b, og, ou;
  if (!make_map_2d(&a0, dGate, c.I, c.rows, 64, 64) || !make_map_2d(&a1, dUp, c.I, c.rows, 64, 64) ||
      !(c.on_load ? make_map_gather(&b, Xp, c.H, c.N) : make_map_2d(&b, Xp, c.H, c.rows, 64, 64)) ||
      !make_map_3d_f32(&og, dWg, c.H, c.I, c.E, 32, 32) ||
      !make_map_3d_f32(&ou, dWu, c.H, c.I, c.E, 32, 32))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_DWGU);
  p.m_tiles = (c.I + GEMM_BM - 1) / GEMM_BM;
  p.n_tiles = (c.H + 255) / 256;
  p.n_problems = 2;
  p.M = c.I;
  p.N = c.H;
  p.ldo = c.H;
  p.out0 = dWg;
  p.out1 = dWu;
  p.first_touch = first_touch;
  p.out_estride = (int64_t)c.I * c.H;
  if (c.on_load)
    return launch_grouped_gemm<EPI_DW, true, true, true, 256, false, false, 2>(a0, a1, b, b, p, c.num_sms, s, &og,
                                                                                &ou);
  return launch_grouped_gemm<EPI_DW, true, true, true, 256, false, false>(a0, a1, b, b, p, c.num_sms, s, &og, &ou);
}

}  // namespace moe
