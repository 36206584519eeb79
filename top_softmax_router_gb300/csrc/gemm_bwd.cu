// Backward grouped GEMMs (per-chunk recompute, dActU, dX) of the expert FFN.
#include "gemm_launch.cuh"

namespace moe {

// Recompute: gate = Xp Wg_e^T, up = Xp Wu_e^T (bf16); Xp as in gemm_gateup_fwd.
cudaError_t gemm_gateup_bwd(const ChunkGemm& c, const uint16_t* Xp, const uint16_t* Wg, const uint16_t* Wu,
                            uint16_t* gate, uint16_t* up, cudaStream_t s) {
  CUtensorMap a, bg, bu;
  if (!(c.on_load ? make_map_gather(&a, Xp, c.H, c.N) : make_map_2d(&a, Xp, c.H, c.rows, 64, 128)) ||
      !make_map_3d(&bg, Wg, c.H, c.I, c.E, 64, 128) ||
      !make_map_3d(&bu, Wu, c.H, c.I, c.E, 64, 128))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_GATEUP_BWD);
  p.nk = c.H / GEMM_BK;
  p.n_tiles = (c.I + 127) / 128;
  p.N = c.I;
  p.ldo = c.I;
  p.out0 = gate;
  p.out1 = up;
  if (c.on_load) {
    if (c.pair) return launch_pair_gemm<EPI_GATEUP, false, true, false, 1>(a, a, bg, bu, p, c.num_sms, s);
    return launch_grouped_gemm<EPI_GATEUP, false, false, false, 256, true, false, 1>(a, a, bg, bu, p, c.num_sms, s);
  }
  if (c.pair) return launch_pair_gemm<EPI_GATEUP, false, true, false>(a, a, bg, bu, p, c.num_sms, s);
  return launch_grouped_gemm<EPI_GATEUP, false, false, false, 256, true, false>(a, a, bg, bu, p, c.num_sms, s);
}

// dActU[r, i] = dYp[r] . Wd_e[:, i]; A = dYp [rows, H] K-major (or, on_load, gathered from dY); B = Wd_e
// [H (K), I (N)] MN-major.
cudaError_t gemm_dact(const ChunkGemm& c, const uint16_t* dYp, const uint16_t* Wd, const float* gates,
                      uint16_t* gate, uint16_t* up, uint16_t* gact, float* dgp, cudaStream_t s) {
  CUtensorMap a, b;
  if (!(c.on_load ? make_map_gather(&a, dYp, c.H, c.N) : make_map_2d(&a, dYp, c.H, c.rows, 64, 128)) ||
      !make_map_3d(&b, Wd, c.I, c.H, c.E, 64, 64))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_DACT);
  p.nk = c.H / GEMM_BK;
  p.n_tiles = (c.I + DACT_BN - 1) / DACT_BN;
  p.N = c.I;
  p.ldo = c.I;
  p.out0 = gate;
  p.out1 = up;
  p.out2 = gact;
  p.gates = gates;
  p.dgp = dgp;
  static_assert(gemm_epi_warps(EPI_DACT) / 4 == DACT_SPLIT, "dgate partial layout");
  if (c.on_load) {
    if (c.pair) return launch_pair_gemm<EPI_DACT, true, false, false, 1>(a, a, b, b, p, c.num_sms, s);
    return launch_grouped_gemm<EPI_DACT, false, true, false, DACT_BN, false, false, 1>(a, a, b, b, p, c.num_sms, s);
  }
  if (c.pair) return launch_pair_gemm<EPI_DACT, true, false, false>(a, a, b, b, p, c.num_sms, s);
  return launch_grouped_gemm<EPI_DACT, false, true, false, DACT_BN, false, false>(a, a, b, b, p, c.num_sms, s);
}

// dXp[r, h] = dGate[r] . Wg_e[:, h] + dUp[r] . Wu_e[:, h] (+ dl[r] Wr[e, h] when dl is given); K runs over I
// twice.  A = dGate / dUp [rows, I] K-major; B = Wg_e / Wu_e [I (K), H (N)] MN-major.
cudaError_t gemm_dx(const ChunkGemm& c, const uint16_t* dGate, const uint16_t* dUp, const uint16_t* Wg,
                    const uint16_t* Wu, const float* dl, const float* Wr, uint16_t* dXp, cudaStream_t s) {
  CUtensorMap a0, a1, b0, b1;
  if (!make_map_2d(&a0, dGate, c.I, c.rows, 64, 128) || !make_map_2d(&a1, dUp, c.I, c.rows, 64, 128) ||
      !make_map_3d(&b0, Wg, c.H, c.I, c.E, 64, 64) || !make_map_3d(&b1, Wu, c.H, c.I, c.E, 64, 64))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_DX);
  p.nk = c.I / GEMM_BK;
  p.n_tiles = (c.H + 255) / 256;
  p.N = c.H;
  p.ldo = c.H;
  p.out0 = dXp;
  p.rt_dl = dl;
  p.rt_w = Wr;
  if (c.pair) return launch_pair_gemm<EPI_STORE, true, false, true>(a0, a1, b0, b1, p, c.num_sms, s);
  return launch_grouped_gemm<EPI_STORE, false, true, false, 256, false, true>(a0, a1, b0, b1, p, c.num_sms, s);
}

}  // namespace moe
