// Forward grouped GEMMs: gate/up with the SwiGLU epilogue, and the down projection.
#include "gemm_launch.cuh"

namespace moe {

// act[r, i] = silu(Xp[r] . Wg_e[i]) * (Xp[r] . Wu_e[i]) for the rows r of expert e.
// A = Xp [rows, H] K-major (or, on_load, gathered from X [N, H]); B tile = [128 rows of Wg_e ; 128 rows of
// Wu_e] K-major.
cudaError_t gemm_gateup_fwd(const ChunkGemm& c, const uint16_t* Xp, const uint16_t* Wg, const uint16_t* Wu,
                            uint16_t* act, cudaStream_t s) {
  CUtensorMap a, bg, bu;
  if (!(c.on_load ? make_map_gather(&a, Xp, c.H, c.N) : make_map_2d(&a, Xp, c.H, c.rows, 64, 128)) ||
      !make_map_3d(&bg, Wg, c.H, c.I, c.E, 64, 128) || !make_map_3d(&bu, Wu, c.H, c.I, c.E, 64, 128))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_GATEUP_FWD);
  p.nk = c.H / GEMM_BK;
  p.n_tiles = (c.I + 127) / 128;
  p.N = c.I;
  p.ldo = c.I;
  p.out0 = act;
  if (c.on_load) {
    if (c.pair) return launch_pair_gemm<EPI_SWIGLU, false, true, false, 1>(a, a, bg, bu, p, c.num_sms, s);
    return launch_grouped_gemm<EPI_SWIGLU, false, false, false, 256, true, false, 1>(a, a, bg, bu, p, c.num_sms, s);
  }
  if (c.pair) return launch_pair_gemm<EPI_SWIGLU, false, true, false>(a, a, bg, bu, p, c.num_sms, s);
  return launch_grouped_gemm<EPI_SWIGLU, false, false, false, 256, true, false>(a, a, bg, bu, p, c.num_sms, s);
}

// Op[r, h] = act[r] . Wd_e[h].  A = act [rows, I] K-major; B = Wd_e [H, I] K-major.
cudaError_t gemm_down(const ChunkGemm& c, const uint16_t* act, const uint16_t* Wd, uint16_t* Op, cudaStream_t s) {
  CUtensorMap a, b;
  // weight box: 256 rows for one CTA, 128 (one CTA's half) for a pair
  if (!make_map_2d(&a, act, c.I, c.rows, 64, 128) ||
      !make_map_3d(&b, Wd, c.I, c.H, c.E, 64, c.pair ? 128 : 256))
    return cudaErrorInvalidValue;
  GemmParams p = base_params(c, GEMM_CTR_DOWN);
  p.nk = c.I / GEMM_BK;
  p.n_tiles = (c.H + 255) / 256;
  p.N = c.H;
  p.ldo = c.H;
  p.out0 = Op;
  if (c.pair) return launch_pair_gemm<EPI_STORE, false, false, false>(a, a, b, b, p, c.num_sms, s);
  return launch_grouped_gemm<EPI_STORE, false, false, false, 256, false, false>(a, a, b, b, p, c.num_sms, s);
}

}  // namespace moe
