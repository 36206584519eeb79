/*
 * CPU oracle -- router logits.  TEST INFRASTRUCTURE ONLY: only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load this.  It shares
 * no code with the CUDA path.
 *
 * Follows: RelayMoE summary, section 2.1 ("each token selects its top-k
 * experts"), and the workload text "router logits = X.W_r plus per-expert
 * bias ... softmax then top-k".
 *
 * The logit of token t for expert e is the fp32 dot product of X[t,:] (bf16,
 * widened exactly) and Wr[e,:] (fp32), accumulated as one fused-multiply-add
 * chain in increasing h from 0.0f, followed by one fp32 addition of bias[e].
 * That order is the contract that makes the top-k decision reproducible
 * bit for bit: the decision is taken in fp32 on both sides.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp (fmaf is the C99 correctly
 * rounded fused multiply-add).
 */
#include <math.h>
#include <stdint.h>

static inline float widen_bf16(uint16_t b) {
  union { uint32_t u; float f; } v;
  v.u = ((uint32_t)b) << 16;
  return v.f;
}

/* logits[r, e] for r in [0, rows): X holds `rows` token rows of length H. */
void oracle_router_logits(const uint16_t* X, const float* Wr, const float* bias,
                          int64_t rows, int64_t H, int64_t E, float* logits) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* x = X + r * H;
    for (int64_t e = 0; e < E; ++e) {
      const float* w = Wr + e * H;
      float acc = 0.0f;
      for (int64_t h = 0; h < H; ++h) acc = fmaf(widen_bf16(x[h]), w[h], acc);
      if (bias) acc = acc + bias[e];
      logits[r * E + e] = acc;
    }
  }
}
