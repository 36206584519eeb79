/*
 * moe_ce.h -- C ABI of libmoe.so, part 3: the vocabulary-projection cross-entropy head with a
 * bounded logit working set, on one GB300 GPU.
 *
 * Sources (page title, then section / equation):
 *   - "bounded-streaming operators" summary, Methodology 2 (Ring-DTP): the tokens-by-vocabulary logit
 *     tensor is never formed whole; each round forms one logit strip of V/P classes, folds its
 *     partial normaliser into a running per-token state (max m, sum z, target logit) and releases
 *     the strip.  eq. (2): peak logit memory O(N V b / P).  eq. (3): the online-softmax recurrence
 *         m' = max(m, max_v y_v),   z' = exp(m - m') z + sum_v exp(y_v - m').
 *     On one device the ring's rounds become a loop over vocabulary strips (no exchange).
 *   - "Training Trillion-Parameter MoE ..." blog, section 3.5: vocabulary-axis chunking of the
 *     cross-entropy by a two-pass scan (global statistics first, then each shard's loss and
 *     gradients), numerically equivalent to the standard implementation.
 *
 * What is computed (X [N, H] bf16 hidden states, W [V, H] bf16 projection, t [N] classes):
 *     y[n, v] = X[n] . W[v]        (bf16 products, fp32 accumulation on the tensor cores)
 *     lse[n]  = log sum_v exp(y[n, v]),   loss[n] = lse[n] - y[n, t_n]
 *   and, for an upstream gradient g[n] of loss[n] (g[n] = 1/N for the mean loss),
 *     d[n, v] = g[n] (exp(y[n, v] - lse[n]) - [v = t_n])      (stored in bf16)
 *     dX[n]   = sum_v d[n, v] W[v]    (fp32 accumulation, stored bf16)
 *     dW[v]   = sum_n d[n, v] X[n]    (fp32)
 *
 * Schedule.  Forward: one persistent tcgen05 GEMM over all classes; each 128-token x 256-class logit
 * tile lives only in tensor memory, where the epilogue folds it into a per-(token, tile) (max, sum)
 * pair and picks out the target logit; a second kernel folds the pairs of each token, tile by tile
 * in class order, by eq. (3).  No logit is written to memory.  Backward (the two-pass scan: lse is
 * the first pass's result): the vocabulary is cut into P strips of ceil(ceil(V/P)/256)*256 classes;
 * for each strip the logits are recomputed, d is written for that strip only (N x strip bf16, the
 * eq. (2) working set), dX accumulates d W_strip in fp32 and dW_strip = d^T X is written.
 *
 * Conventions are those of moe.h (MOE_OK / MOE_ERR_* codes, stream as void*, asynchronous, the
 * caller owns every buffer and the workspace, 16-byte aligned pointers), and:
 *   - shapes: N >= 0; H a multiple of 64; V >= 1; 1 <= P <= V.  Else MOE_ERR_UNSUPPORTED_SHAPE.
 *   - a class outside [0, V) is reported as MOE_ERR_DEVICE_CHECK through the workspace status word
 *     (moe_check_status); its token then gets loss = lse and no target term.
 */
#ifndef TOP_SOFTMAX_ROUTER_MOE_CE_H_
#define TOP_SOFTMAX_ROUTER_MOE_CE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* N tokens of hidden size H, V classes, P vocabulary strips in the backward pass. */
typedef struct moe_ce_config {
  int32_t N, H, V, P;
} moe_ce_config;

/* Workspace bytes of moe_ce_forward and moe_ce_backward (either pointer may be NULL); a function of
 * the shape only.  The backward's largest part is one strip of d: N x strip x 2 bytes. */
int moe_ce_workspace_bytes(const moe_ce_config* cfg, size_t* fwd_bytes, size_t* bwd_bytes);

/* Forward.
 *   X       [N, H] bf16;  W [V, H] bf16;  targets [N] int32
 *   loss    [N] fp32 out: lse - y[target]
 *   lse     [N] fp32 out: log-sum-exp of each token's logits (the backward's input)
 *   loss_mean [1] fp32 out or NULL: sum_n loss[n] / N, summed in a fixed order */
int moe_ce_forward(const moe_ce_config* cfg, const uint16_t* X, const uint16_t* W, const int32_t* targets,
                   float* loss, float* lse, float* loss_mean, void* ws, size_t ws_bytes, void* stream);

/* Backward.
 *   X, W, targets as in the forward; lse [N] from the forward
 *   dloss   [N] fp32: gradient of each token's loss (1/N each for the mean)
 *   dX      [N, H] bf16 out (overwritten)
 *   dW      [V, H] fp32 out (overwritten) */
int moe_ce_backward(const moe_ce_config* cfg, const uint16_t* X, const uint16_t* W, const int32_t* targets,
                    const float* lse, const float* dloss, uint16_t* dX, float* dW, void* ws, size_t ws_bytes,
                    void* stream);

/* Statistics of the last successful moe_ce_* call on this host thread. */
typedef struct moe_ce_stats {
  int32_t strips;              /* strips the backward ran (ceil(V / strip)) */
  int32_t strip_classes;       /* classes per strip */
  int64_t strip_bytes;         /* bytes of d held at once: N * strip * 2 */
  int64_t strip_bound_bytes;   /* eq. (2) without its constant: N * ceil(V/P) * 2 */
  int64_t partial_bytes;       /* forward: the per-(token, tile) (max, sum) pairs, N * ceil(V/256) * 8 */
  int64_t workspace_bytes;     /* workspace the call used */
  int32_t kernel_launches;     /* kernels the call enqueued */
} moe_ce_stats;
int moe_ce_last_stats(moe_ce_stats* out);

#ifdef __cplusplus
}
#endif

#endif /* TOP_SOFTMAX_ROUTER_MOE_CE_H_ */
