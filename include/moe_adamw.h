/*
 * moe_adamw.h -- C ABI of libmoe.so, part 2: the offloaded optimizer step
 * (OffloadStreamAdamW) on one GB300 GPU.
 *
 * Source: "bounded-streaming operators" summary, Methodology 4
 * (OffloadStreamAdamW), eq. (5).  The fp32 optimizer state (master weights
 * and the two Adam moments) stays in host memory.  It is cut into buckets of
 * at most `bucket` parameters, which rotate through `slots` device staging
 * slots on three streams: (i) host-to-device copy of the bucket's state,
 * (ii) a fused AdamW update that also writes the bf16 working weights, and
 * (iii) device-to-host write-back of the updated state.  The device holds
 * O(slots * bucket) bytes of state at any time (eq. (5), M_stage); the step
 * takes about G * max(T_H2D, T_update, T_D2H) for G buckets.  The floor is the
 * host-link round trip of the state, 12 bytes per parameter each way.
 *
 * The update (the pages name AdamW and give no formula; this is AdamW with
 * decoupled weight decay, Loshchilov and Hutter 2019), for step count t >= 1:
 *     p <- p * (1 - lr * weight_decay)
 *     m <- beta1 * m + (1 - beta1) * g
 *     v <- beta2 * v + (1 - beta2) * g * g
 *     p <- p - (lr / (1 - beta1^t)) * m / (sqrt(v) / sqrt(1 - beta2^t) + eps)
 *     w <- bf16(p), rounded to nearest even
 * in fp32 on the device (the bias corrections are formed on the host in
 * double and passed as fp32).  Every parameter is independent, so the
 * bucketing changes no result: every (bucket, slots) choice gives the same
 * bits as every other and as moe_adamw_step.
 *
 * Conventions are those of moe.h (return codes MOE_OK / MOE_ERR_*, stream
 * passed as void*, calls asynchronous, no exception crosses the ABI, the
 * caller owns every buffer), with these additions:
 *   - "host" arrays are page-locked host memory (cudaHostAlloc,
 *     cudaHostRegister, or torch's pin_memory); pageable memory is rejected
 *     with MOE_ERR_INVALID_ARG.  The state arrays must stay untouched by the
 *     host until the stream has passed the call (the write-back is
 *     asynchronous).
 *   - Every array is 16-byte aligned; `bucket` is a multiple of 4.
 *   - The offloaded step runs on three streams the library owns (one set per
 *     host thread and device).  They start after the work already enqueued on
 *     `stream`, and `stream` waits for their last copy before its next work,
 *     so the call behaves as if it ran on `stream`.
 */
#ifndef TOP_SOFTMAX_ROUTER_MOE_ADAMW_H_
#define TOP_SOFTMAX_ROUTER_MOE_ADAMW_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Hyper-parameters of one step.  `step` is t >= 1, the count including this
 * step.  0 <= beta1, beta2 < 1; eps > 0 (eps = 0 is accepted; the update of
 * an element with m = v = 0 is then NaN, as in the formula). */
typedef struct moe_adamw_hparams {
  double lr, beta1, beta2, eps, weight_decay;
  int64_t step;
} moe_adamw_hparams;

/* Element type of the gradient array. */
enum { MOE_GRAD_F32 = 0, MOE_GRAD_BF16 = 1 };

/* Most staging slots one offloaded step may use. */
#define MOE_ADAMW_MAX_SLOTS 16

/* Device bytes of the staging buffer for `slots` slots of `bucket`
 * parameters: slots * 3 * (bucket * 4 rounded up to 256).  Errors:
 * MOE_ERR_INVALID_ARG for bucket < 4, bucket not a multiple of 4, slots
 * outside 1..MOE_ADAMW_MAX_SLOTS, or NULL `bytes`. */
int moe_adamw_staging_bytes(int64_t bucket, int32_t slots, size_t* bytes);

/* The offloaded step of eq. (5).
 *   n            parameters (n >= 0; n = 0 enqueues nothing)
 *   bucket       beta of eq. (5): parameters per bucket (multiple of 4)
 *   slots        s of eq. (5): staging slots, 1..MOE_ADAMW_MAX_SLOTS
 *                (slots = 1 serialises copy, update and write-back)
 *   master       [n] fp32 host (page-locked)   in/out: master weights p
 *   exp_avg      [n] fp32 host (page-locked)   in/out: first moment m
 *   exp_avg_sq   [n] fp32 host (page-locked)   in/out: second moment v
 *   grad         [n] device, fp32 or bf16 (grad_dtype)   in: gradient g
 *   weight       [n] bf16 device               out: working weights bf16(p)
 *   staging      device buffer of at least moe_adamw_staging_bytes(bucket, slots)
 * Bucket b (0-based) covers parameters [b*bucket, min((b+1)*bucket, n)) and
 * uses slot b mod slots; its host-to-device copy waits until the write-back
 * of bucket b - slots has left that slot.
 * Errors: MOE_ERR_INVALID_ARG (NULL or misaligned pointer, pageable host
 * state, device memory passed as host state, bad bucket, slots or grad_dtype,
 * negative n, bad hyper-parameters), MOE_ERR_WORKSPACE_TOO_SMALL (staging),
 * MOE_ERR_CUDA (a copy, launch or event call failed; the streams may then
 * hold part of the step). */
int moe_adamw_offload_step(const moe_adamw_hparams* hp, int64_t n, int64_t bucket, int32_t slots,
                           float* master, float* exp_avg, float* exp_avg_sq, const void* grad,
                           int32_t grad_dtype, uint16_t* weight, void* staging, size_t staging_bytes,
                           void* stream);

/* The same update as one fused kernel on `stream`, in place, on state the
 * device addresses directly: device memory (the update alone, state resident
 * in HBM), or page-locked host memory, which the kernel then reads and writes
 * across the host link with no staging copy (the pages' schedule needs the
 * copy engines; on a GB300 the GPU can address host memory coherently, and
 * this call is that alternative).  Arguments as moe_adamw_offload_step; the
 * three state arrays must all be device memory or all be page-locked host
 * memory.  Errors as moe_adamw_offload_step. */
int moe_adamw_step(const moe_adamw_hparams* hp, int64_t n, float* master, float* exp_avg,
                   float* exp_avg_sq, const void* grad, int32_t grad_dtype, uint16_t* weight,
                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TOP_SOFTMAX_ROUTER_MOE_ADAMW_H_ */
