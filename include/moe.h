/*
 * moe.h -- C ABI of libmoe.so: the chunk-bounded, top-k-softmax-routed
 * Mixture-of-Experts block on one GB300 GPU (sm_103a), forward and backward.
 *
 * The block (sources, by page title and section):
 *   - "bounded-streaming operators" summary, Methodology 1 (PipelinedLLEP),
 *     eq. (1): the N tokens are split into K = min(ceil(N/c), K_max) chunks,
 *     c_eff = ceil(N/K); chunk i holds token positions i, i+K, i+2K, ...
 *     (strided membership).  Each chunk's expert work is recomputed in the
 *     backward pass and released before the next chunk starts (nested
 *     per-chunk checkpoint), so the routed buffers stay within
 *     2 * k * c_eff * H * b bytes whatever the router does ("Memory bound").
 *   - RelayMoE summary, section 2.1: each token selects its top-k experts;
 *     tokens are expanded and permuted to their experts, run through the
 *     expert FFN, then returned and recombined with their gate weights;
 *     sections 1 and 3.1: dropless, padding-free expert compute.
 *   - "Training Trillion-Parameter MoE ..." blog, section 3.3: permute /
 *     unpermute and a grouped GEMM organised by expert-aggregated batches.
 *
 * Conventions for every call:
 *   - Tensors are dense, row-major, on the current CUDA device, with base
 *     pointers aligned to 16 bytes.  "bf16" arguments are uint16_t bit
 *     patterns of bfloat16 values.
 *   - The caller owns every buffer, the workspace and the stream.  The
 *     library allocates no device memory and keeps no device state between
 *     calls; it keeps only host-side statistics (moe_last_stats).  The one
 *     exception is moe_route_noalloc's fixed array, described at its
 *     declaration.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls enqueue kernels and return without synchronising the
 *     host.  Launch errors are returned at once (MOE_ERR_CUDA); errors found
 *     by a kernel (a wait that ran out of time, a bad expert id) are written
 *     to a status word in the workspace and read by moe_check_status.
 *   - moe_route, moe_plan, moe_forward, moe_backward and the hop-schedule calls may be captured
 *     into a CUDA graph (stream capture): they allocate nothing, read nothing back to the host and
 *     enqueue only stream-ordered work (the backward's side stream joins and leaves the capture
 *     through events).  Every launch reads its tile lists from device memory, so a replay after
 *     new input contents routes afresh.  Profiling (moe_profile_enable) must be off while capturing;
 *     moe_check_status synchronises and is not capturable.
 *   - Kernels are launched with programmatic stream serialization (programmatic
 *     dependent launch): a kernel may be scheduled while the previous one in the
 *     stream finishes, and it waits for that kernel before touching memory, so
 *     work the caller enqueues before or after a call is ordered as usual.
 *     Within a call, a few kernels that share no buffer with their predecessor
 *     run beside it and wait for it at their end instead.  moe_set_launch_chaining
 *     turns this off (early waits only) or returns to plain stream order.
 *   - Return codes: MOE_OK (0) or one of the negative MOE_ERR_* codes below.
 *     No C++ exception crosses this boundary.
 *   - Supported shapes: N >= 0; H and I multiples of 64; 1 <= E <= 1024;
 *     1 <= k <= min(E, 32); c >= 1; K_max >= 1.  Anything else returns
 *     MOE_ERR_UNSUPPORTED_SHAPE (or MOE_ERR_INVALID_ARG for negative sizes).
 */
#ifndef TOP_SOFTMAX_ROUTER_MOE_H_
#define TOP_SOFTMAX_ROUTER_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Block shape.  N tokens of hidden size H; E experts, top-k routing; SwiGLU
 * expert FFN of width I; token budget c per chunk and chunk cap K_max
 * (eq. (1) of the bounded-streaming summary). */
typedef struct moe_config {
  int32_t N, H, E, k, I, c, K_max;
} moe_config;

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,         /* NULL/misaligned pointer, negative size */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,   /* H or I not a multiple of 64, k > E, E > 1024, k > 32 */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3, /* ws_bytes below moe_workspace_bytes() */
  MOE_ERR_CUDA = -4,                /* a CUDA runtime call or launch failed; see moe_strerror */
  MOE_ERR_TIMEOUT = -5,             /* a device-side wait ran past its time limit */
  MOE_ERR_DEVICE_CHECK = -6,        /* a kernel found an out-of-range index (e.g. expert id >= E) */
  MOE_ERR_NOT_BUILT = -7            /* a diagnostic the library was built without */
};

/* Statistics of the most recent successful call on this host thread. */
typedef struct moe_stats {
  int32_t K;                       /* chunks, eq. (1) */
  int32_t c_eff;                   /* tokens per chunk (largest chunk), eq. (1) */
  int64_t routed_rows;             /* k * c_eff: permuted rows of the largest chunk */
  int64_t routed_bytes_peak;       /* bytes of H-wide routed buffers live at once */
  int64_t routed_bytes_bound;      /* 2 * k * c_eff * H * 2 ("Memory bound", E_p = 1, b = 2) */
  int64_t inter_bytes_peak;        /* bytes of I-wide expert intermediates live at once */
  int64_t inter_bytes_bound;       /* 3 * k * c_eff * I * 2 */
  int64_t workspace_bytes;         /* workspace bytes the call used */
  int32_t kernel_launches;         /* kernels the call enqueued */
} moe_stats;

/* Workspace sizes in bytes for each call (any argument may be NULL).  One
 * buffer of max(route, fwd, bwd) bytes serves all three calls.  The sizes
 * depend on the shape only, never on the routing (eq. (1): the bound holds
 * whatever the router does).  Returns MOE_OK or a shape error. */
int moe_workspace_bytes(const moe_config* cfg, size_t* route_bytes, size_t* fwd_bytes,
                        size_t* bwd_bytes);

/* Router: logits, top-k and gates (RelayMoE summary 2.1; workload text
 * "softmax then top-k, gates renormalised over top-k").
 *   X        [N, H] bf16      tokens
 *   Wr       [E, H] fp32      router weight (row e = expert e)
 *   bias     [E] fp32 or NULL added to every token's logits
 *   topk_idx [N, k] int32     out: expert ids by descending logit
 *   gates    [N, k] fp32      out: g_j = exp(l_j) / sum_{i<k} exp(l_i)
 * The logit of (t, e) is one fp32 fused-multiply-add chain over h = 0..H-1
 * starting from 0, then one fp32 addition of bias[e]; that fixed order makes
 * the top-k decision reproducible bit for bit.  Equal logits go to the lower
 * expert id.  NaN or infinite inputs are not supported. */
int moe_route(const moe_config* cfg, const uint16_t* X, const float* Wr, const float* bias,
              int32_t* topk_idx, float* gates, void* ws, size_t ws_bytes, void* stream);

/* The per-chunk permutation the forward and backward passes use, exported so
 * that it can be checked (RelayMoE summary 2.1: tokens are expanded and
 * permuted to experts; counting sort by expert id).
 *   topk_idx   [N, k] int32   in
 *   row_route  [K, k*c_eff]   out: for chunk i, row r of its permuted buffer
 *                             holds route t*k + j; rows of one expert are
 *                             contiguous, experts ascend, tokens ascend
 *                             within an expert; entries past chunk i's
 *                             k * n_i rows are left untouched.
 *   row_of     [N, k] int32   out: permuted row (within its chunk) of route (t, j)
 *   expert_off [K, E+1] int32 out: chunk i's rows of expert e are
 *                             expert_off[i][e] .. expert_off[i][e+1]-1
 * K and c_eff follow eq. (1); see moe_chunk_plan. */
int moe_plan(const moe_config* cfg, const int32_t* topk_idx, int32_t* row_route, int32_t* row_of,
             int32_t* expert_off, void* ws, size_t ws_bytes, void* stream);

/* K and c_eff of eq. (1) for this shape (host only, no GPU work). */
int moe_chunk_plan(const moe_config* cfg, int32_t* K, int32_t* c_eff);

/* Forward pass, chunk by chunk (bounded-streaming summary, Methodology 1).
 *   X [N,H] bf16; topk_idx [N,k] int32 and gates [N,k] fp32 from moe_route
 *   Wg, Wu [E, I, H] bf16   gate and up projections (row i of expert e)
 *   Wd     [E, H, I] bf16   down projection
 *   Y      [N, H] bf16      out: Y[t] = sum_j g[t,j] * FFN_{idx[t,j]}(X[t]),
 *                           FFN_e(x) = (silu(x Wg_e^T) * (x Wu_e^T)) Wd_e^T,
 *                           the sum over j taken in fp32 in slot order.
 * Every expert intermediate is stored in bf16 between the GEMMs.  Y is
 * identical bit for bit for every K (the chunking changes order only). */
int moe_forward(const moe_config* cfg, const uint16_t* X, const int32_t* topk_idx,
                const float* gates, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                uint16_t* Y, void* ws, size_t ws_bytes, void* stream);

/* Backward pass with per-chunk recompute (bounded-streaming summary,
 * Methodology 1: nested per-chunk checkpoint; RelayMoE 3.3: intermediates
 * rebuilt and released per step).  Chunks run from K-1 down to 0.
 * Inputs as for moe_route / moe_forward, plus dY [N, H] bf16.
 * Outputs (all overwritten, never accumulated into):
 *   dX     [N, H] bf16         gradient of sum(Y * dY) w.r.t. X, expert and
 *                              router paths, summed in fp32 in a fixed order
 *   dWr    [E, H] fp32         router weight gradient
 *   dWg, dWu [E, I, H] fp32    expert weight gradients
 *   dWd    [E, H, I] fp32
 *   dgates [N, k] fp32 or NULL gradient w.r.t. the gates
 * The selected set is held fixed (top-k is piecewise constant); the bias
 * gets no gradient.  dX and dgates are identical bit for bit for every K;
 * dW* and dWr are bitwise reproducible for a fixed K.
 * The router weight gradient of each chunk runs on a library-owned side
 * stream that forks from and joins `stream` through events.  That stream and
 * its two events are created on the first call from each (host thread,
 * device) and kept until the process exits: a thread that calls this function
 * holds one non-blocking stream and two events per device it used. */
int moe_backward(const moe_config* cfg, const uint16_t* X, const float* Wr, const int32_t* topk_idx,
                 const float* gates, const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                 const uint16_t* dY, uint16_t* dX, float* dWr, float* dWg, float* dWu, float* dWd,
                 float* dgates, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, returns the first device-side error recorded in the
 * workspace's status word since the last check (MOE_OK if none), and
 * clears it. */
int moe_check_status(void* ws, void* stream);

/* Device-side wait limit in nanoseconds used by every bounded wait in the
 * library's kernels (default 2e9).  Values <= 0 restore the default. */
int moe_set_wait_limit_ns(int64_t ns);

/* Form of the row-tile expert GEMMs (gate/up, down, dX, dActU):
 *   MOE_GEMM_AUTO   (default) CTA pairs when the average expert segment of a chunk or hop has at
 *                   least 512 rows, single CTAs otherwise;
 *   MOE_GEMM_SINGLE one CTA per 128-row tile (tcgen05.mma.cta_group::1, M = 128);
 *   MOE_GEMM_PAIR   a CTA pair per 256-row tile (tcgen05.mma.cta_group::2, M = 256).
 * The results are the same bit for bit; only the speed differs.  Applies to later calls from
 * every host thread. */
enum { MOE_GEMM_AUTO = 0, MOE_GEMM_SINGLE = 1, MOE_GEMM_PAIR = 2 };
int moe_set_gemm_form(int form);

/* Launch chaining of the library's kernels (see the conventions above):
 *   MOE_CHAIN_NONE  plain stream order: every kernel starts after the previous one has finished;
 *   MOE_CHAIN_EARLY programmatic dependent launch: a kernel may be scheduled early but waits for its
 *                   predecessor before its first global memory access;
 *   MOE_CHAIN_LATE  (default) as EARLY, and the kernels that share no buffer with their predecessor run
 *                   beside it and wait for it at their end.
 * The results are the same bit for bit in every mode; only the overlap differs.  Applies to later
 * calls from every host thread; returns MOE_ERR_INVALID_ARG for any other value. */
enum { MOE_CHAIN_NONE = 0, MOE_CHAIN_EARLY = 1, MOE_CHAIN_LATE = 2 };
int moe_set_launch_chaining(int mode);

/* How each chunk's (or hop's) routed rows of X and dY reach the expert GEMMs ("Training
 * Trillion-Parameter MoE" blog, section 3.3: the permute fused into its neighbours; bounded-streaming
 * summary, Methodology 1: the routed buffers are what the memory bound counts):
 *   MOE_DISPATCH_GATHER  (default) a gather kernel writes them into permuted buffers Xp, dYp [k c_eff, H]
 *                        that the GEMMs read with tiled loads.  Routed working set: two k c_eff H bf16
 *                        buffers ({Xp, Op} forward, {Xp, dYp then dXp} backward) = the pages' bound.
 *   MOE_DISPATCH_ON_LOAD the GEMMs read them straight from X and dY with TMA row gathers
 *                        (tile::gather4, four rows per copy); no Xp or dYp exists.  Routed working set:
 *                        one buffer (Op forward, dXp backward), half the bound.  Slower: a row tile's rows
 *                        are gathered again for every column tile.
 * The results are the same bit for bit; the workspace sizes (moe_workspace_bytes and
 * moe_hops_workspace_bytes) follow the mode, so query them after choosing it.  Applies to later calls
 * from every host thread; returns MOE_ERR_INVALID_ARG for any other value. */
enum { MOE_DISPATCH_GATHER = 0, MOE_DISPATCH_ON_LOAD = 1 };
int moe_set_dispatch(int mode);

/* Statistics of this host thread's last successful route/forward/backward/plan call. */
int moe_last_stats(moe_stats* out);

/* Human-readable text for a return code; for MOE_ERR_CUDA it includes the
 * CUDA error of the failing call on this host thread. */
const char* moe_strerror(int code);

/* ---- expert-partition ("hop") schedule ----------------------------------
 * RelayMoE summary, sections 3.1 and 3.3: instead of token chunks, the work
 * walks over P partitions of the experts ("hops"): hop h takes experts
 * [floor(h*E/P), floor((h+1)*E/P)) and all of their routes, rebuilds and
 * releases its intermediates before the next hop.  Each expert's weights are
 * read once per pass and its weight gradients are written once, with no
 * per-chunk read-modify-write; the price is that the routed working set is
 * set by the largest hop, which depends on the router (section 3.3), so the
 * caller sizes the workspace for `max_hop_rows` routed rows per hop
 * (moe_hop_rows_worst_case gives N * min(k, experts per hop), always enough).
 * A hop with more rows than max_hop_rows is skipped and reported as
 * MOE_ERR_DEVICE_CHECK through moe_check_status.
 * Arguments, layouts and outputs are those of moe_forward / moe_backward; c
 * and K_max are not used.  Per-token sums run in fp32 in hop order, then slot
 * order, so Y and dX agree with the chunk schedule to rounding (not bit for
 * bit); dW* and dgates are each formed in one hop. */

/* Routed rows per hop that always suffice for P hops: N * min(k, ceil(E / P)). */
int moe_hop_rows_worst_case(const moe_config* cfg, int32_t P, int32_t* rows);

/* Workspace bytes of moe_forward_hops / moe_backward_hops (either may be NULL). */
int moe_hops_workspace_bytes(const moe_config* cfg, int32_t P, int32_t max_hop_rows, size_t* fwd_bytes,
                             size_t* bwd_bytes);

int moe_forward_hops(const moe_config* cfg, int32_t P, int32_t max_hop_rows, const uint16_t* X,
                     const int32_t* topk_idx, const float* gates, const uint16_t* Wg, const uint16_t* Wu,
                     const uint16_t* Wd, uint16_t* Y, void* ws, size_t ws_bytes, void* stream);

int moe_backward_hops(const moe_config* cfg, int32_t P, int32_t max_hop_rows, const uint16_t* X, const float* Wr,
                      const int32_t* topk_idx, const float* gates, const uint16_t* Wg, const uint16_t* Wu,
                      const uint16_t* Wd, const uint16_t* dY, uint16_t* dX, float* dWr, float* dWg, float* dWu,
                      float* dWd, float* dgates, void* ws, size_t ws_bytes, void* stream);

/* ---- instrumentation (host side; no effect on results) ----------------- */

/* Kernel classes timed by the profiler. */
enum {
  MOE_K_ROUTER_LOGITS = 0, MOE_K_ROUTER_TOPK, MOE_K_PLAN, MOE_K_GATHER, MOE_K_GEMM_GATEUP,
  MOE_K_GEMM_DOWN, MOE_K_COMBINE, MOE_K_GEMM_DACT, MOE_K_GEMM_DW, MOE_K_GEMM_DX,
  MOE_K_UNPERMUTE, MOE_K_ROUTER_DW, MOE_K_ZERO, MOE_K_HOP_PLAN, MOE_K_FINAL, MOE_K_ADAMW,
  MOE_K_CE_LOGITS, MOE_K_CE_MERGE, MOE_K_CE_DLOGIT, MOE_K_CE_DX, MOE_K_CE_DW, MOE_K_ROUTE_GRAD, MOE_K_COUNT
};

/* When on, every kernel launch is bracketed by CUDA events on its stream. */
int moe_profile_enable(int on);

/* Synchronises on the recorded events and writes, per kernel class, the
 * number of launches and their summed device time (ms) since the last reset;
 * arrays of MOE_K_COUNT entries.  `names` (may be NULL) receives static
 * strings. */
int moe_profile_read(int32_t* launches, double* total_ms, const char** names);

/* Drops recorded events and counters. */
int moe_profile_reset(void);

/* Diagnostic: where the expert GEMMs wait.  Only in a library built with
 * -DMOE_GEMM_WAIT_STATS (python -m top_softmax_router_gb300.build --wait-stats);
 * otherwise returns MOE_ERR_NOT_BUILT and does nothing.  The first call
 * allocates MOE_GEMM_WAIT_CLASSES * MOE_GEMM_WAIT_FIELDS uint64 counters on the
 * current device (the one allocation this library makes; one device per
 * process) and from then on every row-tile and weight-gradient GEMM launch adds
 * to them, in SM cycles (clock64):
 *   class = form * 16 + epilogue * 2 + two_phase  (form 0: one CTA, 1: CTA
 *   pair; epilogue 0 gate/up + SwiGLU, 1 gate/up recompute, 2 store (down,
 *   dX: two_phase = 1), 3 dActU, 4 weight gradients);
 *   fields: 0 CTAs (pairs: clusters), 1 the MMA warps' lifetime, 2 cycles the
 *   MMA warp waited for a stage's operands, 3 for a free accumulator, 4 cycles
 *   the producer waited for a free stage, 5 K blocks of 64 multiplied.
 * The call synchronises the device, copies the counters to `counters` (may be
 * NULL) and zeroes them if `reset`.  The clock reads and atomics slow the
 * kernels down: the counters attribute waits, they do not time the kernels. */
#define MOE_GEMM_WAIT_CLASSES 32
#define MOE_GEMM_WAIT_FIELDS 8
int moe_diag_gemm_wait_stats(uint64_t* counters, int reset);

/* Diagnostic: enqueues one kernel whose thread waits, through the library's
 * bounded wait, on a barrier that nothing ever signals; after `limit_ns` it
 * records MOE_ERR_TIMEOUT in the workspace status word and returns (no trap,
 * the context stays usable).  Used to test the timeout path. */
int moe_diag_wait_timeout(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream);

/* ---- router without a workspace ---------------------------------------- */

/* Capacity, in fp32 logits (N * E), of the library's fixed router array: 16 MiB. */
#define MOE_ROUTE_NOALLOC_MAX_LOGITS (4 * 1024 * 1024)

/* Router for callers that cannot allocate device memory (the source pages
 * have no counterpart to this call).  Example callers: a serving process
 * whose own pool reserved all device memory at start-up, so a later
 * cudaMalloc fails or fragments the pool; a plugin inside a framework that
 * owns the device allocator and offers no way to borrow a workspace.
 * Arguments and results are those of moe_route (same kernels, bit-identical
 * topk_idx and gates) minus the workspace: the fp32 logits go to a fixed
 * device array of MOE_ROUTE_NOALLOC_MAX_LOGITS floats inside the library,
 * which every GPU that loads the library holds until the process exits.
 * The call allocates nothing.
 *   - N * E above MOE_ROUTE_NOALLOC_MAX_LOGITS returns
 *     MOE_ERR_UNSUPPORTED_SHAPE before any GPU work (use moe_route then).
 *   - The first call on a device looks up the array's device address with
 *     that device current (cudaGetSymbolAddress); make that first call
 *     before any stream capture on the device.
 *   - All calls share the array.  Calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race on it; calls on one stream
 *     are ordered.  Each call writes every logit before reading it, so the
 *     array's previous contents never matter.
 *   - Device-side index checks are not reported (there is no status word).
 *   - The device address is kept for the life of the process.  After
 *     cudaDeviceReset (which destroys the context and the array with it)
 *     the kept address is stale: do not call this function on a device that
 *     has been reset since its first call. */
int moe_route_noalloc(const moe_config* cfg, const uint16_t* X, const float* Wr, const float* bias,
                      int32_t* topk_idx, float* gates, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TOP_SOFTMAX_ROUTER_MOE_H_ */
