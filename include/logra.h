/*
 * logra.h -- C ABI of the LoGRA gradient-sketch / RowAdam library (liblogra.so).
 *
 * Method: "LoGRA: Scaling LLM Reinforcement Learning with Low-Rank Gradient
 * Sketches".  A d x k projection weight W is trained without its d x k
 * gradient G = dY^T X.  During the backward pass every microbatch adds its
 * contribution to a d x r sketch S += dY^T (X A^T) (theclarity.today write-up,
 * "Why it matters": S = G * A^T, G d x k, A r x k, r << d, k), where A is a
 * random-sign matrix redrawn each step and held fixed over that step's
 * microbatches (academy.dair.ai summary, "Gradient sketches").  At update time
 * Ghat = S A is rebuilt tile by tile and consumed by RowAdam, which keeps one
 * running mean-square statistic per row and no first moment (theclarity.today
 * write-up, "What happened").
 *
 * Conventions shared by every call
 *   - Matrices are dense, row-major, with no padding between rows:
 *       X  n x k    activations of one microbatch (one row per token)
 *       dY n x d    output gradients of that microbatch
 *       W  d x k    fp32 master weight (nn.Linear layout: out x in)
 *       S  d x r    fp32 sketch
 *       v  d        fp32 RowAdam second moment, one value per row of W
 *   - Every pointer is a DEVICE pointer (cudaMalloc / torch CUDA memory) on the
 *     current device, owned by the caller, except where a comment says "host".
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and do
 *     not synchronise it.  The library keeps no per-matrix state.
 *   - A = Sigma * fl32(1/sqrt(r)); Sigma[i][j] = +1 or -1, from bit (j mod 64)
 *     of a 64-bit word hashed from (seed, step, i, j div 64) with SplitMix64
 *     (set bit -> -1).  A is regenerated inside the kernels and never stored,
 *     except by logra_sign_matrix.
 *   - Shape rules: n >= 0; d, k >= 1 and multiples of 8 (16-byte rows for
 *     bf16 TMA tiles); r a multiple of 32 in [32, 512].  Other shapes return
 *     LOGRA_ERR_UNSUPPORTED and launch nothing.  n == 0 is a no-op.
 *   - Pointers must be 16-byte aligned (LOGRA_ERR_UNSUPPORTED otherwise).
 *   - Return value: a logra_status.  A non-OK status means nothing was
 *     launched, except LOGRA_ERR_CUDA, which reports a CUDA runtime error
 *     from the launch itself.  Device-side failures (a bounded wait that gave
 *     up) are recorded in a per-device status word read by logra_get_status.
 *   - The library allocates device memory only for an internal scratch
 *     workspace per (device, stream), grown on demand (on first use of a
 *     larger shape) and kept for the life of the process;
 *     logra_reserve_workspace pre-sizes it so that no allocation happens
 *     later (e.g. inside a stream capture).  The first apply on a stream
 *     also allocates, once, that stream's zero-kept scratch: 16 KB of
 *     counters and 8 MB of Gram-pass counts (make one apply on a stream
 *     before capturing its applies).
 */
#ifndef LOGRA_H
#define LOGRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* logra_stream_t; /* identical to cudaStream_t */

enum logra_status {
  LOGRA_OK = 0,
  LOGRA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad dtype     */
  LOGRA_ERR_UNSUPPORTED = 2,   /* shape or alignment outside the rules above */
  LOGRA_ERR_CUDA = 3,          /* CUDA runtime error (see logra_last_cuda_error) */
  LOGRA_ERR_TIMEOUT = 4,       /* a device-side wait gave up (logra_get_status) */
  LOGRA_ERR_NO_DEVICE = 5      /* no usable sm_103 device                    */
};

enum logra_dtype {
  LOGRA_F32 = 0,   /* IEEE binary32                 */
  LOGRA_BF16 = 1   /* bfloat16 (raw 16-bit storage) */
};

/* Text for a status code; never NULL. */
const char* logra_status_string(int status);

/* cudaError_t of the most recent LOGRA_ERR_CUDA on this thread (0 if none). */
int logra_last_cuda_error(void);

/* ABI version: (major << 16) | minor. */
int logra_version(void);

/*
 * Number of kernels this process has launched through the library so far
 * (all devices, all streams).  Host-side counter; lets a caller count the
 * device work behind a sequence of calls.
 */
uint64_t logra_launch_count(void);

/*
 * logra_sign_matrix -- write A = Sigma * fl32(1/sqrt(r)) as an r x k fp32
 * matrix (A_out, device, r*k floats, row-major).  The random-sign projection
 * of the academy.dair.ai summary ("Gradient sketches"); used by tests and by
 * callers that want the explicit matrix.  Bit-exact with any other
 * implementation of the same hash.  Any k >= 1 is accepted here.
 */
int logra_sign_matrix(uint64_t seed, uint64_t step, int r, int64_t k,
                      float* A_out, logra_stream_t stream);

/*
 * logra_sketch_accumulate -- S += dY^T (X A^T) for one microbatch.
 * (theclarity.today write-up, "Why it matters": S = G A^T accumulated during
 * backpropagation; aitop.news post: the full gradient is never built.)
 *   X        n x k, dtype in_dtype (LOGRA_BF16 or LOGRA_F32)
 *   dY       n x d, same dtype
 *   S        d x r fp32, read and written in place (the caller zeroes it at
 *            the first microbatch of a step)
 *   seed     per-matrix seed; step  the optimiser step (A is redrawn per step)
 * Padding tokens are zero rows of X and dY; n is at most 2^28
 * (LOGRA_ERR_UNSUPPORTED above).  bf16 inputs are multiplied exactly and
 * accumulated in fp32; the X A^T intermediate is kept as a two-term bf16
 * expansion (relative error about 2^-16).  fp32 inputs run on the same
 * tensor-core kernels: each element is split into two bf16 terms
 * x = x1 + x2 (|x - x1 - x2| <= 2^-16 |x|, the two-term bf16 splitting of
 * Henry, Tang & Heinecke, ARITH 2019), the planes are stacked along the
 * tokens as X' = [X1; X2; X1; X2], dY' = [dY1; dY1; dY2; dY2], and the bf16
 * sketch of those 4n tokens adds all four cross terms; fp32 inputs must be
 * finite and below bf16's largest finite value (about 3.39e38).
 * Uses the internal workspace: for bf16 inputs about 8 * r * n bytes (an fp32
 * P^T buffer and the two-term bf16 image the accumulate reads;
 * logra_sketch_workspace_bytes gives the exact figure); for fp32 inputs the
 * same for 4n tokens plus 8 * n * (k + d) bytes of stacked planes.
 * S is updated with atomic fp32 additions, so calls that add into the same S
 * (different microbatches of one step) may run concurrently on different
 * streams; the sum is then formed in an unspecified order.
 * Run-to-run determinism: partial sums of the projection and of S are added
 * by TMA reduce-adds whose order depends on CTA timing, so S may differ in
 * its last bits between two identical calls, even on one stream (the spread
 * is rounding-sized, far inside the 1e-3 parity tolerance).  A, and the
 * apply's W, v, bf16 copy and sync sketch for given S bits, are
 * deterministic.
 * CUDA graphs: a captured call keeps using the capturing stream's workspace
 * when replayed, so replays must be ordered with other work on that stream.
 * Once any call on a stream has been captured, that stream's sketch calls
 * clear their projection scratch with a memset on every call (eager calls
 * otherwise skip it when the previous sketch on the stream left it zero).
 */
int logra_sketch_accumulate(const void* X, const void* dY, int in_dtype,
                            int64_t n, int64_t d, int64_t k, int r,
                            uint64_t seed, uint64_t step, float* S,
                            logra_stream_t stream);

/*
 * logra_sketch_item -- one sketch of logra_sketch_accumulate_group: the
 * arguments of logra_sketch_accumulate that differ between sketches (device
 * pointers as there; bf16 X and dY).
 */
typedef struct logra_sketch_item {
  const void* X;            /* n x k bf16 activations of one microbatch        */
  const void* dY;           /* n x d bf16 output gradients of that microbatch  */
  float* S;                 /* d x r fp32 sketch, accumulated in place         */
  int64_t d, k;
  uint64_t seed;            /* this matrix's seed                               */
} logra_sketch_item;

/*
 * logra_sketch_accumulate_group -- logra_sketch_accumulate (bf16) for `count`
 * sketches of one token count n, one rank r and one step, issued from a
 * single caller stream: S += dY^T (X A^T) for every item.  (theclarity.today
 * write-up, "Why it matters": the sketches of a backward pass are
 * independent per weight matrix.)
 *   items   HOST array of `count` items, read during the call only.  Items may
 *           share an S (microbatches of one matrix): S is updated with atomic
 *           additions, so their sum is formed in an unspecified order.
 * The library forks the sketches round robin onto up to 16 side streams of its
 * own (created on the device's first group call and kept), shapes their
 * launches as for logra_set_concurrency(number of side streams used), and
 * joins the side streams back into `stream` before returning: work issued on
 * `stream` afterwards runs after every sketch of the group.  One matrix's
 * small calls then overlap another's, which a single stream cannot do.
 * Each side stream has its own workspace (allocated on first use; make one
 * group call of the largest shapes before capturing groups into a CUDA graph,
 * which records the fork and join like any other).  Every item is checked
 * before anything is launched; a failing launch still joins what was issued.
 * count == 0 or n == 0 is a no-op; n above 2^28 is LOGRA_ERR_UNSUPPORTED.
 */
int logra_sketch_accumulate_group(const logra_sketch_item* items, int count,
                                  int64_t n, int r, uint64_t step,
                                  logra_stream_t stream);

/*
 * logra_linear_backward -- the backward pass of a Linear layer Y = X W^T as
 * LoGRA runs it, for one microbatch (bf16 operands):
 *   dX = dY W           the input gradient, handed to the layer below;
 *   S += dY^T (X A^T)   the sketch, in place of the d x k weight gradient
 *                       dY^T X, which is never formed (theclarity.today
 *                       write-up, "Why it matters"; academy.dair.ai summary,
 *                       "Gradient sketches": no full gradient buffer).
 *   X   n x k bf16 activations of the microbatch
 *   dY  n x d bf16 output gradients of the microbatch
 *   W   d x k bf16 weight, the model's working copy (e.g. the W_bf16_out of
 *       logra_rowadam_apply_ex); may be NULL when dX is NULL
 *   dX  n x k bf16, overwritten: every element is the fp32 tensor-core sum
 *       over d, rounded once to bf16 (nearest even).  NULL: the sketch only.
 *       Must not overlap X, dY, W or S.
 *   S   d x r fp32 sketch, accumulated in place by the same kernels (and
 *       with the same result) as logra_sketch_accumulate.  NULL: dX only
 *       (X, r, seed and step are then not used).
 * dX and S must not both be NULL (LOGRA_ERR_INVALID_ARG); n must be below
 * 2^31, and at most 2^28 when S is given (LOGRA_ERR_UNSUPPORTED).  Launches, in this order on `stream`: one
 * persistent tensor-core kernel for dX (tcgen05 on CTA pairs, 256 x 256
 * output tiles taken from a per-stream tile counter), then the sketch's
 * launches.  dX comes first because the layer below waits for it, the sketch
 * only for the end of the step.  The sketch uses the stream's workspace as
 * logra_sketch_accumulate does; the dX kernel uses two words of the stream's
 * zero-kept counters (16 KB, allocated by the first such call or apply on
 * the stream: make one before capturing calls into a CUDA graph), which it
 * leaves at zero.
 */
int logra_linear_backward(const void* X, const void* dY, const void* W,
                          void* dX, int64_t n, int64_t d, int64_t k, int r,
                          uint64_t seed, uint64_t step, float* S,
                          logra_stream_t stream);

/*
 * logra_rowadam_apply -- RowAdam update rebuilt from the sketch:
 *   Ghat = S A;  v_i <- beta2 v_i + (1-beta2) * mean_j Ghat_ij^2;
 *   W_ij <- W_ij - lr * c * Ghat_ij / sqrt(v_i + eps).
 * (theclarity.today write-up, "What happened": per-row squared magnitudes, no
 * first moment; c is the step scale of the predicted-KL controller, which the
 * pages do not define, so the caller supplies it.)
 *   W          d x k fp32 master weight, updated in place
 *   S          d x r fp32 sketch (read only)
 *   v          d fp32, updated in place
 *   norms_out  device, 2 doubles, overwritten: {||S||_F^2, ||dW||_F^2} where
 *              dW is the fp32 update added to W -- the controller's inputs.
 *              May be NULL.
 * Uses the internal workspace: the Gram image of A (r x r, two bf16 terms),
 * the two-term bf16 image of S (d x r x 4 bytes) and d x 4 bytes of row
 * factors plus small partials (logra_apply_workspace_bytes gives the figure).
 */
int logra_rowadam_apply(float* W, const float* S, float* v, int64_t d,
                        int64_t k, int r, uint64_t seed, uint64_t step,
                        float beta2, float eps, float lr, float c,
                        double* norms_out, logra_stream_t stream);

/*
 * logra_rowadam_apply_ex -- logra_rowadam_apply plus two optional outputs
 * (either may be NULL):
 *   W_bf16_out      d x k bf16 copy of the updated master weight
 *                   (round to nearest even), the model's working weights.
 *   sync_sketch_out d x r fp32, S'_i = -lr * c * S_i / sqrt(v_i + eps) with the
 *                   updated v: logra_reconstruct(S', accumulate=1) on a rollout
 *                   worker adds the same update to its weights (academy.dair.ai
 *                   summary: the update is a product of two small matrices,
 *                   which makes policy synchronisation cheaper).
 */
int logra_rowadam_apply_ex(float* W, const float* S, float* v, int64_t d,
                           int64_t k, int r, uint64_t seed, uint64_t step,
                           float beta2, float eps, float lr, float c,
                           double* norms_out, uint16_t* W_bf16_out,
                           float* sync_sketch_out, logra_stream_t stream);

/*
 * logra_rowadam_apply_bc -- logra_rowadam_apply_ex with Adam's bias correction
 * of the second moment.  The pages name Adam's correction but leave RowAdam's
 * open (academy.dair.ai summary), so the plain calls above apply none; this
 * variant scales the step by the corrected v_hat_i = v_i / (1 - beta2^t)
 * (Kingma & Ba, "Adam", ICLR 2015, Algorithm 1):
 *   dW_ij = -lr * c * Ghat_ij / sqrt(v_hat_i + eps),
 * and the sync sketch and ||dW||^2 use the same v_hat.  The stored v stays the
 * uncorrected running average.
 *   t   the number of RowAdam updates of this matrix including this one
 *       (t >= 1; t = 0 is the uncorrected step).  t < 0, or t >= 1 with beta2
 *       outside [0, 1), returns LOGRA_ERR_INVALID_ARG.
 * Other arguments as for logra_rowadam_apply_ex.
 */
int logra_rowadam_apply_bc(float* W, const float* S, float* v, int64_t d,
                           int64_t k, int r, uint64_t seed, uint64_t step,
                           float beta2, float eps, float lr, float c, int64_t t,
                           double* norms_out, uint16_t* W_bf16_out,
                           float* sync_sketch_out, logra_stream_t stream);

/*
 * logra_apply_item -- one matrix of logra_rowadam_apply_group: the arguments of
 * logra_rowadam_apply_ex that differ between matrices.  Device pointers as
 * there; norms_out, W_bf16_out and sync_sketch_out may be NULL.
 */
typedef struct logra_apply_item {
  float* W;                 /* d x k fp32 master weight, updated in place */
  const float* S;           /* d x r fp32 sketch (read only)              */
  float* v;                 /* d fp32 second moment, updated in place     */
  int64_t d, k;
  uint64_t seed;            /* this matrix's seed (A is drawn per matrix) */
  float lr, c;
  double* norms_out;        /* 2 doubles: {||S||_F^2, ||dW||_F^2}         */
  uint16_t* W_bf16_out;     /* d x k bf16 copy of the updated W           */
  float* sync_sketch_out;   /* d x r, S'_i = -lr c S_i / sqrt(v_i + eps)  */
  int64_t t;                /* 0: RowAdam as defined; t >= 1: the bias-corrected step of
                               logra_rowadam_apply_bc for this matrix's t-th update */
} logra_apply_item;

/*
 * logra_rowadam_apply_group -- logra_rowadam_apply_ex for `count` matrices of
 * one rank r and one step: every output equals what `count` separate
 * logra_rowadam_apply_ex calls write (W, v, the bf16 copy and the sync sketch
 * bit for bit; the norms up to the order of their fp64 partial sums).
 *   items   HOST array of `count` items, read during the call only.  The
 *           matrices must not overlap in memory.
 * The matrices are processed in launch groups of up to 8: each group is one
 * preparation launch, one row-norm launch and one update launch whose work
 * units span all of the group's matrices, so small matrices (attention
 * projections of a layer) share the GPU with large ones instead of each
 * paying its own pipeline fill and tail (the update is the fused
 * reconstruct-and-update pass of the theclarity.today write-up, "What
 * happened").  Workspace: logra_apply_group_workspace_bytes(items, count, r)
 * bytes of the stream's scratch.  count == 0 is a no-op.
 */
int logra_rowadam_apply_group(const logra_apply_item* items, int count, int r,
                              uint64_t step, float beta2, float eps,
                              logra_stream_t stream);

/* Workspace bytes logra_rowadam_apply_group needs for these items (0 if an
 * item's shape is invalid). */
size_t logra_apply_group_workspace_bytes(const logra_apply_item* items,
                                         int count, int r);

/*
 * logra_rowadam_predict -- the norms logra_rowadam_apply would report with
 * c = 1, writing nothing else (W and v untouched).  Because dW is linear in c,
 * ||dW(c)||^2 = c^2 * norms_out[1]; a controller can pick c from this before
 * applying (academy.dair.ai summary, "Step control": the KL change is
 * predicted before the update is applied).
 *   norms_out  device, 2 doubles, overwritten.
 */
int logra_rowadam_predict(const float* S, const float* v, int64_t d, int64_t k,
                          int r, uint64_t seed, uint64_t step, float beta2,
                          float eps, float lr, double* norms_out,
                          logra_stream_t stream);

/* logra_rowadam_predict_bc -- logra_rowadam_predict for the bias-corrected
 * step of logra_rowadam_apply_bc (t as there). */
int logra_rowadam_predict_bc(const float* S, const float* v, int64_t d, int64_t k,
                             int r, uint64_t seed, uint64_t step, float beta2,
                             float eps, float lr, int64_t t, double* norms_out,
                             logra_stream_t stream);

/*
 * logra_reconstruct -- dW_out (+)= S A, the d x k matrix rebuilt from a d x r
 * sketch (policy synchronisation to rollout workers; academy.dair.ai summary).
 *   out_dtype  LOGRA_F32 or LOGRA_BF16 (bf16: round to nearest even)
 *   accumulate 0: overwrite dW_out; 1: dW_out += S A (bf16: computed in fp32,
 *              rounded once).
 */
int logra_reconstruct(const float* S, int64_t d, int64_t k, int r,
                      uint64_t seed, uint64_t step, void* dW_out,
                      int out_dtype, int accumulate, logra_stream_t stream);

/*
 * logra_get_status -- synchronise `stream`, then return and clear the device
 * status word of the current device: LOGRA_OK, or LOGRA_ERR_TIMEOUT if a
 * kernel's bounded wait gave up since the last call.
 */
int logra_get_status(logra_stream_t stream);

/*
 * logra_reserve_workspace -- grow the scratch workspace that calls on
 * (current device, `stream`) use to at least `bytes` now (synchronous
 * cudaMalloc), so later calls on that stream allocate nothing.  Each
 * (device, stream) pair has its own workspace, so calls on different streams
 * may overlap; calls on one stream are ordered by the stream.  Returns
 * LOGRA_ERR_CUDA if the allocation fails.
 */
int logra_reserve_workspace(size_t bytes, logra_stream_t stream);

/* Workspace bytes a sketch / apply call of this shape needs. */
size_t logra_sketch_workspace_bytes(int64_t n, int64_t d, int64_t k, int r, int in_dtype);
size_t logra_apply_workspace_bytes(int64_t d, int64_t k, int r);

/*
 * logra_sketch_accumulate_noalloc -- logra_sketch_accumulate for bf16 inputs
 * that never allocates device memory.  (The paper has no counterpart: this is
 * a deployment variant of the same operation, same arguments minus the dtype.)
 *
 * Meant for callers that are not allowed to call cudaMalloc: frameworks
 * whose caching allocator owns all device memory and forbids side
 * allocations, latency-critical loops that must not block in the driver,
 * and runtimes whose device memory is fixed at start-up.
 *
 * Scratch: instead of the per-stream workspace, the call uses one fixed
 * device array compiled into the library (logra_noalloc_scratch_bytes()
 * bytes, 32 MiB), which every GPU that loads the library holds until the
 * process exits.  A shape whose scratch need
 * (logra_sketch_workspace_bytes(n, d, k, r, LOGRA_BF16)) exceeds it returns
 * LOGRA_ERR_UNSUPPORTED and launches nothing.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) and caches it;
 * make that first call before any stream capture.  All calls, on every
 * stream of a device, share the one array and the array keeps the last
 * call's contents (each call clears, with cudaMemsetAsync, the part it
 * accumulates into and overwrites the rest before reading it): calls whose
 * execution overlaps on the GPU race and corrupt each other's results, so
 * order them (one stream, or events).  S, X and dY rules as for
 * logra_sketch_accumulate.
 */
int logra_sketch_accumulate_noalloc(const void* X, const void* dY, int64_t n, int64_t d, int64_t k, int r,
                                    uint64_t seed, uint64_t step, float* S, logra_stream_t stream);

/* Size in bytes of the fixed scratch array used by logra_sketch_accumulate_noalloc. */
size_t logra_noalloc_scratch_bytes(void);

/*
 * logra_set_concurrency -- tell the library on how many streams the caller
 * issues sketch calls at the same time (default 1; process-wide, any thread).
 * It only shapes launches, never results: with streams > 1 each call's
 * accumulate kernel runs on fewer, longer-running CTAs (at least 12 * streams
 * 32-token chunks each) and its projection on one CTA per 256-token group
 * over the whole k range (no partial sums), which leaves SMs to the other
 * streams' kernels and removes the partial-sum traffic; a call still keeps at
 * least its fair share of the SMs (SM count / streams) unless its one-stream
 * grid is smaller (a projection with fewer groups than that splits their k
 * ranges evenly over the fair share).
 * With one stream every call spreads over all SMs.  Returns
 * LOGRA_ERR_INVALID_ARG outside [1, 64].
 */
int logra_set_concurrency(int streams);

/*
 * logra_debug_inject -- TEST ONLY.  fault = 1 makes the next pipelined kernel
 * launch drop one producer arrival, so that its consumer's bounded wait runs
 * out and the kernel records LOGRA_ERR_TIMEOUT and exits cleanly (no trap, no
 * hang); fault = 0 clears it.  The wait limit is `timeout_cycles` clock ticks
 * (0 keeps the current limit).
 */
int logra_debug_inject(int fault, uint64_t timeout_cycles);

#ifdef __cplusplus
}
#endif

#endif /* LOGRA_H */
