/*
 * mhc.h -- C ABI of the GB300 (sm_103a) mHC seam library, libmhc.so.
 *
 * The manifold-constrained hyper-connection (mHC) seam of DeepSeek-V4.1-style
 * decoders, as described on the vLLM pull-request pages
 *   [A] "[ROCm][DSV4.1][Perf] Use AITER mHC for the delayed pre block" (#56503)
 *   [B] "[ROCm][DSv4.1] Fix TileLang mHC pre on 64-wide wavefronts and use the
 *        fused kernels on the AMD path" (#56342)
 * Every pointer argument is a caller-owned DEVICE pointer (CUDA global
 * memory) unless stated otherwise; the library never allocates device
 * memory, frees or synchronises inside a call, and only mhc_seam_host copies
 * between host and device (its purpose; on two library streams created once
 * per device).  Calls are
 * asynchronous on the given stream (a cudaStream_t passed as void*; NULL is
 * the legacy default stream).  Every call works on the CURRENT CUDA device:
 * the stream and every device pointer must belong to it.  Arguments are
 * checked on the host before any launch: a rejected call launches nothing
 * and returns the status.
 *
 * Types: bf16 tensors are passed as uint16_t bit patterns; fp32 as float.
 * All tensors are dense, row-major, and every array pointer must be 16-byte
 * aligned.
 */
#ifndef MHC_H
#define MHC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mhc_status {
    MHC_OK = 0,
    MHC_ERR_INVALID_ARGUMENT = 1, /* NULL, misaligned or aliasing pointer, bad count   */
    MHC_ERR_UNSUPPORTED = 2,      /* valid but outside the shapes this library handles */
    MHC_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed               */
    MHC_ERR_TIMEOUT = 4           /* a bounded device-side wait gave up (see below)      */
} mhc_status;

/*
 * mhc_pre_delayed -- the delayed mHC pre block ([A], commit message and
 * section "Why V4.1 cannot just reuse MHCPreOp": it collapses the sublayer's
 * input with the PREVIOUS seam's pre-mix and returns this seam's pre-mix;
 * "Approach": the projection with each row's sum of squares, then the post
 * and comb gates with all the Sinkhorn iterations; "Result": the collapse is
 * a plain fp32 weighted sum, bit-exact between implementations;
 * [B] "Measurements": the optional RMSNorm fold x * rsqrt * norm_weight is
 * evaluated in fp32 and rounded once).  Per token t, with K = n*C and
 * x_flat[t][i*C + c] = x[t][i][c]:
 *   r      = 1 / sqrt(sum_k x_flat^2 / K + rms_eps)
 *   l[m]   = r * (x_flat . fn[m]) * alpha_seg(m) + bias[m],  m < 2n + n^2,
 *            alpha_seg = alpha[0] (m < n), alpha[1] (m < 2n), alpha[2] (rest)
 *   pre_out[i]  = sigmoid(l[i]);  post_out[i] = 2 sigmoid(l[n + i])
 *   comb_out    = sinkhorn_iters Sinkhorn iterations on comb logits
 *                 l[2n + i*n + j] (row i = source stream, column j =
 *                 destination): iteration 1 = row softmax, + sinkhorn_eps on
 *                 every entry, column normalisation; later iterations = row
 *                 then column normalisation
 *   h[c]   = ((pre_in[0] x[0][c] + pre_in[1] x[1][c]) + pre_in[2] x[2][c])
 *            + pre_in[3] x[3][c], every product and sum rounded to fp32
 *   layer_input[c] = bf16(h[c])                                 (norm_weight NULL)
 *                  = bf16(h[c] / sqrt(mean_c h^2 + norm_eps) * w[c])  (fold)
 *
 *  x            [T, n, C] bf16   residual streams (read only)
 *  pre_in       [T, n]    fp32   incoming pre-mix of the previous seam
 *  fn           [2n+n^2, n*C] fp32  projection weight
 *  bias         [2n+n^2]  fp32
 *  alpha        [3]       fp32   pre / post / comb logit scales
 *  norm_weight  [C] bf16 or NULL (NULL: no RMSNorm fold)
 *  T            tokens, >= 0 (T == 0 launches nothing and returns MHC_OK)
 *  n            streams; this library supports n == 4 only
 *  C            hidden size; multiple of 8, 8 <= C <= 6144
 *  sinkhorn_iters >= 1 (the pages use 20)
 *  rms_eps, norm_eps, sinkhorn_eps  >= 0 (the pages' workload: 1e-6 each)
 *  pre_out [T,n], post_out [T,n], comb_out [T,n,n] fp32; layer_input [T,C] bf16
 *  logits_out   [T, 2n+n^2] fp32 or NULL (debug / parity layer)
 *  workspace    device scratch of at least mhc_pre_workspace_bytes(T, n, C)
 *               bytes, 256-byte aligned, owned by the caller; NULL is allowed
 *               when that size is 0.  Its contents on entry do not matter
 *               (the call writes everything it later reads); it may be reused
 *               by consecutive calls on one stream, but two calls that can
 *               run concurrently need separate workspaces.
 *  stream       cudaStream_t
 * Outputs must not overlap any input or the workspace (pre_out must not
 * alias pre_in: ping-pong two buffers across seams).  Errors:
 * MHC_ERR_INVALID_ARGUMENT (also: workspace too small or misaligned),
 * MHC_ERR_UNSUPPORTED, MHC_ERR_CUDA.  One kernel launch per call below 256
 * tokens; from 256 tokens two: fn split into its bf16 planes (one copy, in
 * the workspace), then the tensor-core kernel.
 */
mhc_status mhc_pre_delayed(const uint16_t *x, const float *pre_in, const float *fn,
                           const float *bias, const float *alpha,
                           const uint16_t *norm_weight, int64_t T, int n, int C,
                           int sinkhorn_iters, float rms_eps, float norm_eps,
                           float sinkhorn_eps, float *pre_out, float *post_out,
                           float *comb_out, uint16_t *layer_input, float *logits_out,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Workspace bytes mhc_pre_delayed needs for a shape on the current device
 * (host only).  0 when the shape runs on the CUDA-core kernel (fewer than 256
 * tokens, or a hidden size the tensor-core kernel does not take); otherwise
 * the per-call copy of fn split into three bf16 planes (2,949,120 bytes at
 * C = 5120, shared by every cluster), plus T x 16 bytes (rounded to 256)
 * that mhc_pre uses; the same size serves mhc_pre_delayed, mhc_pre and
 * mhc_post_pre_delayed.
 * Returns 0 as well for shapes mhc_pre_delayed rejects.
 */
size_t mhc_pre_workspace_bytes(int64_t T, int n, int C);

/*
 * mhc_pre_delayed_noalloc -- mhc_pre_delayed for callers that cannot
 * allocate device memory, and so cannot pass a workspace: for example a
 * serving engine that reserves all free device memory for its caches up front
 * and forbids later allocations, a plugin that only receives tensors from its
 * host application, or a latency-critical path that cannot afford
 * cudaMalloc's implicit device synchronisation.  (The pages describe no such
 * entry point; it has no counterpart there.)
 *
 * Same arguments, meaning, layouts and results as mhc_pre_delayed, minus the
 * workspace.  It always runs the tensor-core kernel, with its scratch in a
 * fixed device array of MHC_NOALLOC_SCRATCH_BYTES that the library holds on
 * every GPU that loads it, until the process exits; it never calls
 * cudaMalloc, cudaFree or any allocating routine.  The array holds one copy
 * of fn's planes, packed by a first launch; the tensor-core kernel then runs
 * on the whole GPU as in mhc_pre_delayed (two launches per call).
 *  C            multiple of 256, 256 <= C <= 5120 (else MHC_ERR_UNSUPPORTED)
 * First call on a device: resolves the array's device address and sets the
 * kernel up for that device (no allocation); make that first call outside any
 * stream capture.  Nothing in the array needs to start at zero: each call
 * rewrites the part it reads before reading it.  Every call shares the one
 * array: calls whose kernels can overlap on the GPU (different streams, or
 * graphs replayed concurrently) race on it and must be serialised by the
 * caller.  The array's address belongs to the current device, so x must be
 * device memory of the current device and the stream (when not NULL) a
 * stream of it: otherwise MHC_ERR_INVALID_ARGUMENT, returned before anything
 * is set up or launched.  Other errors as mhc_pre_delayed.
 */
#define MHC_NOALLOC_SCRATCH_BYTES 2949120u
mhc_status mhc_pre_delayed_noalloc(const uint16_t *x, const float *pre_in, const float *fn,
                                   const float *bias, const float *alpha,
                                   const uint16_t *norm_weight, int64_t T, int n, int C,
                                   int sinkhorn_iters, float rms_eps, float norm_eps,
                                   float sinkhorn_eps, float *pre_out, float *post_out,
                                   float *comb_out, uint16_t *layer_input, float *logits_out,
                                   void *stream);

/*
 * mhc_post -- the mHC post block ([A] "Result": the mhc_post call sites go
 * through MHCPostOp; the post mixes the residual streams through comb and
 * adds the post-gated sublayer output):
 *   x_new[t][j][c] = bf16( sum_i comb[t][i][j] * x[t][i][c] + post[t][j] * y[t][c] )
 * accumulated in fp32, rounded once.
 *  x     [T, n, C] bf16;  y [T, C] bf16 (sublayer output)
 *  comb  [T, n, n] fp32;  post [T, n] fp32 (from mhc_pre_delayed)
 *  x_new [T, n, C] bf16; may be exactly x (in place); must not otherwise
 *        overlap an input.
 *  n == 4; C multiple of 8; T >= 0.  Errors as mhc_pre_delayed.
 *  One kernel launch per call.
 */
mhc_status mhc_post(const uint16_t *x, const uint16_t *y, const float *comb,
                    const float *post, int64_t T, int n, int C, uint16_t *x_new,
                    void *stream);

/*
 * mhc_pre -- the non-delayed mHC pre block (the V4 form, MHCPreOp, that [A]
 * "Why V4.1 cannot just reuse MHCPreOp" contrasts with the delayed one; its
 * norm_weight= keyword per [B] "The bug"): the same gates, comb and fold as
 * mhc_pre_delayed, but the collapse uses THIS token's own pre-mix,
 *   h[t][c] = ((pre[t][0] x[t][0][c] + pre[t][1] x[t][1][c]) + ...) + ...,
 * with pre[t] exactly the fp32 values written to pre_out.  Equivalently:
 * mhc_pre_delayed with pre_in := its own pre_out.  No pre_in argument; all
 * other arguments as mhc_pre_delayed.  Below 256 tokens (and for hidden sizes
 * the tensor-core kernel does not take) one kernel, where the finalising CTA
 * sends each token's pre to the cluster before the collapse; from 256 tokens
 * three launches: fn's planes, the tensor-core kernel for the gates only,
 * then a streaming collapse and fold with the pre it wrote, in the
 * tensor-core kernel's order of summation (mhc_pre_workspace_bytes covers
 * both: the planes plus T * 16 bytes of scratch).
 */
mhc_status mhc_pre(const uint16_t *x, const float *fn, const float *bias, const float *alpha,
                   const uint16_t *norm_weight, int64_t T, int n, int C, int sinkhorn_iters,
                   float rms_eps, float norm_eps, float sinkhorn_eps, float *pre_out,
                   float *post_out, float *comb_out, uint16_t *layer_input, float *logits_out,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * mhc_post_pre_delayed -- one seam boundary in a single call: the PREVIOUS
 * seam's post (as mhc_post, on x, y, comb, post) followed by THIS seam's
 * delayed pre (as mhc_pre_delayed) on its result x_new.  A decoder runs
 * ... pre(s) -> sublayer -> post(s) -> pre(s+1) ..., and post(s) and
 * pre(s+1) meet at x_new ([A] "Result": the seam's launch count is the
 * figure the pages track; the next seam's pre reads exactly the x_new the
 * post writes).
 *  x, y, comb, post, x_new  as mhc_post (comb/post: the previous seam's
 *                            outputs); x_new is written.
 *  all other arguments      as mhc_pre_delayed, with x_new in place of x.
 * Results are bit-identical to mhc_post followed by mhc_pre_delayed on the
 * same arguments.  Below 256 tokens (and for hidden sizes the tensor-core
 * kernel does not take) this is ONE kernel: each CTA forms x_new for its
 * column slice of the tile, writes it out and runs the pre block on it from
 * shared memory (x is read once).  From 256 tokens on it is three launches:
 * the post kernel, fn's planes, then the tensor-core pre kernel; the
 * workspace is then needed as for mhc_pre_delayed (mhc_pre_workspace_bytes).
 * Aliasing: x_new may be exactly x; comb_out may be exactly comb and
 * post_out exactly post (one gate buffer carried along a chain); pre_out
 * must not overlap pre_in; nothing else may overlap.
 * Errors as mhc_pre_delayed; additionally y, comb, post, x_new are
 * required, 16-byte aligned.
 */
mhc_status mhc_post_pre_delayed(const uint16_t *x, const uint16_t *y, const float *comb,
                                const float *post, uint16_t *x_new, const float *pre_in,
                                const float *fn, const float *bias, const float *alpha,
                                const uint16_t *norm_weight, int64_t T, int n, int C,
                                int sinkhorn_iters, float rms_eps, float norm_eps,
                                float sinkhorn_eps, float *pre_out, float *post_out,
                                float *comb_out, uint16_t *layer_input, float *logits_out,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Model-entry broadcast seam ([A] "Approach": at the model's entry the
 * projection's operand is x, narrower than the streams, and AITER declines
 * that case; [A] "Test Plan": the delayed
 * block is tested with the carried pre-mix and with the model-entry one).
 * At the model's entry the n residual streams are n copies of one hidden
 * state x[t][c] (the embedding output), so these calls take x as [T, C] and
 * read it as every stream:  x_b[t][i][c] = x[t][c], i < n.
 *
 * mhc_pre_delayed_broadcast -- mhc_pre_delayed on x_b, with pre_in the
 *   model-entry pre-mix the caller supplies.  In closed form the projection
 *   operand narrows to C columns (x_flat . fn[m] = x . sum_i fn[m][i*C ..],
 *   r = 1/sqrt(sum_c x^2 / C + rms_eps)) and h = the fp32 sum of
 *   pre_in[i] * x in stream order; the kernels compute it as the n-stream
 *   block on x_b, so every output is bit-identical to mhc_pre_delayed on an
 *   explicit copy x_b.  x is read once per token (C * 2 bytes instead of
 *   n * C * 2).
 * mhc_pre_broadcast -- mhc_pre (non-delayed) on x_b, the same way.
 *  x  [T, C] bf16; all other arguments, the workspace, the plan and the
 *     errors as mhc_pre_delayed / mhc_pre (x's byte range is T * C * 2).
 */
mhc_status mhc_pre_delayed_broadcast(const uint16_t *x, const float *pre_in, const float *fn,
                                     const float *bias, const float *alpha,
                                     const uint16_t *norm_weight, int64_t T, int n, int C,
                                     int sinkhorn_iters, float rms_eps, float norm_eps,
                                     float sinkhorn_eps, float *pre_out, float *post_out,
                                     float *comb_out, uint16_t *layer_input, float *logits_out,
                                     void *workspace, size_t workspace_bytes, void *stream);
mhc_status mhc_pre_broadcast(const uint16_t *x, const float *fn, const float *bias,
                             const float *alpha, const uint16_t *norm_weight, int64_t T, int n,
                             int C, int sinkhorn_iters, float rms_eps, float norm_eps,
                             float sinkhorn_eps, float *pre_out, float *post_out,
                             float *comb_out, uint16_t *layer_input, float *logits_out,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * mhc_post_broadcast -- mhc_post on x_b: the entry seam's post, which turns
 * the single hidden state into the n residual streams,
 *   x_new[t][j][c] = bf16( sum_i comb[t][i][j] * x[t][c] + post[t][j] * y[t][c] ),
 * with mhc_post's arithmetic (bit-identical to mhc_post on x_b).
 *  x [T, C] bf16 (read once per column); y, comb, post, x_new, errors as
 *  mhc_post; x_new [T, n, C] must not overlap x or any other input.
 */
mhc_status mhc_post_broadcast(const uint16_t *x, const uint16_t *y, const float *comb,
                              const float *post, int64_t T, int n, int C, uint16_t *x_new,
                              void *stream);

/*
 * mhc_seam_host -- one seam, the delayed pre block then the post block on
 * the same residual (mhc_pre_delayed, then mhc_post with that call's comb
 * and post), for activations in page-locked HOST memory: the end-to-end call
 * for a caller whose tokens live on the host.
 *  x_h [T, n, C] bf16, y_h [T, C] bf16, pre_in_h [T, n] fp32: HOST inputs.
 *  fn, bias, alpha, norm_weight: DEVICE weights, as mhc_pre_delayed.
 *  x_new_h [T, n, C] bf16, pre_out_h [T, n] fp32: HOST outputs (required);
 *  post_out_h [T, n], comb_out_h [T, n, n] fp32 and layer_input_h [T, C]
 *  bf16: HOST outputs, each optional (NULL: not copied back).
 *  Every host pointer must be page-locked (cudaHostAlloc / cudaHostRegister):
 *  MHC_ERR_INVALID_ARGUMENT otherwise.  x_new_h may be exactly x_h; no other
 *  host ranges may overlap.
 *  workspace: DEVICE, 256-byte aligned, at least
 *  mhc_seam_host_workspace_bytes(T, n, C) bytes (two chunks of device copies
 *  of the activations plus the pre block's workspace); owned by the caller,
 *  and calls that share one must be ordered on the same stream.
 * The tokens go in chunks (1024 tokens from 2048 on; one chunk below 512;
 * no chunk under 256 tokens, so every chunk takes the kernel the whole call
 * would): chunk k's kernels run on `stream` while chunk k+1 is copied in and
 * chunk k-1 copied out on two library-owned streams (created once per
 * device).  The outputs are bit-identical to mhc_pre_delayed + mhc_post on
 * device copies.  Asynchronous: the host outputs are complete when `stream`
 * reaches the point after this call; capturable in a CUDA graph (the
 * library streams fork from and join back to `stream`).  Host enqueue is
 * serialised by a process-wide lock.  Errors as mhc_pre_delayed.
 */
size_t mhc_seam_host_workspace_bytes(int64_t T, int n, int C);
mhc_status mhc_seam_host(const uint16_t *x_h, const uint16_t *y_h, const float *pre_in_h,
                         const float *fn, const float *bias, const float *alpha,
                         const uint16_t *norm_weight, int64_t T, int n, int C,
                         int sinkhorn_iters, float rms_eps, float norm_eps, float sinkhorn_eps,
                         uint16_t *x_new_h, float *pre_out_h, float *post_out_h,
                         float *comb_out_h, uint16_t *layer_input_h, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Pre-packed weights for the tensor-core path (from 256 tokens).  fn is a
 * weight: the tensor-core kernel otherwise converts it, at the start of every
 * call, into three exact bf16 planes (fn = hi + mid + lo) in its MMA operand
 * layout, one copy per 16-CTA cluster in the workspace.  Packed once, the
 * planes are read by every cluster from one shared copy and the per-call
 * conversion disappears.
 *
 * mhc_pre_packed_bytes -- size of the packed planes for (n, C): 16 regions
 *   of ceil(C/512) x 18 KB (2.95 MB at C = 5120); 0 when the tensor-core kernel does
 *   not take C (C a multiple of 256 up to 5120, n == 4).  Host only.
 * mhc_pre_pack -- write the planes of fn [2n+n^2, n*C] fp32 (device) to
 *   packed (device, 256-byte aligned, at least mhc_pre_packed_bytes; must not
 *   overlap fn).  One kernel on `stream`.  The planes stay valid while fn
 *   is unchanged: re-pack after writing fn.  MHC_ERR_UNSUPPORTED for a C the
 *   tensor-core kernel does not take.
 * mhc_pre_delayed_packed -- mhc_pre_delayed with the planes packed ahead:
 *   bit-identical outputs.  fn (device) is still required, for calls under
 *   256 tokens (the cluster kernel reads fn directly); packed, packed_bytes
 *   as written by mhc_pre_pack for the same fn and C.  No workspace.
 *   Errors as mhc_pre_delayed; MHC_ERR_INVALID_ARGUMENT for a NULL,
 *   misaligned or short packed buffer, or a C without packed planes.
 */
size_t mhc_pre_packed_bytes(int n, int C);
mhc_status mhc_pre_pack(const float *fn, int n, int C, void *packed, size_t packed_bytes,
                        void *stream);
mhc_status mhc_pre_delayed_packed(const uint16_t *x, const float *pre_in, const float *fn,
                                  const void *packed, size_t packed_bytes, const float *bias,
                                  const float *alpha, const uint16_t *norm_weight, int64_t T,
                                  int n, int C, int sinkhorn_iters, float rms_eps,
                                  float norm_eps, float sinkhorn_eps, float *pre_out,
                                  float *post_out, float *comb_out, uint16_t *layer_input,
                                  float *logits_out, void *stream);

/* Static description of the status code (never NULL). */
const char *mhc_status_string(mhc_status status);

/*
 * Device status of the current device: synchronises the device, then reads
 * and clears the library's device-side status word.  MHC_ERR_TIMEOUT means a
 * bounded wait inside a kernel gave up since the last call (that launch's
 * outputs are garbage).  After such a timeout the kernel stops issuing loads,
 * still waits -- with bounded waits the timeout does not cut short -- for
 * its own TMA and bulk loads, its tensor-core MMAs and the last bytes its
 * cluster peers push into it, then frees its tensor memory and returns.
 * Should one of those drain waits also give up, the kernel returns anyway
 * (a copy still in flight is then not waited for).  No test provokes a
 * timeout.  MHC_ERR_CUDA if the synchronisation or the read failed.
 */
mhc_status mhc_device_status(void);

/*
 * Launch plan of mhc_pre_delayed for a shape, without launching (host only,
 * no device needed for the shape checks).  kernel: 1 = cluster kernel
 * (warp-level MMA, one tile of up to 32 tokens per 16-CTA cluster, the tokens
 * spread evenly over the co-resident clusters), 2 = tensor-core kernel
 * (128-token tiles, used from 256 tokens on when C is a multiple of 256 and at
 * most 5120); grid/cluster: CTAs launched and CTAs per cluster (grid 0 when no
 * device is current); tokens_per_tile (for kernel 1 without a current device:
 * min(T, 32)).
 * Returns the status mhc_pre_delayed would return for the shape checks.
 * Any output pointer may be NULL.
 */
mhc_status mhc_pre_delayed_plan(int64_t T, int n, int C, int *kernel, int *grid,
                                int *cluster, int *tokens_per_tile);

/*
 * Launch overlap between consecutive seam kernels (programmatic dependent
 * launch, a CUDA launch attribute; the pages' own kernels have no
 * counterpart: this is a scheduling option of this library, it changes no
 * result).  enable != 0: from then on mhc_post and mhc_pre_delayed's
 * cluster kernel (the one used below 256 tokens and for hidden sizes the
 * tensor-core kernel does not take) are launched so that they may start
 * while the previous kernel in the stream is still running.  The pre kernel
 * then loads fn, bias, alpha and norm_weight, and sets itself up, before it
 * waits for that kernel; it reads x and pre_in, and mhc_post reads all of
 * its inputs, only after the wait.
 * Contract while enabled: fn, bias, alpha and norm_weight must not be
 * written by the kernel (or copy) issued just before mhc_pre_delayed on the
 * same stream; they are weights, written once, in a decode step.  Outputs
 * are bit-identical with and without the overlap.  Works under stream
 * capture (the graph keeps the programmatic edges).  Process-wide, off at
 * load.  Returns the previous setting (0 or 1).
 */
int mhc_set_launch_overlap(int enable);

/* Library version, (major << 16) | minor. */
int mhc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MHC_H */
