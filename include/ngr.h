/*
 * ngr.h -- C ABI of the fused pre-norm linear layer library for NVIDIA GB300
 * (sm_103a).
 *
 * The library computes a LayerNorm or RMSNorm row reduction whose normalized
 * rows feed a dense matrix product directly, with a bias and/or SiLU
 * epilogue.  The normalized activations exist only in on-chip memory and
 * are never written to device memory: for M > 32 each tile of x is
 * normalized in shared memory on its way to the tensor core; for
 * decode-sized batches (M <= 32) each CTA of the weight-streaming kernel
 * normalizes its slice of the tokens in shared memory once and streams its
 * weight tiles against it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers to dense row-major arrays owned
 *    by the caller.  The library allocates no device memory and frees none;
 *    temporaries live in the caller's `workspace` (see ngr_workspace_bytes).
 *  - x is [M, K]; W is [N, K] (the nn.Linear layout: y = a . W^T); gamma and
 *    beta are [K]; bias is [N]; y is [M, N].  Every tensor has the element
 *    type `dtype` (NGR_F16 or NGR_BF16).  Statistics, the normalization and
 *    the accumulation are FP32; y is rounded to nearest-even once.
 *  - Alignment: the kernels read rows of a 16-byte pitch, so when K and N
 *    (F for the chains) are multiples of 8 every pointer must be 16-byte
 *    aligned.  Every entry point also takes any K and N (F): when one is not
 *    a multiple of 8 it copies its operands into the workspace with rows
 *    padded by zeros to a multiple of 8 (weights also get zero rows up to a
 *    multiple of 8), runs the aligned kernels with statistics over the real
 *    columns only, and copies the real columns of its outputs back
 *    ([MMF] §五 optimization 1: a 513 x 14337 activation).  Pointers then
 *    need only 2-byte alignment (for the single-layer entry points y needs
 *    16 bytes when N % 8 == 0), ngr_workspace_bytes includes the copies and
 *    the weights are copied on every such call.  The folded layer is the
 *    exception: its weight is prepared once in the padded layout (see
 *    ngr_fold_prepare).  The workspace is 256-byte aligned.  M is arbitrary
 *    (M == 0 is a no-op that returns NGR_OK).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous: the call returns once the kernels are
 *    launched.  Argument errors are detected before anything is launched and
 *    returned as a negative ngr_status; launch failures return
 *    NGR_ERR_CUDA.  Errors raised inside a kernel (a bounded wait that ran
 *    out) are recorded in the workspace's error word: read them with
 *    ngr_workspace_error.  With the environment variable NGR_DEBUG=1 every
 *    call synchronizes its stream and returns that word's status itself.
 *    With NGR_TRACE=1 every call prints the kernel variant it chose (tile
 *    width, stages, grid) to stderr.
 *  - The kernels need an sm_103 device (GB300); any other device gives
 *    NGR_ERR_ARCH.  There is no fallback path.
 *  - Calls are thread-safe.  Two calls that share one workspace must be
 *    ordered (the same stream, or synchronized).
 *
 * Sources, cited by page title and section:
 *  [LNF] "LayerNorm 融合算子如何让大模型推理再快 15%？深度拆解 ATB 的实现"
 *  [MMF] "昇腾CANN的MatMul融合玩法，让大模型推理快3倍"
 *  [ATB] "CANN推理加速库ascend-transformer-boost ATB算子融合实战：昇腾NPU上
 *        LayerNorm+MatMul融合与Llama2大模型推理优化深度指南"
 */
#ifndef NGR_H
#define NGR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no
 * CUDA header. */
typedef struct CUstream_st *ngr_stream_t;

typedef enum { NGR_F16 = 0, NGR_BF16 = 1 } ngr_dtype;

typedef enum {
    NGR_OK = 0,
    NGR_ERR_NULL = -1,      /* a required pointer is NULL */
    NGR_ERR_SHAPE = -2,     /* M < 0, K <= 0, N <= 0, or too large */
    NGR_ERR_ALIGN = -3,     /* K or N not a multiple of 8 (where required), or a pointer misaligned */
    NGR_ERR_DTYPE = -4,     /* dtype is not NGR_F16 / NGR_BF16 */
    NGR_ERR_WORKSPACE = -5, /* workspace NULL or smaller than ngr_workspace_bytes */
    NGR_ERR_ARCH = -6,      /* no sm_103 device current */
    NGR_ERR_CUDA = -7,      /* a CUDA runtime/driver call failed */
    NGR_ERR_TIMEOUT = -8,   /* a kernel's bounded wait ran out (see ngr_workspace_error) */
    NGR_ERR_ARG = -9        /* any other invalid argument */
} ngr_status;

/* Operation codes for ngr_workspace_bytes. */
typedef enum {
    NGR_OP_LAYERNORM_LINEAR = 0,
    NGR_OP_RMSNORM_LINEAR = 1,
    NGR_OP_LINEAR_SILU = 2,
    NGR_OP_FFN = 3,
    NGR_OP_NORM_LINEAR = 4,   /* ngr_fused_norm_linear_act */
    NGR_OP_MLP = 5,           /* ngr_fused_mlp */
    NGR_OP_SWIGLU = 6,        /* ngr_fused_norm_swiglu */
    NGR_OP_MLP_SWIGLU = 7,    /* ngr_fused_mlp_swiglu */
    NGR_OP_LINEAR_RESIDUAL_NORM = 8  /* ngr_fused_linear_residual_norm */
} ngr_op;

/* Row normalization applied to x before the first product. */
typedef enum {
    NGR_NORM_NONE = 0,
    NGR_NORM_LAYER = 1,       /* (x - mu) rstd gamma + beta */
    NGR_NORM_RMS = 2          /* x rstd gamma */
} ngr_norm;

/* Activation applied after the bias. */
typedef enum {
    NGR_ACT_NONE = 0,
    NGR_ACT_SILU = 1,         /* z / (1 + exp(-z)) */
    NGR_ACT_RELU = 2,         /* max(z, 0) */
    NGR_ACT_GELU = 3          /* z (1 + erf(z / sqrt 2)) / 2, the exact form */
} ngr_act;

/* Bytes of device workspace that `op` needs for these sizes.  For the
 * two-GEMM ops (FFN, MLP, MLP_SWIGLU) and SWIGLU pass the hidden width F as
 * N; their intermediate H is included only if `ffn_h_in_workspace` is
 * nonzero.  Pure host arithmetic: needs no GPU and never fails (returns 0
 * for invalid sizes). */
size_t ngr_workspace_bytes(int op, int64_t M, int64_t K, int64_t N,
                           int ffn_h_in_workspace);

/* y = LayerNorm(x) . W^T (+ bias).
 * Per row i: mu = mean_k x[i,k]; var = mean_k (x[i,k] - mu)^2 (biased);
 * a[i,k] = (x[i,k] - mu) / sqrt(var + eps) * gamma[k] + beta[k];
 * y[i,n] = sum_k a[i,k] W[n,k] + bias[n].
 * [LNF] §1.1 (statistics, normalize, affine), §2.1 (LayerNormLinearFusion:
 * layer_norm then matmul with the weight transposed, the normalized rows kept
 * on chip), §2.3 (FP32 statistics); [ATB] LayerNormMatMul fusion
 * (fused_layernorm_matmul(x, w, bias)).
 * bias may be NULL.  gamma, beta, W, x, y, workspace may not. */
int ngr_fused_layernorm_linear(const void *x, const void *gamma,
                               const void *beta, const void *W,
                               const void *bias, float eps, int64_t M,
                               int64_t K, int64_t N, int dtype, void *y,
                               void *workspace, size_t workspace_bytes,
                               ngr_stream_t stream);

/* y = RMSNorm(x) . W^T (+ bias).
 * a[i,k] = x[i,k] / sqrt(mean_k x[i,k]^2 + eps) * gamma[k]; no beta.
 * [MMF] §二 strategy 3 (fused_rms_norm_matmul(x, w.T)); [ATB] Llama2 section
 * (RMSNorm feeding the projections).  bias may be NULL. */
int ngr_fused_rmsnorm_linear(const void *x, const void *gamma, const void *W,
                             const void *bias, float eps, int64_t M, int64_t K,
                             int64_t N, int dtype, void *y, void *workspace,
                             size_t workspace_bytes, ngr_stream_t stream);

/* y = SiLU(x . W^T + bias), SiLU(z) = z / (1 + exp(-z)); bias (may be NULL)
 * is added before the activation.
 * [MMF] §二 strategy 1 (fused_matmul_silu(x, w.T)). */
int ngr_fused_linear_silu(const void *x, const void *W, const void *bias,
                          int64_t M, int64_t K, int64_t N, int dtype, void *y,
                          void *workspace, size_t workspace_bytes,
                          ngr_stream_t stream);

/* FFN chain: H = SiLU(x . W1^T) [M, F], y = H . W2^T [M, K].
 * W1 is [F, K], W2 is [K, F].  H is written to device memory exactly once
 * and read once: into `h` ([M, F], dtype) when non-NULL, else into the
 * workspace (size it with ffn_h_in_workspace = 1).
 * [MMF] §二 strategy 2 (fused_matmul_silu_matmul(x, w1.T, w2.T)). */
int ngr_ffn_linear_silu_linear(const void *x, const void *W1, const void *W2,
                               int64_t M, int64_t K, int64_t F, int dtype,
                               void *h, void *y, void *workspace,
                               size_t workspace_bytes, ngr_stream_t stream);

/* The general fused layer: y = act(norm(x) . W^T + bias), norm one of
 * ngr_norm, act one of ngr_act (others give NGR_ERR_ARG).  gamma is needed
 * unless norm is NGR_NORM_NONE, beta only with NGR_NORM_LAYER (ignored
 * otherwise); bias may be NULL.  Workspace: NGR_OP_NORM_LINEAR.
 * [LNF] §1.1, §2.1; [MMF] §二 strategies 1 and 3 and the table of fused GEMM
 * instructions (MatMul + ReLU / GELU / SiLU). */
int ngr_fused_norm_linear_act(int norm, int act, const void *x,
                              const void *gamma, const void *beta,
                              const void *W, const void *bias, float eps,
                              int64_t M, int64_t K, int64_t N, int dtype,
                              void *y, void *workspace, size_t workspace_bytes,
                              ngr_stream_t stream);

/* The two-layer fusion chain:
 *   H = act(norm(x) . W1^T + b1) [M, F],  y = H . W2^T + b2 [M, K].
 * W1 is [F, K], W2 is [K, F]; b1 [F] and b2 [K] may be NULL.  H is written
 * once and read once, into `h` ([M, F]) when non-NULL, else into the
 * workspace (NGR_OP_MLP with ffn_h_in_workspace = 1).  norm / act / gamma /
 * beta as in ngr_fused_norm_linear_act.
 * [LNF] §3.3 (LayerNorm -> MatMul -> BiasAdd -> ReLU -> MatMul -> BiasAdd
 * fused as one chain). */
int ngr_fused_mlp(int norm, int act, const void *x, const void *gamma,
                  const void *beta, const void *W1, const void *b1,
                  const void *W2, const void *b2, float eps, int64_t M,
                  int64_t K, int64_t F, int dtype, void *h, void *y,
                  void *workspace, size_t workspace_bytes, ngr_stream_t stream);

/* SwiGLU with its norm: a = norm(x);
 *   h[i, j] = SiLU(a[i, :] . Wg[j, :]) * (a[i, :] . Wu[j, :])  [M, F].
 * Wg (gate) and Wu (up) are [F, K].  The two products share every
 * normalized x tile on chip and h is written once.  Workspace:
 * NGR_OP_SWIGLU.  [ATB] Llama2 inference, model structure and fusion
 * opportunities (the FFN's SwiGLU, a SiLU-gated linear transform, fused
 * with its matmuls; one RMSNorm feeding several projections). */
int ngr_fused_norm_swiglu(int norm, const void *x, const void *gamma,
                          const void *beta, const void *Wg, const void *Wu,
                          float eps, int64_t M, int64_t K, int64_t F, int dtype,
                          void *h, void *workspace, size_t workspace_bytes,
                          ngr_stream_t stream);

/* The Llama MLP: h as ngr_fused_norm_swiglu, then y = h . Wd^T [M, K] with
 * Wd [K, F].  h goes to `h` ([M, F]) when non-NULL, else to the workspace
 * (NGR_OP_MLP_SWIGLU with ffn_h_in_workspace = 1).  [ATB] as above (the
 * RMSNorm -> MatMul -> SiLU -> MatMul path of the decoder layer). */
int ngr_fused_mlp_swiglu(int norm, const void *x, const void *gamma,
                         const void *beta, const void *Wg, const void *Wu,
                         const void *Wd, float eps, int64_t M, int64_t K,
                         int64_t F, int dtype, void *h, void *y, void *workspace,
                         size_t workspace_bytes, ngr_stream_t stream);

/* A norm after the product (the output projection fused with the RMSNorm
 * that follows it):
 *   h = x . W^T + bias + residual  [M, N]   (bias, residual may be NULL),
 *   y = norm(h) over each row's N columns: LayerNorm (h - mu) rstd gamma +
 *       beta or RMSNorm h rstd gamma, with gamma, beta of length N.
 * norm: 1 = LayerNorm, 2 = RMSNorm.  h goes to `h` when non-NULL (the
 * residual stream a transformer keeps), else to the workspace
 * (NGR_OP_LINEAR_RESIDUAL_NORM with ffn_h_in_workspace = 1).  The product's
 * epilogue adds bias and residual and writes h once; one statistics pass
 * per h row then writes y.  [MMF] §五 optimization 3 (MatMul(Output) fused
 * with the following RMSNorm). */
int ngr_fused_linear_residual_norm(int norm, const void *x, const void *W,
                                   const void *bias, const void *residual,
                                   const void *gamma, const void *beta,
                                   float eps, int64_t M, int64_t K, int64_t N,
                                   int dtype, void *h, void *y, void *workspace,
                                   size_t workspace_bytes, ngr_stream_t stream);

/* Inference-mode weight fold, step 1 of 2 ([LNF] §6.2: with gamma and beta
 * fixed, gamma is folded into the matmul weight once, ahead of the calls).
 * norm: 1 = LayerNorm, 2 = RMSNorm (beta ignored, may be NULL).  With K8,
 * N8 = K, N rounded up to multiples of 8 (K8 = K, N8 = N when aligned), it
 * writes
 *   Wf[n,k]    = gamma[k] W[n,k] rounded to `dtype`   ([N, K8] rows, dtype;
 *                columns K..K8 zero),
 *   cb[n]      = c[n]  = sum_k Wf[n,k] (from the rounded Wf)   (FP32),
 *   cb[N8 + n] = b'[n] = sum_k beta[k] W[n,k] + bias[n]      (FP32),
 * so cb is FP32 [2, N8] (zero past N).  bias may be NULL.  Wf and cb must be
 * 16-byte aligned, the other pointers 2-byte aligned (16-byte aligned and
 * K, N multiples of 8 select the vectorized kernel).  Reads W once, writes
 * Wf once. */
int ngr_fold_prepare(int norm, const void *gamma, const void *beta,
                     const void *W, const void *bias, int64_t K, int64_t N,
                     int dtype, void *Wf, float *cb, ngr_stream_t stream);

/* Inference-mode weight fold, step 2 of 2: the same layer as
 * ngr_fused_layernorm_linear (norm = 1) or ngr_fused_rmsnorm_linear
 * (norm = 2), from the folded weight:
 *   y[i,n] = rstd_i (x[i,:] . Wf[n,:]) - rstd_i mu_i c[n] + b'[n]
 * (RMSNorm: mu = 0), mu and rstd the FP32 row statistics of x.  The matrix
 * product runs on raw x; no normalized operand exists at all.  Wf and cb
 * are in ngr_fold_prepare's layout ([N, K8], [2, N8]).  Workspace as for the
 * unfolded op (ngr_workspace_bytes of NGR_OP_LAYERNORM_LINEAR or
 * NGR_OP_RMSNORM_LINEAR).  [LNF] §6.2. */
int ngr_fused_norm_linear_folded(int norm, const void *x, const void *Wf,
                                 const float *cb, float eps, int64_t M,
                                 int64_t K, int64_t N, int dtype, void *y,
                                 void *workspace, size_t workspace_bytes,
                                 ngr_stream_t stream);

/* Variant of ngr_fused_layernorm_linear for callers that cannot allocate
 * device memory and so cannot supply a workspace -- for example code running
 * where every device allocation is planned or owned by someone else, or an
 * embedding that can only pass input and output tensors.  It computes the
 * same y = LayerNorm(x) . W^T (+ bias; bias may be NULL) as
 * ngr_fused_layernorm_linear, with the same arguments minus the workspace.
 * The paper has no counterpart; this is a deployment variant.
 *
 * Unlike ngr_fused_layernorm_linear it makes no zero-padded copies (they
 * would need scratch of the operands' size): K and N must be multiples of 8
 * and x, gamma, beta, W, bias and y 16-byte aligned, else NGR_ERR_ALIGN.  It
 * always runs the tile kernel without a K split, and never the decode
 * kernel, so for small M or few output tiles it can be slower than the
 * workspace entry point.
 *
 * Its scratch (per-row statistics, FP32 gamma/beta, the error word) is one
 * fixed array of about 256 KiB in the library's device memory, present on
 * every GPU that loads the library until the process exits.  The call
 * allocates nothing.  Limits: M <= NGR_NOALLOC_MAX_M and
 * K <= NGR_NOALLOC_MAX_K, else NGR_ERR_SHAPE.  The first call in each CUDA
 * context looks up the array's device address (cudaGetSymbolAddress), so
 * make that first call before any stream capture.  All calls share the one
 * array, which keeps the last call's contents; each call rewrites what it
 * reads, but calls that overlap on the GPU race on it and must not be
 * issued.  Errors: argument checks and launch failures as for the other
 * entry points; a kernel whose bounded wait ran out leaves its mark in the
 * array's error word, which ngr_noalloc_error reads (with NGR_DEBUG=1 every
 * call does that before returning). */
#define NGR_NOALLOC_MAX_M 16384
#define NGR_NOALLOC_MAX_K 16384
int ngr_fused_layernorm_linear_noalloc(const void *x, const void *gamma,
                                       const void *beta, const void *W,
                                       const void *bias, float eps, int64_t M,
                                       int64_t K, int64_t N, int dtype, void *y,
                                       ngr_stream_t stream);

/* The error word of ngr_fused_layernorm_linear_noalloc, for callers without
 * a workspace: synchronize `stream`, then return and clear the word kept in
 * the library's fixed array (NGR_OK, or NGR_ERR_TIMEOUT when a kernel of
 * the last call gave up on a bounded wait).  NGR_ERR_CUDA if the
 * synchronization or the read fails.  Allocates nothing.  The paper has no
 * counterpart. */
int ngr_noalloc_error(ngr_stream_t stream);

/* Step a1 alone: per-row FP32 statistics into stats[2*M] as (mu, rstd)
 * pairs.  norm: 1 = LayerNorm, 2 = RMSNorm (mu = 0).  [LNF] §1.1, §2.3.
 * Exposed so the statistics stage can be checked by itself. */
int ngr_row_stats(int norm, const void *x, float eps, int64_t M, int64_t K,
                  int dtype, float *stats, ngr_stream_t stream);

/* Synchronize `stream`, then return and clear the error word kept in
 * `workspace` (NGR_OK, or NGR_ERR_TIMEOUT when a kernel's bounded wait ran
 * out).  NGR_ERR_CUDA if the synchronization itself fails. */
int ngr_workspace_error(void *workspace, ngr_stream_t stream);

/* Launch one tiny kernel whose mbarrier wait can never complete, bounded by
 * `timeout_us`; it must give up, record NGR_ERR_TIMEOUT in the workspace's
 * error word and exit.  Exercises the bounded-wait path without faulting or
 * hanging the device.  Needs ngr_workspace_bytes(any op, 0, 8, 8, 0) bytes. */
int ngr_debug_bounded_wait(void *workspace, uint32_t timeout_us,
                           ngr_stream_t stream);

/* Tuning aid: restrict the choice of the tile kernel (M > 32) for every
 * later call in this process, on every thread.  `pair`: -1 let the planner
 * decide, 0 the single-CTA kernel (128-row tiles), 1 the CTA-pair kernel
 * (256-row tiles; only taken when M > 128), 2 the multicast cluster kernel
 * (clusters of two CTA pairs sharing each weight box, 512 x 464 tiles; only
 * taken when M > 256; bn and nsub are ignored).  `bn`: 0 any, else the N tile
 * (or sub-tile) width, one of 128, 192, 224, 256.  `nsub`: 0 any, else the
 * N sub-tiles per CTA-pair tile, 1 or 2 (2 only with bn 192, 224 or 256).  The
 * planner picks the cheapest variant that satisfies all three; if none does
 * it ignores the restriction.  ngr_set_tile_config(-1, 0, 0) restores the
 * default.  The environment variables NGR_PAIR, NGR_BN and NGR_NSUB give
 * the initial setting.  Returns NGR_OK or NGR_ERR_ARG. */
int ngr_set_tile_config(int pair, int bn, int nsub);

/* Inspection aid: the tile-kernel variant a call of `op` with these sizes
 * would launch on the current device, with a workspace of
 * ngr_workspace_bytes(op, M, K, N, 0) bytes, for its main product (the
 * chains' second product; NGR_OP_NORM_LINEAR is planned as if it had a
 * norm).  Writes plan[0..5] = pair (0 single CTA, 1 CTA
 * pair, 2 multicast cluster of two pairs), N (sub-)tile
 * width, sub-tiles per tile, K splits, CTAs, pipeline stages.  Returns
 * NGR_OK, NGR_ERR_ARG (bad op, or a shape that takes the decode or gated
 * kernel), NGR_ERR_NULL, or NGR_ERR_ARCH / NGR_ERR_CUDA. */
int ngr_tile_plan(int op, int64_t M, int64_t K, int64_t N, int *plan);

/* Profiling aid: time every kernel of this thread's next `n_calls` calls.
 * Each such call records CUDA events (the library's own, created here; no
 * device memory) on its stream just before and just after each kernel it
 * launches, at most NGR_MAX_KERNELS_PER_CALL per call.  Recording between a
 * call's kernels keeps them from overlapping, so time whole calls with this
 * off.  Returns NGR_OK, NGR_ERR_ARG for n_calls <= 0, NGR_ERR_CUDA if
 * events cannot be created. */
#define NGR_MAX_KERNELS_PER_CALL 4
int ngr_kernel_timing_start(int n_calls);

/* End the timing started by ngr_kernel_timing_start: wait for its events and
 * write the time in milliseconds of kernel k of timed call c to
 * ms[c * NGR_MAX_KERNELS_PER_CALL + k] (-1 where the call launched fewer
 * kernels), for as many calls as `capacity` floats hold.  Returns the number
 * of calls timed (>= 0) or a negative ngr_status. */
int ngr_kernel_timing_stop(float *ms, int capacity);

/* Human-readable name of a status code (static storage). */
const char *ngr_status_string(int status);

/* Text describing the last CUDA failure seen by this thread (the call that
 * failed and the CUDA error); empty if none.  Static thread-local storage. */
const char *ngr_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int ngr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NGR_H */
