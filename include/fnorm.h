/*
 * fnorm.h -- libfnorm: normalisation with per-slice statistics on NVIDIA
 * GB300 (sm_103a), as a C ABI.
 *
 * Sources (web pages; titles as on the pages, each page a sequence of
 * reasoning blocks counted from 1):
 *   Kimi-K2.6__l1_p34  InstanceNorm2d(64) on x[112,64,512,512].
 *   Kimi-K2.6__l2_p79  Conv3d -> x*m_c -> InstanceNorm3d -> clamp[-1,1]
 *                      -> x*m_c -> max over channels.
 *   Kimi-K2.6__l2_p73  Conv2d -> BatchNorm2d (training) -> x*2.0.
 * The convolutions that precede these steps on the pages are not part of
 * this library: callers pass the convolution's output.
 *
 * Conventions shared by every entry point
 *  - Tensors are contiguous, row-major, with the slice (spatial) axis
 *    innermost: x is [N][C][S] where S is the product of the spatial sizes.
 *  - Pointers named x, y, m, gamma, ... are DEVICE pointers owned by the
 *    caller. The library allocates no memory of its own.
 *  - Calls are asynchronous and ordered on `stream` (NULL = the legacy
 *    default stream). A returned FNORM_OK means the work was validated and
 *    enqueued; execution errors surface at the caller's next synchronisation.
 *  - Argument errors are returned before anything is launched and leave every
 *    output untouched. No C++ exception crosses this interface.
 *  - Element counts use 64-bit indices throughout (N*C*S may exceed 2^31).
 *  - N*C == 0 or S == 0 is a no-op that returns FNORM_OK.
 *  - Results are deterministic: the same inputs give bitwise-identical
 *    outputs (all reductions combine partial results in a fixed order).
 *  - Statistics: the mean and the biased variance (divide by the element
 *    count) over each slice, combined across threads, CTAs and clusters with
 *    the Chan/Welford pairwise update; normalisation is
 *    (x - mean) * rsqrt(var + eps) computed in fp32. Element counts inside
 *    the merges are fp32 values, exact up to 2^24 per merged part; above
 *    that (a slice or BatchNorm channel of more than 16,777,216 values that
 *    is not a multiple of the rounding step) a count carries a relative
 *    rounding error of at most 2^-24, which moves the merge weights and the
 *    variance by the same relative amount -- far below fp32 output accuracy.
 *  - Fast paths need x and y 16-byte aligned and the slice length a multiple
 *    of one 16-byte vector; other (element-aligned) inputs take a scalar-load
 *    path with the same results. Pointers not aligned to their element size
 *    are rejected with FNORM_ERR_ALIGNMENT.
 */
#ifndef FNORM_H
#define FNORM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FNORM_API __attribute__((visibility("default")))
#else
#define FNORM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* fnorm_stream_t;

typedef enum fnorm_status {
  FNORM_OK = 0,
  FNORM_ERR_INVALID_ARG = 1, /* bad size, null pointer, bad eps, overlapping buffers */
  FNORM_ERR_UNSUPPORTED = 2, /* valid request this build cannot serve (e.g. dtype combination) */
  FNORM_ERR_ALIGNMENT = 3,   /* pointer not aligned to its element size */
  FNORM_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  FNORM_ERR_TIMEOUT = 5      /* a device-side bounded wait expired (see fnorm_get_last_error) */
} fnorm_status;

typedef enum fnorm_dtype {
  FNORM_F32 = 0, /* IEEE binary32 */
  FNORM_BF16 = 1 /* bfloat16; computed in fp32, stored with round-to-nearest-even */
} fnorm_dtype;

/*
 * InstanceNorm forward, affine = False (Kimi-K2.6__l1_p34, blocks 1-2: the
 * per-(n,c) mean and biased variance over the H*W plane, then
 * (x - mean)/sqrt(var + eps) with eps = 1e-5 by default).
 *
 *   x         [N*C][S] input of type in_dtype.
 *   y         [N*C][S] output of type out_dtype. y may equal x (in place);
 *             any other overlap is rejected.
 *   eps       >= 0 (finite). With eps = 0 a constant slice yields NaN.
 *   mean_out  optional [N*C] fp32: the slice means (NULL to skip).
 *   rstd_out  optional [N*C] fp32: 1/sqrt(var + eps) (NULL to skip).
 * Every (in_dtype, out_dtype) pair of F32/BF16 is supported.
 * A slice is read from HBM once and written once whenever it fits in one
 * thread-block cluster (up to 2 MiB of input per slice); longer slices are
 * read twice (statistics pass, then normalisation pass). Out of place, with
 * fp32 input and output, 16-byte aligned x and y, S a multiple of 4, S above
 * 2^19 and N*C at most a quarter of the SM count, the few long slices are
 * spread over all SMs as fnorm_instancenorm_ws does, with y itself holding
 * the per-chunk statistics between the three launches (y's contents before
 * the call completes are unspecified, as for any output); the same holds for
 * fnorm_instancenorm_affine. In place, or otherwise, each long slice is
 * streamed by one cluster.
 * Statistics are accumulated in fp32 and merged in a fixed order: results are
 * deterministic for a given call shape and agree with the exact definition to
 * fp32 accuracy.
 */
FNORM_API fnorm_status fnorm_instancenorm(const void* x, void* y, int64_t N, int64_t C, int64_t S,
                                fnorm_dtype in_dtype, fnorm_dtype out_dtype, float eps,
                                float* mean_out, float* rstd_out, fnorm_stream_t stream);

/*
 * fnorm_instancenorm with a caller workspace, for a few slices too long for
 * one thread-block cluster (more than 2 MiB of fp32 each, e.g. x[1,1,8192,8192]):
 * the per-chunk statistics go to the workspace instead of y, which also serves
 * in-place calls (fnorm_instancenorm streams those through one cluster per
 * slice, leaving most SMs idle). Same arguments, results and errors as
 * fnorm_instancenorm, plus:
 *
 *   workspace        device memory of at least
 *                    fnorm_instancenorm_workspace_size(N, C, S) bytes,
 *                    256-byte aligned, owned by the caller; its contents need
 *                    no initialisation and are overwritten. Calls that
 *                    overlap in time must not share a workspace. It may be
 *                    NULL when that size is 0.
 *   workspace_bytes  its size.
 *
 * With fp32 input and output, 16-byte aligned x and y, S a multiple of 4, S
 * above 2^19 and N*C at most a quarter of the current device's SM count (the
 * workspace size is likewise that of the current device), the slices are
 * normalised as a BatchNorm over the [1, N*C, S] view: a statistics launch
 * over 64 KiB chunks of every slice (all SMs, per-chunk partials in the
 * workspace), for slices of 16 Mi values or more a launch that merges each
 * slice's partials, and an apply launch that merges them (or takes the merged
 * value) in a fixed order and normalises (x is read twice, the second time
 * partly from L2). Every other
 * call takes fnorm_instancenorm's own plan and leaves the workspace untouched.
 * The results agree with the exact definition to fp32 accuracy on either path.
 */
FNORM_API size_t fnorm_instancenorm_workspace_size(int64_t N, int64_t C, int64_t S);
FNORM_API fnorm_status fnorm_instancenorm_ws(const void* x, void* y, int64_t N, int64_t C,
                                             int64_t S, fnorm_dtype in_dtype,
                                             fnorm_dtype out_dtype, float eps, float* mean_out,
                                             float* rstd_out, void* workspace,
                                             size_t workspace_bytes, fnorm_stream_t stream);

/*
 * InstanceNorm forward with per-channel affine parameters (the module's
 * affine = True option; Kimi-K2.6__l1_p34, block 2 notes the default is
 * affine = False, and Kimi-K2.6__l2_p73, block 1 states the affine step
 * "normalise, times gamma, plus beta"):
 *   y = (x - mean) * (rstd * gamma[c]) + beta[c]   for slice q = n*C + c.
 *
 *   gamma, beta  optional [C] fp32 device arrays, 4-byte aligned (NULL means
 *                1 / 0; with both NULL this is fnorm_instancenorm). They may
 *                not overlap y, mean_out or rstd_out.
 * Every other argument, the paths and the traffic are those of
 * fnorm_instancenorm: the parameters add 8 bytes per channel of reads.
 */
FNORM_API fnorm_status fnorm_instancenorm_affine(const void* x, void* y, const float* gamma,
                                       const float* beta, int64_t N, int64_t C, int64_t S,
                                       fnorm_dtype in_dtype, fnorm_dtype out_dtype, float eps,
                                       float* mean_out, float* rstd_out, fnorm_stream_t stream);

/*
 * Fused post-convolution epilogue (Kimi-K2.6__l2_p79, block 1: the pipeline
 * scaled = conv_out*m, InstanceNorm over the spatial extent, clamp, a second
 * multiply by m, then the max over the channel dimension), fp32:
 *
 *   v      = x[n,c,s] * m[c]
 *   t      = (v - mean_nc(v)) / sqrt(var_nc(v) + eps)
 *   y[n,s] = max over c of  m[c] * clamp(t, clamp_lo, clamp_hi)
 *
 *   x       [N][C][S] fp32.       m [C] fp32.       y [N][S] fp32.
 *   argmax  optional [N][S] int64: the channel index of the maximum, the
 *           lowest index among equal maxima (NULL to skip).
 *   clamp   clamp_lo <= clamp_hi; clamp(t) = min(max(t, lo), hi).
 * y and argmax must not overlap x, m or each other.
 * With x/y/argmax 16-byte aligned and S a multiple of 4, a cluster of CTAs
 * handles each sample in one launch: x is read from HBM once for the
 * statistics, and the output pass re-reads it from L2 (the leading part of
 * each channel's range from shared memory), so HBM sees about one read of x
 * while the input fits in L2. Other shapes stream each slice twice.
 * Rounding: the statistics are fp32 and the results agree with the exact
 * definition to fp32 accuracy; without argmax the clamp is evaluated as an
 * equivalent saturating multiply-add, so y may differ from the argmax call's
 * y in the last bits. Results are deterministic for a given call shape.
 */
FNORM_API fnorm_status fnorm_instancenorm_epilogue(const float* x, const float* m, float* y, int64_t* argmax,
                                         int64_t N, int64_t C, int64_t S, float eps,
                                         float clamp_lo, float clamp_hi, fnorm_stream_t stream);

/*
 * Bytes of device workspace fnorm_batchnorm_train and
 * fnorm_batchnorm_local_stats need for this shape: the per-(run, chunk)
 * partial statistics (for runs of at most 16 values, per-column partials and
 * per-channel coefficients, whichever layout is larger) plus 256 bytes for a
 * grid-barrier counter (a multiple of 256; 0 when N*C*S == 0).
 */
FNORM_API size_t fnorm_batchnorm_workspace_size(int64_t N, int64_t C, int64_t S);

/*
 * Training-mode BatchNorm forward with a trailing scale factor
 * (Kimi-K2.6__l2_p73, blocks 1-2: BatchNorm2d in training mode followed by
 * x*scaling_factor; running statistics update with momentum, the running
 * variance taking the unbiased estimate as Kimi-K2.6__l2_p79 block 1 states):
 *
 *   per channel c over all (n, s): mean_c, var_c (biased), n_c = N*S
 *   y = scale * (gamma_c * (x - mean_c) * rsqrt(var_c + eps) + beta_c)
 *   running_mean_c <- (1 - momentum) * running_mean_c + momentum * mean_c
 *   running_var_c  <- (1 - momentum) * running_var_c
 *                     + momentum * var_c * n_c / (n_c - 1)
 *
 *   x, y          [N][C][S] fp32; y may equal x (in place).
 *   gamma, beta   optional [C] fp32 (NULL means 1 and 0).
 *   running_mean, running_var  optional [C] fp32, updated in place
 *                 (NULL: not updated). Both or neither.
 *   save_mean, save_rstd  optional [C] fp32: mean_c and rsqrt(var_c + eps).
 *   workspace     device memory of at least
 *                 fnorm_batchnorm_workspace_size(N, C, S) bytes, 256-byte
 *                 aligned, owned by the caller; its contents need no
 *                 initialisation and are overwritten. Calls that overlap in
 *                 time must not share a workspace.
 * Requires N*S >= 2 (the unbiased estimate needs two values).
 * x is read twice (statistics, then normalisation in reverse order so that
 * the tail of the first pass is still in L2) and y written once; two kernel
 * launches. Runs of at most 16 values (S <= 16, e.g. BatchNorm over [N, C])
 * take a column form instead: per-column statistics over blocks of rows, a
 * per-channel merge, then the normalisation (three launches).
 */
FNORM_API fnorm_status fnorm_batchnorm_train(const float* x, float* y, const float* gamma, const float* beta,
                                   float scale, float* running_mean, float* running_var,
                                   float momentum, float eps, float* save_mean, float* save_rstd,
                                   int64_t N, int64_t C, int64_t S, void* workspace,
                                   size_t workspace_bytes, fnorm_stream_t stream);

/*
 * Eval-mode BatchNorm forward with a trailing scale factor (Kimi-K2.6__l2_p73,
 * block 1: in eval mode the module normalises with its running statistics;
 * block 2: the per-channel factor gamma*scale/sqrt(running_var + eps) and
 * shift that the page folds into the convolution's weights and bias):
 *
 *   y = scale * (gamma_c * (x - running_mean_c) * rsqrt(running_var_c + eps)
 *                + beta_c)
 *
 *   x, y          [N][C][S] fp32; y may equal x (in place); any other overlap
 *                 is rejected.
 *   gamma, beta   optional [C] fp32 (NULL means 1 and 0).
 *   running_mean, running_var  required [C] fp32, read only (nothing is
 *                 updated in eval mode). A negative running_var + eps gives
 *                 NaN outputs for that channel, as the formula does.
 * One launch; x is read once and y written once (8 bytes per element).
 */
FNORM_API fnorm_status fnorm_batchnorm_eval(const float* x, float* y, const float* gamma,
                                            const float* beta, float scale,
                                            const float* running_mean, const float* running_var,
                                            float eps, int64_t N, int64_t C, int64_t S,
                                            fnorm_stream_t stream);

/*
 * Multi-process (synchronised) training BatchNorm: the batch is split along N
 * across R processes (one per GPU) and the per-channel statistics are
 * exchanged once -- the one exchange step of this method
 * (Kimi-K2.6__l2_p73, blocks 1-2, BatchNorm2d statistics over (N, H, W),
 * computed here over the union of the shards).
 *
 * Step 1, every rank: fnorm_batchnorm_local_stats writes stats_out [C][4]
 * fp32 (16-byte aligned device memory): per channel (count, mean, M2, 0) of
 * this rank's shard x [N][C][S], merged in a fixed order. workspace as for
 * fnorm_batchnorm_train. An empty shard (N*S == 0) writes zeros (the merge
 * identity).
 * Step 2, the caller gathers the R arrays in rank order into stats_all
 * [R][C][4] (e.g. an all-gather over NCCL).
 * Step 3, every rank: fnorm_batchnorm_apply_stats merges stats_all per
 * channel in rank order (every rank obtains bit-identical statistics), writes
 * y = scale * (gamma * (x - mean) * rsqrt(var + eps) + beta) for its shard,
 * the saved statistics, and updates running_mean/running_var with the merged
 * count (unbiased estimate; the merged count must be >= 2). Arguments as for
 * fnorm_batchnorm_train; no workspace. A rank whose shard is empty (N*S == 0)
 * still merges stats_all and updates its running and saved statistics.
 * Runs of at most 16 values (S <= 16) take column forms in both steps (every
 * rank of a group uses the same form, since S is the same on every rank).
 */
FNORM_API fnorm_status fnorm_batchnorm_local_stats(const float* x, float* stats_out, int64_t N,
                                                   int64_t C, int64_t S, void* workspace,
                                                   size_t workspace_bytes, fnorm_stream_t stream);
FNORM_API fnorm_status fnorm_batchnorm_apply_stats(const float* x, float* y, const float* stats_all,
                                                   int64_t R, const float* gamma, const float* beta,
                                                   float scale, float* running_mean,
                                                   float* running_var, float momentum, float eps,
                                                   float* save_mean, float* save_rstd, int64_t N,
                                                   int64_t C, int64_t S, fnorm_stream_t stream);

/*
 * fnorm_batchnorm_train without a workspace argument, for callers that cannot
 * allocate device memory: code held to a fixed memory budget reserved up
 * front, plugins whose host owns the allocator and forbids allocation after
 * start-up, and steady-state loops where a cudaMalloc (which may synchronise
 * the device) is not acceptable. The source pages have no counterpart to this
 * entry point; it exists only for such callers.
 *
 * Same arguments, results and errors as fnorm_batchnorm_train, minus
 * workspace/workspace_bytes. The partial statistics go to a scratch array
 * that the library itself holds in device memory: 2 MiB (2,097,152 bytes) on
 * every GPU that loads the library, kept until the process exits. Shapes with
 * fnorm_batchnorm_workspace_size(N, C, S) above 2 MiB are refused with
 * FNORM_ERR_UNSUPPORTED before any GPU work.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it; make that
 * first call before any stream capture begins. The call allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).
 *
 * All calls on a device share the one array, and it keeps whatever the last
 * call left there; nothing in it needs to start at zero because every call
 * writes each partial before reading it. Calls whose work overlaps on the
 * GPU (other streams, other host threads) race on the array: order them on
 * one stream or synchronise between them.
 */
FNORM_API fnorm_status fnorm_batchnorm_train_noalloc(const float* x, float* y, const float* gamma,
                                                     const float* beta, float scale,
                                                     float* running_mean, float* running_var,
                                                     float momentum, float eps, float* save_mean,
                                                     float* save_rstd, int64_t N, int64_t C,
                                                     int64_t S, fnorm_stream_t stream);

/* A static, human-readable name for a status code. */
FNORM_API const char* fnorm_status_string(fnorm_status status);

/*
 * Reads and clears the device error word of the current device: the first
 * device-side failure (a bounded wait that expired) recorded by any kernel
 * since the last call. Synchronises the current device first. Returns
 * FNORM_OK when nothing was recorded, FNORM_ERR_TIMEOUT after an expired
 * wait, FNORM_ERR_CUDA if the word could not be read.
 */
FNORM_API fnorm_status fnorm_get_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
FNORM_API int fnorm_version(void);

/*
 * Tuning and testing (not needed in normal use).
 *
 * The library reads its tuning switches -- environment variables named
 * FNORM_* that force a kernel path or launch shape for experiments and tests
 * (FNORM_FORCE_PATH, FNORM_SPLIT_SHAPE, FNORM_EPI_CLUSTER, FNORM_BN_SPLIT and
 * the others listed with the library's documentation) -- once per process, at
 * the first call that plans a launch. fnorm_tuning_reload() reads them again
 * (after the process changed its environment); it must not run concurrently
 * with any other libfnorm call.
 *
 * fnorm_debug_force_timeout(1) makes one CTA of every later launch that has a
 * bounded-wait test hook (the epilogue range kernels, the split InstanceNorm
 * kernel, the staged and resident BatchNorm kernels) wait, after its last
 * cluster barrier, on a barrier that nothing completes: the wait expires
 * after its 1 s limit, the kernel records FNORM_ERR_TIMEOUT in the device
 * error word (fnorm_get_last_error) and returns, and the results are still
 * written. fnorm_debug_force_timeout(0) turns it off (the default). It exists
 * to test the failure path; no environment variable enables it.
 */
FNORM_API void fnorm_tuning_reload(void);
FNORM_API void fnorm_debug_force_timeout(int on);

/*
 * fnorm_debug_fail_launches(n): the next n calls of the computing entry
 * points that pass their argument checks return FNORM_ERR_CUDA without
 * launching anything, as a failed launch would (outputs untouched). n <= 0
 * clears it. It exists to test callers' error paths; nothing else sets it.
 *
 * Every computing entry point also opens an NVTX range named after itself
 * around its planning and launches, for profilers that collect NVTX.
 */
FNORM_API void fnorm_debug_fail_launches(int n);

#ifdef __cplusplus
}
#endif

#endif /* FNORM_H */
