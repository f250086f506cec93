/*
 * nrc -- normalization-fused, channel-mixing Conv1d blocks on one GB300 (sm_103a).
 *
 * C ABI of libnrc.so.  Three blocks, each stated on a PopcornBench page as a
 * composition of PyTorch modules:
 *
 *   nrc_prenorm_dilconv_residual   "Kimi-K2.6 l2_p12", problem statement:
 *       out = x + Conv1d(ReLU(BatchNorm1d_eval(x))), kernel_size 3,
 *       padding = dilation (so the output length equals L), C_in = C_out.
 *   nrc_conv1d_groupnorm           "FW-GLM-5-1 l2_p35", problem analysis:
 *       Conv1d(C_in -> C_out, kernel_size, stride, padding, dilation, bias
 *       optional) followed by GroupNorm(num_groups, C_out, eps, affine).
 *   nrc_linear_bn_swish            "Kimi-K2.6 l2_p97", problem statement:
 *       Linear(in, out) -> BatchNorm1d(out) (training: batch statistics and
 *       running-stat update; eval: running statistics) -> + scalar bias ->
 *       / divide_value -> x * sigmoid(x).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer to caller-owned, contiguous
 *   memory in PyTorch's default layout: activations (N, C, L) with L fastest,
 *   conv weights (C_out, C_in, 3) with the tap index fastest, Linear weights
 *   (out_features, in_features) with in_features fastest.
 * - The library never allocates.  Scratch space is the caller's `workspace`
 *   (device memory, 256-byte aligned, at least *_workspace_size() bytes).
 *   One exception: nrc_prenorm_dilconv_residual_noalloc keeps its scratch in
 *   a fixed library-owned device array instead (see its block below).
 * - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *   is the legacy default stream).  No call synchronises the host.  The
 *   workspace and outputs must not be reused until the stream has passed the
 *   call.
 * - Stream capture: the device-buffer entry points enqueue only memsets and
 *   kernel launches on `stream`, so a call can be captured into a CUDA graph
 *   and replayed.  A replay gives the same result as the call, bit for bit.
 *   Make the first call on a device outside capture: it sets the kernels'
 *   shared-memory limit and looks up the library's device symbols.  The
 *   host-buffer entries (*_host) use library streams and are not capturable.
 * - Argument errors are reported by the return value before anything is
 *   launched; a failed launch returns NRC_ERR_CUDA.  A device-side wait that
 *   gives up (see nrc_set_wait_timeout_ns) is recorded in the device status
 *   word and reported by nrc_query_status().  No call throws or aborts.
 * - Arithmetic: fp32 storage is computed with three bf16 tensor-core products
 *   per term (hi*hi + lo*hi + hi*lo with v = hi + lo), accumulated in fp32;
 *   bf16 storage with one bf16 product, accumulated in fp32.
 */
#ifndef NRC_H_
#define NRC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NRC_OK = 0,
    NRC_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, overlap, bad value */
    NRC_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels implement */
    NRC_ERR_ALIGNMENT = 3,     /* workspace (or a vector pointer) misaligned */
    NRC_ERR_WORKSPACE = 4,     /* workspace_bytes smaller than the query returned */
    NRC_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
    NRC_ERR_TIMEOUT = 6        /* a device-side wait gave up (nrc_query_status) */
} nrc_status;

typedef enum {
    NRC_F32 = 0,               /* x, out, conv weight and conv bias stored fp32 */
    NRC_BF16 = 1               /* ... stored bf16 (BatchNorm parameters stay fp32) */
} nrc_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *nrc_status_string(nrc_status s);

/* Library version as major*10000 + minor*100 + patch. */
int nrc_version(void);

/* ------------------------------------------------------------------------
 * Pre-norm residual block ("Kimi-K2.6 l2_p12", problem statement)
 *
 *   s_c   = gamma[c] / sqrt(running_var[c] + bn_eps)
 *   z     = max(0, (x - running_mean[c]) * s_c + beta[c])   for 0 <= t < L,
 *           0 outside (the conv's zero padding applies to z, after BN+ReLU)
 *   out[n,o,t] = x[n,o,t] + bias[o]
 *                + sum_c sum_k W[o,c,k] * z[n, c, t - dilation + k*dilation]
 *
 * x, out:        (N, C, L), dtype `dt`.  out must not overlap x.
 * bn_*:          (C) fp32 each (BatchNorm1d eval-mode buffers and affine).
 * conv_weight:   (C, C, 3), dtype `dt`.
 * conv_bias:     (C), dtype `dt`, or NULL for no bias.
 * kernel_size must be 3 and padding must equal dilation (only then does the
 * output length equal L, which the residual add needs): otherwise
 * NRC_ERR_UNSUPPORTED.  dilation >= 1.  C <= 2048.
 * workspace:     >= nrc_prenorm_dilconv_residual_workspace_size(C, dt) bytes;
 *                it receives the repacked weights on every call.
 * ------------------------------------------------------------------------ */
size_t nrc_prenorm_dilconv_residual_workspace_size(int C, nrc_dtype dt);

nrc_status nrc_prenorm_dilconv_residual(
    const void *x, void *out, nrc_dtype dt, int N, int C, int L,
    int kernel_size, int dilation, int padding,
    const float *bn_running_mean, const float *bn_running_var,
    const float *bn_gamma, const float *bn_beta, float bn_eps,
    const void *conv_weight, const void *conv_bias,
    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Pre-norm residual block with BatchNorm1d in TRAINING mode ("Kimi-K2.6
 * l2_p12", the correctness discussion of batch against running statistics;
 * the running-buffer update as "Kimi-K2.6 l2_p97" states it for BatchNorm1d)
 *
 *   mu[c]  = mean of x[:, c, :] over all N*L values
 *   var[c] = mean of (x[:, c, :] - mu[c])^2 over the same values (biased)
 *   out    = the block above with mu, var in place of running_mean, running_var
 *   running_mean[c] <- (1 - bn_momentum)*running_mean[c] + bn_momentum*mu[c]
 *   running_var[c]  <- (1 - bn_momentum)*running_var[c]
 *                      + bn_momentum*var[c]*N*L/(N*L - 1)
 *   *num_batches_tracked += 1
 *
 * Arguments as in nrc_prenorm_dilconv_residual, and:
 * running_mean, running_var: (C) fp32 device buffers, read and updated in
 *   place; either may be NULL (that buffer is neither read nor updated; the
 *   output never depends on them).
 * num_batches_tracked: one int64 on the device, or NULL.
 * bn_momentum: finite (PyTorch's default is 0.1).  N*L >= 2.
 * workspace: >= nrc_prenorm_dilconv_residual_train_workspace_size(N, C, L, dt)
 *   bytes, 16-byte aligned: the eval block's workspace, then a (mean, M2)
 *   partial per 2 KB segment of every row, and the batch mean and variance.
 * Three steps on `stream`: a row-statistics kernel (x read once), a per-channel
 * merge that writes the batch statistics and updates the buffers, then the
 * eval-mode block's launches.  Every argument error returns before the first
 * launch, so a rejected call leaves the buffers untouched.
 * ------------------------------------------------------------------------ */
size_t nrc_prenorm_dilconv_residual_train_workspace_size(int N, int C, int L, nrc_dtype dt);

nrc_status nrc_prenorm_dilconv_residual_train(
    const void *x, void *out, nrc_dtype dt, int N, int C, int L,
    int kernel_size, int dilation, int padding,
    float *bn_running_mean, float *bn_running_var, long long *num_batches_tracked,
    const float *bn_gamma, const float *bn_beta, float bn_eps, float bn_momentum,
    const void *conv_weight, const void *conv_bias,
    void *workspace, size_t workspace_bytes, void *stream);

/* Training-mode block on HOST buffers (end-to-end path; a library
 * convenience, the pages have no counterpart).  Same computation, arguments
 * and errors as nrc_prenorm_dilconv_residual_train, with x_host, out_host,
 * bn_gamma_host, bn_beta_host, conv_weight_host and conv_bias_host in HOST
 * memory (pinned for the copies to overlap), while the running buffers and
 * num_batches_tracked stay DEVICE buffers updated in place.  The batch
 * statistics need every sample first, so the chunks of chunk_n samples (first
 * and last smaller) go through two phases: x is copied into one device copy
 * of the whole batch chunk by chunk, each chunk's row statistics computed
 * behind its copy; after the merge, the block runs on chunk j while chunk
 * j-1's output is copied out.  Two library-owned streams and `stream`,
 * ordered by events.  Results are those of the device entry on the whole batch
 * (the statistics merge in the same order; each chunk's block call uses the
 * one-wave or multi-wave kernel its size asks for, which give bitwise equal
 * results).
 * workspace: DEVICE memory, 256-byte aligned, of at least
 *   nrc_prenorm_dilconv_residual_train_host_workspace_size(N, C, L, dt,
 *   chunk_n) bytes (the device entry's workspace, a device copy of x, two out
 *   chunk buffers and the parameters); chunk_n <= 0 returns
 *   NRC_ERR_INVALID_ARG.  Asynchronous: synchronising `stream` makes out_host
 *   valid.  Calls from several host threads are serialised inside the library. */
size_t nrc_prenorm_dilconv_residual_train_host_workspace_size(int N, int C, int L, nrc_dtype dt,
                                                              int chunk_n);

nrc_status nrc_prenorm_dilconv_residual_train_host(
    const void *x_host, void *out_host, nrc_dtype dt, int N, int C, int L,
    int kernel_size, int dilation, int padding,
    float *bn_running_mean, float *bn_running_var, long long *num_batches_tracked,
    const float *bn_gamma_host, const float *bn_beta_host, float bn_eps, float bn_momentum,
    const void *conv_weight_host, const void *conv_bias_host, int chunk_n,
    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Pre-norm residual block on HOST buffers.  Same computation and errors as
 * nrc_prenorm_dilconv_residual ("Kimi-K2.6 l2_p12", problem statement), for
 * callers whose x and out live in host memory.
 *
 * x_host, out_host: (N, C, L) in host memory, dtype `dt`; page-locked
 *   (cudaHostAlloc / pinned) memory lets the copies overlap the GPU work,
 *   pageable memory still works but serialises.
 * bn_*_host, weight_host, bias_host: as in nrc_prenorm_dilconv_residual but in
 *   host memory (bias_host may be NULL).
 * chunk_n: samples per pipeline chunk (>= 1; clamped to N).  The batch flows
 *   through two device buffers: the copy-in of chunk j+1, the GEMM of chunk j
 *   and the copy-out of chunk j-1 run at once, on two library-owned streams
 *   (created once per device) and `stream`, ordered by events.
 * workspace: DEVICE memory, 256-byte aligned, of at least
 *   nrc_prenorm_dilconv_residual_host_workspace_size(N, C, L, dt, chunk_n)
 *   bytes (weight image, parameters, two x and two out chunk buffers).
 * Asynchronous: work already on `stream` comes first; `stream` resumes after
 * the last copy-out, so synchronising `stream` makes out_host valid.  Calls
 * from several host threads are serialised inside the library (they share the
 * per-device streams); host buffers must stay valid until then.
 * ------------------------------------------------------------------------ */
size_t nrc_prenorm_dilconv_residual_host_workspace_size(int N, int C, int L, nrc_dtype dt,
                                                        int chunk_n);

nrc_status nrc_prenorm_dilconv_residual_host(
    const void *x_host, void *out_host, nrc_dtype dt, int N, int C, int L,
    int kernel_size, int dilation, int padding,
    const float *bn_running_mean_host, const float *bn_running_var_host,
    const float *bn_gamma_host, const float *bn_beta_host, float bn_eps,
    const void *conv_weight_host, const void *conv_bias_host, int chunk_n,
    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Allocation-free pre-norm residual block.  The pages have no counterpart:
 * this is a library convenience, not part of the method.
 *
 * Same computation, arguments and errors as nrc_prenorm_dilconv_residual, but
 * without a workspace: the scratch (the repacked weight image) lives in a
 * fixed array in the library's own device memory, so the call allocates
 * nothing.  It is for callers that cannot hand the library scratch memory --
 * code whose device memory belongs to a host framework's allocator that
 * forbids side allocations, or loops that must not call cudaMalloc/cudaFree.
 *
 * Limit: the array is nrc_prenorm_dilconv_residual_noalloc_max_bytes() (4 MiB),
 * present on every GPU that loads the library until the process exits; it
 * holds fp32 C <= 512 or bf16 C <= 768.  Larger C returns NRC_ERR_WORKSPACE.
 * Argument errors are checked first and return the same codes as
 * nrc_prenorm_dilconv_residual; the size limit is checked next; no CUDA call
 * is made before both pass.
 * The first call on a device looks up the array's device address (one
 * cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  cudaDeviceReset() on a device makes
 * the cached address stale: do not use this entry point on that device after
 * a reset.  All calls share the array and each rewrites what it uses, so
 * nothing needs clearing, but calls that overlap on the GPU (several streams
 * or host threads at once) race on it.
 * ------------------------------------------------------------------------ */
size_t nrc_prenorm_dilconv_residual_noalloc_max_bytes(void);

nrc_status nrc_prenorm_dilconv_residual_noalloc(
    const void *x, void *out, nrc_dtype dt, int N, int C, int L,
    int kernel_size, int dilation, int padding,
    const float *bn_running_mean, const float *bn_running_var,
    const float *bn_gamma, const float *bn_beta, float bn_eps,
    const void *conv_weight, const void *conv_bias, void *stream);

/* ------------------------------------------------------------------------
 * Conv1d + GroupNorm ("FW-GLM-5-1 l2_p35", problem analysis and its
 * normalisation kernel; the module's constructor takes kernel_size, stride,
 * padding, dilation, eps and affine)
 *
 *   T_out    = floor((T + 2*padding - dilation*(kernel_size - 1) - 1) / stride) + 1
 *   y[n,o,t] = bias[o] + sum_c sum_k W[o,c,k] * x[n, c, t*stride - padding + k*dilation]
 *              (x = 0 outside [0, T)),  0 <= t < T_out
 *   group g = o / (C_out / num_groups)
 *   mu, var  = mean and biased variance of y over the group's channels and all t
 *   out      = (y - mu) / sqrt(var + eps) * gamma[o] + beta[o]
 *
 * x: (N, C_in, T) fp32.  out: (N, C_out, T_out) fp32, must not overlap x; when
 * the tiles do not fit one wave of resident CTAs it also holds y between the
 * call's two kernels.
 * conv_weight: (C_out, C_in, kernel_size) fp32.  conv_bias: (C_out) or NULL.
 * gn_gamma, gn_beta: (C_out) fp32, both NULL for affine=False.
 * kernel_size >= 1, stride >= 1, padding >= 0, dilation >= 1 and T_out >= 1
 * (else INVALID_ARG); kernel_size <= 64 (else UNSUPPORTED).
 * C_out % num_groups == 0 (else INVALID_ARG); when C_out > 256 the group
 * size must divide 256 (else UNSUPPORTED).
 * workspace: >= nrc_conv1d_groupnorm_workspace_size(...) bytes with the same
 * shape and conv arguments (0 from the query: invalid arguments).
 * ------------------------------------------------------------------------ */

/* T_out of the conv above, or 0 when the arguments are invalid or the kernel
 * does not fit the padded input. */
int nrc_conv1d_output_length(int T, int kernel_size, int stride, int padding, int dilation);

size_t nrc_conv1d_groupnorm_workspace_size(int N, int C_in, int C_out, int T,
                                           int kernel_size, int stride, int padding,
                                           int dilation, int num_groups);

nrc_status nrc_conv1d_groupnorm(
    const float *x, float *out, int N, int C_in, int C_out, int T,
    int kernel_size, int stride, int padding, int dilation,
    const float *conv_weight, const float *conv_bias,
    int num_groups, const float *gn_gamma, const float *gn_beta, float eps,
    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Conv1d + GroupNorm on HOST buffers (end-to-end path).  The pages have no
 * counterpart: a library convenience.
 *
 * Same computation, arguments and errors as nrc_conv1d_groupnorm, with
 * x_host, out_host, conv_weight_host, conv_bias_host, gn_gamma_host and
 * gn_beta_host in HOST memory (pinned for the copies to overlap).  A sample's
 * group statistics involve that sample alone, so the batch runs in chunks of
 * chunk_n samples (the last one smaller if N asks): the parameters are copied
 * once, then the copy-in of chunk j+1, nrc_conv1d_groupnorm on chunk j and the
 * copy-out of chunk j-1 run at once, on two library-owned streams and
 * `stream`, ordered by events.  Each chunk is an ordinary device-entry call on
 * its samples: the results are bitwise those of the device entry on the whole
 * batch when both take the same kernel path, and agree to rounding otherwise
 * (a chunk whose tiles fit one wave takes the fused one-kernel path where the
 * whole batch may not).
 * workspace: DEVICE memory, 256-byte aligned, of at least
 *   nrc_conv1d_groupnorm_host_workspace_size(..., chunk_n) bytes (the device
 *   entry's workspace for one chunk, the parameters, two x and two out chunk
 *   buffers); 0 from the query: invalid arguments.  chunk_n <= 0 returns
 *   NRC_ERR_INVALID_ARG.
 * Asynchronous: work already on `stream` comes first; `stream` resumes after
 * the last copy-out, so synchronising `stream` makes out_host valid.  Calls
 * from several host threads are serialised inside the library.
 * ------------------------------------------------------------------------ */
size_t nrc_conv1d_groupnorm_host_workspace_size(int N, int C_in, int C_out, int T,
                                                int kernel_size, int stride, int padding,
                                                int dilation, int num_groups, int chunk_n);

nrc_status nrc_conv1d_groupnorm_host(
    const float *x_host, float *out_host, int N, int C_in, int C_out, int T,
    int kernel_size, int stride, int padding, int dilation,
    const float *conv_weight_host, const float *conv_bias_host,
    int num_groups, const float *gn_gamma_host, const float *gn_beta_host, float eps,
    int chunk_n, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Linear + BatchNorm1d + scalar bias + divide + Swish ("Kimi-K2.6 l2_p97")
 *
 *   y = x W^T + lin_bias                                 (B x out_f)
 *   training=1: mu_j, var_j = batch mean and biased variance of column j;
 *               running_mean = (1-m)*running_mean + m*mu
 *               running_var  = (1-m)*running_var  + m*var*B/(B-1)
 *               *num_batches_tracked += 1 (if not NULL)
 *   training=0: mu = running_mean, var = running_var, nothing updated
 *   u   = ((y - mu)/sqrt(var + eps) * gamma + beta + *add_bias) / divide_value
 *   out = u * sigmoid(u)
 *
 * x: (B, in_f) fp32.  out: (B, out_f) fp32, no overlap with x; in training
 * mode it holds y between kernels, in eval mode the GEMM's epilogue writes the
 * result straight into it (one GEMM launch after the x repack, y never stored).  lin_weight: (out_f, in_f).  lin_bias: (out_f) or NULL.
 * bn_gamma/bn_beta: (out_f) or both NULL (1 and 0).  running_mean/var:
 * (out_f), read in eval mode, read and updated in place in training mode.
 * num_batches_tracked: one int64 or NULL.  add_bias: DEVICE pointer to one
 * fp32 value (read on the device, so the call never syncs).  divide_value
 * must be non-zero.  training=1 needs B >= 2 (unbiased variance).
 * momentum in [0, 1].
 * ------------------------------------------------------------------------ */
size_t nrc_linear_bn_swish_workspace_size(int B, int in_f, int out_f);

nrc_status nrc_linear_bn_swish(
    const float *x, float *out, int B, int in_f, int out_f,
    const float *lin_weight, const float *lin_bias,
    const float *bn_gamma, const float *bn_beta,
    float *bn_running_mean, float *bn_running_var, int64_t *num_batches_tracked,
    float bn_eps, float bn_momentum, int training,
    const float *add_bias, float divide_value,
    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Linear + BatchNorm1d + bias + divide + Swish on HOST buffers (end-to-end
 * path).  The pages have no counterpart: a library convenience.
 *
 * Same computation and argument rules as nrc_linear_bn_swish, with x_host
 * (B, in_f), out_host (B, out_f), lin_weight_host (out_f, in_f),
 * lin_bias_host / bn_gamma_host / bn_beta_host (out_f, or NULL as there) and
 * add_bias_host (one value) in HOST memory (pinned for the copies to overlap),
 * while bn_running_mean / bn_running_var (and num_batches_tracked) stay DEVICE
 * buffers, updated in place as in the device entry.
 * Each output feature's batch statistics involve that feature alone, so the
 * call runs in chunks of chunk_f output features (rounded up to whole 128-
 * feature tiles; the first and last chunks are smaller): x is copied in and
 * packed once, then the copy-in of chunk j+1's weight rows, the chain of
 * chunk j (GEMM, and in training mode the finalize and normalize kernels) and
 * the copy-out of chunk j-1's columns run at once, on two library-owned
 * streams (created once per device) and `stream`, ordered by events.  Results
 * are bitwise those of nrc_linear_bn_swish.
 * workspace: DEVICE memory, 256-byte aligned, of at least
 *   nrc_linear_bn_swish_host_workspace_size(B, in_f, out_f, chunk_f) bytes
 *   (the x image and statistics for one chunk, x, the parameters, two weight
 *   and two output chunk buffers); 0 from the query: invalid arguments.
 * Errors: those of nrc_linear_bn_swish, and NRC_ERR_INVALID_ARG for
 * chunk_f <= 0.
 * Asynchronous: work already on `stream` comes first; `stream` resumes after
 * the last copy-out, so synchronising `stream` makes out_host valid.  Calls
 * from several host threads are serialised inside the library.
 * ------------------------------------------------------------------------ */
size_t nrc_linear_bn_swish_host_workspace_size(int B, int in_f, int out_f, int chunk_f);

nrc_status nrc_linear_bn_swish_host(
    const float *x_host, float *out_host, int B, int in_f, int out_f,
    const float *lin_weight_host, const float *lin_bias_host,
    const float *bn_gamma_host, const float *bn_beta_host,
    float *bn_running_mean, float *bn_running_var, int64_t *num_batches_tracked,
    float bn_eps, float bn_momentum, int training,
    const float *add_bias_host, float divide_value, int chunk_f,
    void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Status and fault handling
 * ------------------------------------------------------------------------ */
/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns NRC_OK, NRC_ERR_TIMEOUT (a device wait gave up; the
 * kernel returned early and its outputs are undefined) or NRC_ERR_CUDA. */
nrc_status nrc_query_status(void *stream);

/* Where the last recorded device error happened (a wait-site id, 0 if none). */
int nrc_last_error_site(void);

/* Limit of every device-side wait, in nanoseconds (default 2e9).  Applies to
 * launches made after the call. */
void nrc_set_wait_timeout_ns(uint64_t ns);

/* Limit of ONE wait site only: the grid-wide barrier of the one-wave
 * Conv1d + GroupNorm kernel (wait site 9), where every CTA has finished its
 * copies and MMAs before it waits.  ns = 0 returns that site to the general
 * limit above.  A wait that gives up there records NRC_ERR_TIMEOUT (site 9),
 * and the CTA returns without normalising its tile; the next call, made with
 * the limit restored, is unaffected.  This exists to exercise a real kernel's
 * give-up path; every other wait keeps the general limit.  Applies to
 * launches made after the call. */
void nrc_set_grid_barrier_timeout_ns(uint64_t ns);

/* Fault-path self test: launches one CTA whose thread waits, with the given
 * limit, on an mbarrier that nothing ever arrives at.  The wait gives up and
 * records NRC_ERR_TIMEOUT exactly like a stalled pipeline would; the launch
 * itself returns NRC_OK.  Read the outcome with nrc_query_status. */
nrc_status nrc_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* ------------------------------------------------------------------------
 * Launch trace (device timing of the library's own kernels)
 * ------------------------------------------------------------------------ */
/* on=1: drop earlier records and bracket every kernel launch made from now on
 * with two CUDA events recorded on the launch's stream; on=0: stop recording
 * (records are kept for reading). */
void nrc_trace_enable(int on);

/* Number of launches recorded since tracing was last enabled. */
int nrc_trace_count(void);

/* Record i: the kernel's name (static string) and its device duration in ms
 * (waits for the record's end event). */
nrc_status nrc_trace_get(int i, const char **name, float *ms);

#ifdef __cplusplus
}
#endif
#endif /* NRC_H_ */
