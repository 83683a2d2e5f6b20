/*
 * b200norm.h -- C ABI of the fused residual-add + normalization kernels for
 * NVIDIA GB300 (sm_103a).
 *
 * Operators (ONNX Runtime contrib operators, as described by the README pages
 * of the webgpu-kernels packages):
 *   b200norm_skip_rms    com.microsoft.SkipSimplifiedLayerNormalization
 *   b200norm_gated_rms   com.microsoft.GatedRMSNorm
 *   b200norm_skip_group  com.microsoft.SkipGroupNorm
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer to a dense, contiguous,
 *     row-major tensor owned by the caller.  The library never allocates,
 *     frees or synchronises; it only enqueues kernels on `stream`.
 *   - Pointers need only be aligned to their element size.  16-byte aligned
 *     pointers (with spans that are whole 16-byte vectors) take the vector
 *     path; anything else takes a scalar path with identical results.
 *   - Element types: B200NORM_F32 (IEEE binary32), B200NORM_F16 (IEEE
 *     binary16) and B200NORM_BF16 (bfloat16: the upper half of a binary32).
 *     The pages' type constraints list float32 and float16 only, and the
 *     GatedRMSNorm README, Description, says bfloat16 is not implemented
 *     there; this library adds it as a storage type with the same arithmetic
 *     (binary32 compute, one rounding to nearest-even at each store).  For
 *     SkipGroupNorm the gamma/beta type M is B200NORM_F32 or T itself, and
 *     also B200NORM_F16 when T is B200NORM_F32; other pairs return
 *     B200NORM_ERR_UNSUPPORTED.
 *   - Rounding: the residual sum S is formed in binary32 as
 *     (x + skip) + bias -- no add at all when bias is NULL -- and rounded once
 *     to nearest-even at the tensor type; statistics are taken over that
 *     rounded S (SkipGroupNorm README, Description).  Every later
 *     intermediate is binary32; only the final store narrows to T.
 *   - Outputs must not overlap any input or each other
 *     (B200NORM_ERR_INVALID_ARGUMENT).
 *   - Argument errors are reported before anything is enqueued.  Launch
 *     failures return B200NORM_ERR_CUDA.  A call on empty tensors returns
 *     B200NORM_OK and enqueues nothing.
 *   - b200norm_last_error() returns a thread-local, human-readable reason for
 *     the last non-OK status returned on the calling thread.
 *   - Calls are stateless apart from the caller-provided SkipGroupNorm
 *     workspace, and may be issued from several host threads at once.
 *   - Kernels are launched with programmatic dependent launch allowed: one
 *     may be scheduled while the previous kernel on the stream drains, but it
 *     waits for that kernel to complete (and its writes to be visible) before
 *     touching memory, so stream order is kept.
 */
#ifndef B200NORM_H
#define B200NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define B200NORM_API __attribute__((visibility("default")))
#else
#define B200NORM_API
#endif

/* Same object as cudaStream_t (declared here so that this header does not
 * need the CUDA headers).  NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* b200norm_stream_t;

typedef enum {
    B200NORM_F32 = 0,
    B200NORM_F16 = 1,
    B200NORM_BF16 = 2
} b200norm_dtype;

typedef enum {
    B200NORM_OK = 0,
    B200NORM_ERR_INVALID_ARGUMENT = 1, /* bad pointer, shape, attribute or overlap   */
    B200NORM_ERR_UNSUPPORTED = 2,      /* element type or shape the library refuses   */
    B200NORM_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed        */
    B200NORM_ERR_WORKSPACE = 4,        /* SkipGroupNorm workspace missing / too small */
    B200NORM_ERR_DEVICE_TIMEOUT = 5    /* a device-side wait gave up (see below)      */
} b200norm_status;

/* Contract version of this ABI (1). */
B200NORM_API int b200norm_version(void);

/* Static string naming a status code. */
B200NORM_API const char* b200norm_status_string(b200norm_status status);

/* Reason for the last non-OK status returned on the calling thread ("" if
 * none).  The pointer stays valid until the next call on this thread. */
B200NORM_API const char* b200norm_last_error(void);

/*
 * SkipSimplifiedLayerNormalization
 * (com.microsoft.SkipSimplifiedLayerNormalization README: Description,
 * Inputs, Outputs, Attributes):
 *
 *   S[r, j]      = round_T((input[r, j] + skip[r, j]) + bias[j])
 *   output[r, j] = round_T(S[r, j] * (1 / sqrt(mean_j(S[r, :]^2) + epsilon)) * gamma[j])
 *
 *   input, skip          T, (rows, hidden), row-major.  rows is the product of
 *                        the leading axes: (token_count) or (batch * sequence).
 *   gamma                T, (hidden).
 *   bias                 T, (hidden), or NULL when absent.
 *   output               T, (rows, hidden).
 *   input_skip_bias_sum  T, (rows, hidden): receives S; NULL when not requested.
 *   epsilon              >= 0 and not NaN; the operator default is
 *                        9.999999960041972e-13 (float32 of 1e-12).
 *
 * rows == 0 is a no-op.  hidden must be > 0.
 */
B200NORM_API b200norm_status b200norm_skip_rms(const void* input, const void* skip,
                                               const void* gamma, const void* bias, void* output,
                                               void* input_skip_bias_sum, int64_t rows,
                                               int64_t hidden, b200norm_dtype T, float epsilon,
                                               b200norm_stream_t stream);

/*
 * Same as b200norm_skip_rms, and also writes the per-row statistics outputs
 * that the operator schema lists (SkipSimplifiedLayerNormalization README,
 * Outputs: mean, inv_std_var, element type U = float32, shape of the input
 * with the last axis replaced by 1):
 *   mean[r]        = 0 (the simplified form does not centre the row)
 *   inv_std_var[r] = 1 / sqrt(mean_j(S[r, :]^2) + epsilon)
 * Either pointer may be NULL.  Both are float32 device arrays of `rows`.
 */
B200NORM_API b200norm_status b200norm_skip_rms_stats(const void* input, const void* skip,
                                                     const void* gamma, const void* bias,
                                                     void* output, void* input_skip_bias_sum,
                                                     float* mean, float* inv_std_var,
                                                     int64_t rows, int64_t hidden,
                                                     b200norm_dtype T, float epsilon,
                                                     b200norm_stream_t stream);

/*
 * GatedRMSNorm (com.microsoft.GatedRMSNorm README: Description, Inputs,
 * Attributes):
 *
 *   for each contiguous span r of C elements (rows = numel / C):
 *   y[r, j] = round_T(x[r, j] * (1 / sqrt(mean_j(x[r, :]^2) + epsilon))
 *                     * scale[j] * SiLU(gate[r, j])),   SiLU(g) = g / (1 + e^-g)
 *
 *   x, gate, y   T, numel elements (any rank >= 1, folded to (numel / C, C)).
 *   scale        T, C elements: (C), (1, C) and (C, 1) are the same vector.
 *   numel        must be a multiple of C; numel == 0 is a no-op.
 *   C            > 0.
 *   epsilon      >= 0 and not NaN; operator default 1e-5.
 *
 * Every intermediate, SiLU included, is binary32.
 */
B200NORM_API b200norm_status b200norm_gated_rms(const void* x, const void* gate,
                                                const void* scale, void* y, int64_t numel,
                                                int64_t C, b200norm_dtype T, float epsilon,
                                                b200norm_stream_t stream);

/* Synchronise `stream`, then read the device-side record of the pipelined row
 * schedule on the current device.  SkipSimplifiedLayerNormalization and
 * GatedRMSNorm calls with short rows (at most 32 16-byte vectors) may run a
 * kernel that streams its inputs through shared memory; its waits on copy
 * completion are bounded (about one second), and one that gives up records
 * B200NORM_ERR_DEVICE_TIMEOUT in a per-device word and returns early (that
 * call's outputs are then undefined).  Returns B200NORM_OK, or
 * B200NORM_ERR_DEVICE_TIMEOUT (and clears the record) if any such launch on
 * the device gave up since the last call; B200NORM_ERR_CUDA if the read
 * failed.  No correct launch records anything. */
B200NORM_API b200norm_status b200norm_rows_status(b200norm_stream_t stream);

/*
 * SkipGroupNorm (com.microsoft.SkipGroupNorm README: Description, Inputs,
 * Outputs, Attributes, Type constraints):
 *
 *   S = round_T((X + skip) + bias)                          (bias may be NULL)
 *   Y = round_T(act((S - mean) * rstd * gamma[c] + beta[c])), evaluated in
 *       binary32, rstd = 1 / sqrt(var + epsilon), act = SiLU (z / (1 + e^-z))
 *       when activation == 1, identity when 0.
 *   mean and var (population) are taken per batch item n and group g over the
 *   C / groups channels of g and every spatial position.
 *
 *   x, y, s   T.  Physical layout (N, H, W, C) when channels_last != 0, else
 *             (N, C, H, W).  N, C, H, W below are the LOGICAL sizes.
 *   skip      T.  skip_rank / skip_dims give its shape:
 *               - exactly x's physical shape                     full skip;
 *               - (N, C) or (N, 1, 1, C)       one value per (n, c), at
 *                                              offset n * C + c, both layouts.
 *             A (N, 1, 1, C) skip when H == W == 1 is an exact match and takes
 *             the full route (same offsets, same results).
 *   bias      T, (C), or NULL.
 *   gamma, beta  M, (C).  M is B200NORM_F32 or T, or B200NORM_F16 when T is
 *             B200NORM_F32.
 *   s         receives S when not NULL.
 *   groups    > 0 and must divide C.
 *   activation  0 (none) or 1 (SiLU); required.
 *   epsilon   >= 0 and not NaN; operator default 1e-5.
 *   workspace device memory of at least
 *             b200norm_skip_group_workspace_size(...) bytes, 256-byte aligned,
 *             ZERO-FILLED before its first use (b200norm_workspace_init does
 *             that).  A call that completes normally leaves it ready for the
 *             next call.  Calls that share a workspace must not overlap on the
 *             device (enqueue them on one stream).
 *
 * Device-side waits inside the kernels (on other CTAs at a grid barrier, or
 * on a bulk copy into shared memory) are bounded: a wait that does not
 * complete within about one second makes the kernel record
 * B200NORM_ERR_DEVICE_TIMEOUT in the workspace and return early (outputs are
 * then undefined).  b200norm_workspace_status() reads that record.
 */
B200NORM_API size_t b200norm_skip_group_workspace_size(int64_t N, int64_t C, int64_t H,
                                                       int64_t W, int groups, b200norm_dtype T,
                                                       int channels_last);

B200NORM_API b200norm_status b200norm_skip_group(
    const void* x, const void* skip, int skip_rank, const int64_t* skip_dims, const void* bias,
    const void* gamma, const void* beta, void* y, void* s, int64_t N, int64_t C, int64_t H,
    int64_t W, b200norm_dtype T, b200norm_dtype M, int groups, float epsilon, int activation,
    int channels_last, void* workspace, size_t workspace_bytes, b200norm_stream_t stream);

/*
 * SkipGroupNorm without a workspace, for callers that cannot allocate device
 * memory: for example a plugin whose host passes it only its input and output
 * buffers and provides no allocator, or a service that reserved its device
 * memory up front and must not allocate (and possibly fail or synchronise)
 * while serving a request.  The operator pages have no counterpart of this
 * entry point; it exists only because of that constraint.
 *
 * Arguments and results are those of b200norm_skip_group without
 * `workspace` / `workspace_bytes`.  Instead the library uses a fixed scratch
 * array of 256 + 2 MiB bytes in device memory, which every GPU that loads
 * the library holds until the process exits.  A call fits exactly when
 * b200norm_skip_group_workspace_size() of its shape is at most that size;
 * with L = C / groups * H * W, NHWC shapes with at most 32 groups and
 * N * ceil(L / 4096) <= 4,096 fit, and NCHW shapes fit when
 * N * groups * ceil(L / 4096) <= 131,072.  A larger shape returns
 * B200NORM_ERR_UNSUPPORTED (see b200norm_last_error); use
 * b200norm_skip_group with a workspace for it.  Every argument is checked
 * before anything is enqueued, as for b200norm_skip_group: a call that
 * returns an error has enqueued nothing.  No call allocates or frees memory.
 *
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current, and keeps it for the
 *     life of the process: make that first call before any stream capture
 *     begins, and do not use the library across a cudaDeviceReset().
 *   - Each call clears the scratch's barrier counters on `stream` before its
 *     kernels; the slots keep the previous call's contents and are always
 *     written before they are read.
 *   - A bounded device-side wait that gives up (see b200norm_skip_group)
 *     records B200NORM_ERR_DEVICE_TIMEOUT in the scratch, where it stays,
 *     through later calls, until b200norm_skip_group_noalloc_status() reads
 *     and clears it.
 *   - All calls on a device share the one array: calls whose work overlaps on
 *     the GPU (different streams without ordering between them) race and give
 *     undefined results.  Order them, e.g. issue them on one stream.
 */
B200NORM_API b200norm_status b200norm_skip_group_noalloc(
    const void* x, const void* skip, int skip_rank, const int64_t* skip_dims, const void* bias,
    const void* gamma, const void* beta, void* y, void* s, int64_t N, int64_t C, int64_t H,
    int64_t W, b200norm_dtype T, b200norm_dtype M, int groups, float epsilon, int activation,
    int channels_last, b200norm_stream_t stream);

/* Synchronise `stream`, then read and clear the device-side error record of
 * b200norm_skip_group_noalloc's scratch on the current device: B200NORM_OK,
 * or B200NORM_ERR_DEVICE_TIMEOUT if a bounded wait of an earlier call gave up
 * (that call's outputs are undefined).  B200NORM_ERR_CUDA if the copy failed.
 * Allocates nothing. */
B200NORM_API b200norm_status b200norm_skip_group_noalloc_status(b200norm_stream_t stream);

/* Zero-fill a SkipGroupNorm workspace (cudaMemsetAsync on `stream`). */
B200NORM_API b200norm_status b200norm_workspace_init(void* workspace, size_t workspace_bytes,
                                                     b200norm_stream_t stream);

/* Synchronise `stream`, then read the workspace's device-side error record:
 * B200NORM_OK, or B200NORM_ERR_DEVICE_TIMEOUT if a bounded wait gave up (the
 * workspace must then be re-initialised).  B200NORM_ERR_CUDA if the copy
 * failed. */
B200NORM_API b200norm_status b200norm_workspace_status(const void* workspace,
                                                       b200norm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* B200NORM_H */
