/*
 * ce.h -- fused softmax cross-entropy forward + gradient on one GB300 GPU.
 *
 * The operation is the GPU-fused cross-entropy loss of the rumus project page
 * (milestone M7a: log-sum-exp stabilised, with the gradient computed in the
 * same pass as the loss), whose per-row steps are Pass 1 (Steps 1-4) of the
 * cross_entropy.wgsl source page of rumus 0.1.1 and whose batch reduction is
 * that page's Pass 2.  For logits z[B][C] and integer targets t[B]:
 *
 *   l_b       = logsumexp(z_b) - z_b[t_b]                      (per row)
 *   *loss_out = (1/B) * sum_b l_b                               (one fp32)
 *   grad[b][c] = (softmax(z_b)[c] - [c == t_b]) / B             ([B][C])
 *
 * Every entry point is plain C: device or host pointers and sizes, no
 * framework types.  All device pointers are owned by the caller.
 */
#ifndef CE_H
#define CE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the logits and of the gradient (always the same type). */
typedef enum {
    CE_F32 = 0,  /* IEEE fp32                                           */
    CE_BF16 = 1, /* bfloat16; computed in fp32, gradient rounded to nearest even */
    CE_F16 = 2   /* IEEE fp16 (binary16); computed in fp32, gradient rounded to
                    nearest even (subnormal results kept)                */
} ce_dtype;

/* Return codes.  Host-detectable errors return before anything is launched. */
typedef enum {
    CE_OK = 0,
    CE_ERR_NULL = 1,     /* a required pointer is NULL                          */
    CE_ERR_SHAPE = 2,    /* B < 1, C < 1, B or C above 2^31-1, or bytes overflow */
    CE_ERR_DTYPE = 3,    /* dtype is not a ce_dtype                             */
    CE_ERR_ALIGN = 4,    /* a pointer is not aligned to its element size        */
    CE_ERR_CUDA = 5,     /* a CUDA runtime call failed (see ce_last_cuda_error) */
    CE_ERR_OVERLAP = 6,  /* an output (grad_out, loss_out) overlaps an input or
                            the other output                                    */
    CE_ERR_POINTER = 7,  /* a pointer is not accessible from the current device */
    CE_ERR_CAPTURE = 8,  /* the call needs to grow its workspace while the
                            stream is being captured; call once uncaptured first */
    CE_ERR_PATH = 9,     /* a forced path/split cannot run this shape           */
    CE_ERR_SCRATCH = 10, /* ce_fwd_bwd_noalloc: more rows than its static scratch
                            array holds                                          */
    CE_ERR_REDUCTION = 11 /* reduction is not a ce_reduction                    */
} ce_status;

/* How the row losses l_b are reduced (ce_fwd_bwd_ex, ce_forward). */
typedef enum {
    CE_REDUCE_MEAN = 0, /* loss_out[0] = (1/B) sum_b l_b; grad = (softmax - onehot) / B  */
    CE_REDUCE_SUM = 1,  /* loss_out[0] = sum_b l_b;       grad = softmax - onehot        */
    CE_REDUCE_NONE = 2  /* loss_out[b] = l_b ([B] fp32);  grad row b = d l_b / d z_b      */
} ce_reduction;

/* Kernel paths (for ce_fwd_bwd_path and ce_query_plan). */
typedef enum {
    CE_PATH_AUTO = 0,      /* let the library choose                                */
    CE_PATH_ROWS_WARP = 1, /* one warp per row, rows staged by TMA: rows of up to
                              8 KB held in registers, rows of up to 48 KB swept in
                              shared memory (CE_PATH_AUTO takes the swept form
                              where 8 warps per SM fit, up to ~27 KB)             */
    CE_PATH_ROW_SPLIT = 2, /* rows (or row slices across a cluster of `split` CTAs)
                              staged once in shared memory by TMA                    */
    CE_PATH_STREAM = 3,    /* any row: chunk partials, then a recompute-and-write
                              pass (a second launch; logits read twice from HBM)    */
    CE_PATH_ROW_TWOPASS = 4, /* any row, one CTA per row: a running max and sum over
                              chunks staged by TMA, then the gradient from a second
                              read of the row (served by L2).  CE_PATH_AUTO takes it
                              for rows one CTA cannot hold in registers             */
    CE_PATH_ROWS_ONLINE = 5 /* the loss alone (grad_out NULL), any row: one warp per
                              row, read once from global memory with a running max
                              and a rescaled sum per lane.  CE_PATH_AUTO takes it
                              for the loss alone on rows past 8 KB in batches of
                              at least 8 rows per SM.  With a gradient, or for the
                              softmax forward: CE_ERR_PATH                          */
} ce_path;

/*
 * ce_fwd_bwd -- loss and gradient of softmax cross-entropy over rows.
 *
 *   logits    device, [B][C] row-major contiguous, element type `dtype`
 *             (row b starts at element b*C); read only.
 *   targets   device, [B] int32 class indices.  A target outside [0, C) is a
 *             data error, not a launch error: that row's loss is NaN (so
 *             *loss_out is NaN), its gradient is softmax/B with no one-hot
 *             term, and the per-stream device error count is incremented
 *             (read it with ce_get_device_errors).  Nothing traps.
 *   B, C      rows and classes, 1 <= B, C <= 2^31-1.
 *   dtype     a ce_dtype.  (f16 is the half-precision type of the rumus
 *             project page's milestone M11, FP16 mixed precision, whose shaders
 *             run with their scalar type aliased to f16.)
 *   loss_out  device, one fp32: (1/B) * sum_b l_b.  The row losses are summed
 *             in a fixed order, so the value is bitwise reproducible for the
 *             same inputs on the same GPU model, whichever path runs.
 *   grad_out  device, [B][C] row-major contiguous, element type `dtype`; must
 *             not overlap logits, targets or loss_out.
 *   stream    a cudaStream_t (NULL = the legacy default stream).
 *
 * Pointers must be aligned to their element size (4 bytes for fp32 and
 * int32, 2 for bf16 and f16) and accessible from the current device.  The call is
 * asynchronous on `stream`; the first call on a stream (or the first that
 * needs more than before: a larger B, or the streaming path's partials)
 * allocates the stream's small workspace (B floats plus counters) with
 * cudaMalloc, which may synchronise the device.  The outgrown workspace is
 * kept, not freed, until ce_release_workspaces (kernels in flight and CUDA
 * graphs captured earlier still use it).  Calls on one stream are ordered;
 * calls on different streams use different workspaces and may run
 * concurrently.  Returns a ce_status.
 */
int ce_fwd_bwd(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
               float *loss_out, void *grad_out, void *stream);

/*
 * ce_fwd_bwd_path -- ce_fwd_bwd with the kernel path forced (tests, tuning).
 *   path   a ce_path; CE_PATH_AUTO behaves exactly as ce_fwd_bwd.
 *   split  CE_PATH_ROW_SPLIT: CTAs per row (1, 2, 3, 4, 6 or 8; 0 = choose;
 *          f16 rows need slices of at most 64 KB per CTA);
 *          CE_PATH_STREAM: classes per chunk (multiple of 8; 0 = choose);
 *          CE_PATH_ROWS_ONLINE: 1 + the kernel build (0 .. 4; 0 = choose);
 *          ignored otherwise.
 * Returns CE_ERR_PATH when the forced path cannot hold the row in shared
 * memory; otherwise as ce_fwd_bwd.  All paths give results within the same
 * tolerances, and the same loss bits for the same row losses.
 */
int ce_fwd_bwd_path(const void *logits, const int32_t *targets, int64_t B, int64_t C,
                    int dtype, float *loss_out, void *grad_out, void *stream, int path,
                    int split);

/*
 * ce_fwd_bwd_ex -- ce_fwd_bwd with a reduction, an upstream gradient, and an
 * optional gradient.  The rumus project page's backward for this loss (M7a)
 * scales the gradient precomputed in the forward pass by the upstream
 * gradient, a device scalar; this entry point fuses that scale into the
 * gradient's single write.
 *
 *   reduction   a ce_reduction (see above): the loss written to loss_out and
 *               the row factor of the gradient (1/B for the mean, else 1).
 *   grad_scale  device pointer or NULL (= 1): for CE_REDUCE_MEAN and
 *               CE_REDUCE_SUM one fp32 multiplying the whole gradient (the
 *               upstream gradient of the reduced loss); for CE_REDUCE_NONE
 *               [B] fp32, row b's gradient multiplied by grad_scale[b].
 *               Read on the device; 4-byte aligned.
 *   loss_out    device: one fp32 (mean, sum) or [B] fp32 (none).
 *   grad_out    device [B][C] in the logits' dtype, or NULL: loss only (the
 *               gradient is neither computed nor written; the logits are the
 *               only large read and nothing large is written).
 * The sum is formed in the same fixed order as the mean (bitwise
 * reproducible); per-row losses are written directly.  Outputs must not
 * overlap inputs or each other.  Returns a ce_status (CE_ERR_REDUCTION for an
 * unknown reduction).
 */
int ce_fwd_bwd_ex(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
                  int reduction, const float *grad_scale, float *loss_out, void *grad_out,
                  void *stream);

/* ce_fwd_bwd_ex with the kernel path forced, as in ce_fwd_bwd_path. */
int ce_fwd_bwd_ex_path(const void *logits, const int32_t *targets, int64_t B, int64_t C,
                       int dtype, int reduction, const float *grad_scale, float *loss_out,
                       void *grad_out, void *stream, int path, int split);

/*
 * ce_forward -- the loss alone (inference): ce_fwd_bwd_ex with grad_scale and
 * grad_out NULL.  The rumus project page's loss forward (M7a) without the
 * precomputed gradient.
 */
int ce_forward(const void *logits, const int32_t *targets, int64_t B, int64_t C, int dtype,
               int reduction, float *loss_out, void *stream);

/*
 * ce_softmax_fwd -- the row-wise softmax forward of the rumus project page
 * (milestone M8c: row-wise softmax with log-sum-exp stability, forward and
 * backward kernels):
 *   probs_out[b][c] = exp(z[b][c] - m_b) / sum_c' exp(z[b][c'] - m_b)
 * computed by the same kernels as the loss (Steps 1, 2 and 4 of Pass 1 of the
 * cross_entropy.wgsl source page, with no target and no 1/B), written once
 * in the logits' dtype.  logits and probs_out: device, [B][C] row-major,
 * `dtype`, not overlapping.  Asynchronous on `stream`; returns a ce_status.
 */
int ce_softmax_fwd(const void *logits, int64_t B, int64_t C, int dtype, void *probs_out,
                   void *stream);

/* ce_softmax_fwd on a forced path and split, as for ce_fwd_bwd_path. */
int ce_softmax_fwd_path(const void *logits, int64_t B, int64_t C, int dtype, void *probs_out,
                        void *stream, int path, int split);

/*
 * ce_softmax_bwd -- the row-wise softmax backward of the same milestone (M8c):
 *   dx[b][c] = p[b][c] * (dy[b][c] - sum_c' p[b][c'] dy[b][c'])
 * for probabilities p (the forward's output) and the upstream gradient dy,
 * all device [B][C] row-major in `dtype`; the row's dot product is formed in
 * fp32 in a fixed order.  dx may be p or dy itself (in place) but may not
 * overlap them otherwise.  Rows whose bytes are a multiple of 16 and at most
 * 64 KB, with 16-byte aligned tensors, read p and dy once; other rows read
 * them twice.  Asynchronous on `stream`; returns a ce_status.
 */
int ce_softmax_bwd(const void *probs, const void *dy, int64_t B, int64_t C, int dtype,
                   void *dx_out, void *stream);

/*
 * ce_fwd_bwd_host -- ce_fwd_bwd for logits and targets in host memory: the
 * same L (the same bits) and gradient, with the copies to the device made by
 * the library.  logits_host [B][C] in `dtype` and targets_host [B] int32:
 * host memory (page-locked for asynchronous copies; pageable memory works,
 * with copies the host waits for), left unchanged until `stream` reaches the
 * end of the call; loss_host: one fp32 in host memory,
 * written when `stream` reaches the end of the call (synchronise the stream
 * before reading it); grad_out: device [B][C] in `dtype`, as for ce_fwd_bwd
 * (the gradient stays on the device for the backward pass).  The batch goes
 * through in chunks of rows (a multiple of 16 rows, at most 64 MiB of
 * logits each, about a quarter of a smaller batch): a chunk's copy in runs on a library stream while the kernel
 * of the chunk before runs on `stream`, and the call's work all lies between
 * its start and its end on `stream`.  The gradient has the bits of ce_fwd_bwd
 * whenever grad_out is 16-byte aligned.  The library keeps per-stream staging
 * buffers (two chunks) and two helper streams until ce_release_workspaces.
 * Not capturable (CE_ERR_CAPTURE while `stream` is being captured).  Returns a
 * ce_status; argument checks as for ce_fwd_bwd.
 */
int ce_fwd_bwd_host(const void *logits_host, const int32_t *targets_host, int64_t B, int64_t C,
                    int dtype, float *loss_host, void *grad_out, void *stream);

/*
 * ce_fwd_bwd_host_grad -- ce_fwd_bwd_host with the gradient returned to host
 * memory too: grad_host [B][C] in `dtype`, host memory (page-locked for
 * asynchronous copies), written when `stream` reaches the end of the call.
 * Each chunk's gradient is copied out on a second library stream while later
 * chunks are copied in and computed, so the two directions of the copy
 * engines overlap.  The loss and the gradient have the bits of ce_fwd_bwd on
 * 16-byte aligned device buffers.  Staging: two chunks of logits and two of
 * gradient per stream.  Outputs may not overlap the inputs.  Otherwise as
 * ce_fwd_bwd_host.
 */
int ce_fwd_bwd_host_grad(const void *logits_host, const int32_t *targets_host, int64_t B,
                         int64_t C, int dtype, float *loss_host, void *grad_host, void *stream);

/*
 * ce_query_plan -- the launch that ce_fwd_bwd would make for this shape on
 * the current device (path, split, total CTAs, threads per CTA, dynamic shared
 * memory per CTA, kernel launches per call).  Any output pointer may be NULL.
 * The loss alone (grad_out NULL) runs the same launch except on rows past
 * 8 KB in batches of at least 8 rows per SM, which take CE_PATH_ROWS_ONLINE.
 */
int ce_query_plan(int64_t B, int64_t C, int dtype, int *path, int *split, int *ctas,
                  int *threads, int *smem_bytes, int *launches);

/*
 * ce_get_device_errors -- read and clear the device error counters of the
 * workspace used by `stream` on the current device: the number of rows seen
 * with an out-of-range target, and the number of bounded waits that gave up
 * (a copy that never completed; the kernel then skips its work and returns
 * instead of hanging).  Synchronises `stream`.  Either output may be NULL.
 */
int ce_get_device_errors(void *stream, int32_t *bad_targets, int32_t *timeouts);

/*
 * Free every workspace of every device: the current one of each stream and
 * the ones outgrown before.  A workspace that grows (a larger B, or the
 * streaming path, on the same stream) is replaced, not freed, because kernels
 * in flight and CUDA graphs captured with earlier calls still use the old
 * one; a graph keeps working, with its own workspace (whose device error
 * counters ce_get_device_errors no longer reads), until this call.  Call it
 * only when the streams are idle and no graph captured with a library call
 * will be replayed.
 */
int ce_release_workspaces(void);

/*
 * ce_fwd_bwd_noalloc -- ce_fwd_bwd for callers that cannot allocate device
 * memory.  The pages have no counterpart; this entry point exists for the
 * library's users.  Some callers may not call cudaMalloc at all: code that
 * runs under a memory manager which owns the whole device, code with a device
 * memory budget fixed at start-up, and code that must never stall on the
 * implicit device synchronisation cudaMalloc and cudaFree can cause.  This
 * entry point allocates nothing: its scratch (a completion ticket, two error
 * counters and one fp32 loss per row, 1 MiB + 256 bytes in all) lives in a
 * statically sized device array of the library, which every GPU that loads
 * the library holds until the process exits.
 *
 *   Arguments, layout, ownership, checks and results are those of ce_fwd_bwd
 *   (the same kernels, the same bits).  Limit: B <= 262144 rows, any C; a
 *   larger B returns CE_ERR_SCRATCH before any launch.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  Every call shares the one array and clears its
 *   ticket and counters on `stream` first, so calls whose kernels overlap on
 *   the GPU (other streams, other host threads) race and must be serialised
 *   by the caller.  The device error counters of this entry point are not
 *   readable through ce_get_device_errors; an out-of-range target still makes
 *   the loss NaN.
 */
int ce_fwd_bwd_noalloc(const void *logits, const int32_t *targets, int64_t B, int64_t C,
                       int dtype, float *loss_out, void *grad_out, void *stream);

/* Static text for a ce_status value. */
const char *ce_status_string(int status);

/* Text of the last CUDA error seen by this thread in the library ("" if none). */
const char *ce_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* CE_H */
