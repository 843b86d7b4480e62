/*
 * gn.h -- C ABI of libgn.so: GroupNorm forward and backward on NVIDIA GB300
 * (sm_103a), hand-written CUDA kernels behind plain pointers and sizes.
 *
 * The operation ("Kimi-K2.6 l1_p35" POPCORNBENCH transcript, opening problem
 * analysis; "baracuda-kernels src/norm/group_norm_backward.rs", module comment
 * and GroupNormBackwardArgs): an activation [N, C, *spatial] is viewed as
 * [N, C, HW] with HW = product of the spatial extents.  The C channels form G
 * groups of Cg = C/G consecutive channels.  For every sample n and group g,
 *     mean = average of x over the Cg*HW elements of (n, g)
 *     var  = biased variance over the same elements (divisor Cg*HW)
 *     rstd = 1 / sqrt(var + eps)
 *     y    = (x - mean) * rstd * gamma[c] + beta[c]
 * and the backward, with g_i = gamma[c] * dy_i and xhat = (x - mean) * rstd,
 *     dx     = rstd * (g - avg_(n,g)(g) - xhat * avg_(n,g)(g * xhat))
 *     dgamma[c] = sum over n, hw of dy * xhat
 *     dbeta[c]  = sum over n, hw of dy
 *
 * Memory layouts ("Fix GroupNorm NHWC one-pass backward execution",
 * NVIDIA/apex PR #2018, reproducer: channels_last activations):
 *     GN_LAYOUT_NCHW: element (n, c, hw) at offset (n*C + c)*HW + hw
 *     GN_LAYOUT_NHWC: element (n, c, hw) at offset (n*HW + hw)*C + c
 * gn_fwd / gn_bwd take tensors densely packed in one of these layouts;
 * gn_fwd_ex / gn_bwd_ex (below) take strided views.
 *
 * Types: x, y, dy, dx are all of `dtype` (fp32, fp16, bf16 or fp64); every
 * reduction and every intermediate is fp32.  gamma, beta, dgamma, dbeta are
 * fp32 [C]; mean and rstd are fp32 [N*G] indexed n*G + g.  y and dx are
 * rounded once, to nearest even, from fp32.  fp64 is a storage type
 * ("baracuda-kernels src/norm/group_norm_backward.rs", GroupNormBackwardPlan::
 * select: f64 among the wired element types, under a precision guarantee of
 * fp32 math with an fp32 accumulator): its values are converted to fp32 on
 * load and written back exactly; it runs on the two-kernel path only.
 *
 * Ownership and execution: every pointer except `workspace_bytes`-sized
 * scalars is a DEVICE pointer owned by the caller.  The library allocates
 * nothing; each call validates its arguments on the host and then enqueues its
 * kernels asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 * stream) of the current device.  Results are bit-identical from run to run
 * for the same arguments on the same device.
 *
 * Workspace: a caller-provided device buffer of at least gn_workspace_size()
 * bytes, 16-byte aligned, borrowed for the duration of the call ("baracuda-
 * kernels src/norm/group_norm_backward.rs", workspace_size / run: the caller
 * lends scratch memory sized by the plan).  Its contents are dead between
 * calls: it may hold anything when a call starts (fresh from a caching
 * allocator, or left by a call of another shape), because every call first
 * zero-fills, on `stream`, the few bytes at its start that hold the error
 * word (offset 0) and the arrival counters of its cross-CTA reductions, and
 * only then runs its kernels.  The rest is scratch that each call writes
 * before it reads.  Two calls that are in flight at the same time must not
 * share one workspace.
 */
#ifndef GN_H_
#define GN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GN_API __attribute__((visibility("default")))
#else
#define GN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gn_layout { GN_LAYOUT_NCHW = 0, GN_LAYOUT_NHWC = 1 } gn_layout;
typedef enum gn_dtype {
  GN_DTYPE_F32 = 0,
  GN_DTYPE_F16 = 1,
  GN_DTYPE_BF16 = 2,
  GN_DTYPE_F64 = 3 /* storage only: fp32 arithmetic (see above) */
} gn_dtype;
typedef enum gn_op { GN_OP_FWD = 0, GN_OP_BWD = 1 } gn_op;

/* Status codes ("baracuda-kernels src/norm/group_norm_backward.rs",
 * GroupNormBackwardPlan::select / can_implement / run: invalid problems,
 * unsupported element types, a workspace that is too small). */
typedef enum gn_status {
  GN_OK = 0,
  GN_ERR_INVALID = 1,     /* bad sizes, G not dividing C, missing or overlapping buffers */
  GN_ERR_UNSUPPORTED = 2, /* unknown layout or dtype, or a problem too large to launch */
  GN_ERR_WORKSPACE = 3,   /* workspace NULL, not 16-byte aligned or smaller than gn_workspace_size() */
  GN_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed (see gn_last_cuda_error) */
  GN_ERR_TIMEOUT = 5      /* gn_workspace_status only: a bounded wait inside a kernel of the
                             last call on that workspace ran out, so that call's outputs are
                             not valid */
} gn_status;

/* Bytes of workspace that gn_fwd (op = GN_OP_FWD) or gn_bwd (op = GN_OP_BWD)
 * needs for this problem on the current device; the value is the same for
 * both ops, so one workspace serves a forward and its backward.  0 for
 * invalid or empty problems.  Host-only: launches nothing.  ("baracuda-kernels
 * src/norm/group_norm_backward.rs", workspace_size.) */
GN_API size_t gn_workspace_size(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
                         int dtype);

/* Forward.  Reads x [N, C, HW] (layout, dtype), gamma [C] and beta [C]
 * (either may be NULL: weight 1 / bias 0).  Writes y (same shape, layout and
 * dtype as x), mean [N*G] and rstd [N*G].  y may be the same buffer as x
 * (in place); any other overlap between y, x, mean and rstd is rejected.
 * N, C or HW equal to 0: returns GN_OK and launches nothing.
 * Errors are reported before anything is enqueued, except GN_ERR_CUDA from a
 * failed launch. */
GN_API int gn_fwd(const void* x, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
           const float* gamma, const float* beta, float eps, void* y, float* mean, float* rstd,
           void* workspace, size_t workspace_bytes, void* stream);

/* Backward ("baracuda-kernels src/norm/group_norm_backward.rs",
 * GroupNormBackwardArgs: dy, x, gamma, saved mean, saved rstd -> dx, dgamma,
 * dbeta).  mean and rstd are the forward's outputs for the same x.  gamma may
 * be NULL (weight 1).  dgamma and dbeta may each be NULL (not computed).
 * dx may be the same buffer as dy (in place); any other overlap is rejected.
 * N or C equal to 0: GN_OK, nothing launched.  HW equal to 0 (or N == 0 with
 * C > 0): dgamma and dbeta, when given, are set to 0 (an empty sum) with
 * cudaMemsetAsync and no kernel is launched. */
GN_API int gn_bwd(const void* dy, const void* x, const float* mean, const float* rstd,
           const float* gamma, int64_t N, int64_t C, int64_t HW, int64_t G, int layout,
           int dtype, void* dx, float* dgamma, float* dbeta, void* workspace,
           size_t workspace_bytes, void* stream);

/* Strided views ("baracuda-kernels src/norm/group_norm_backward.rs",
 * GroupNormBackwardPlan::select: the plan takes views of rank 2 to 8; "Kimi-
 * K2.6 l1_p35" POPCORNBENCH transcript, on inputs that are not contiguous).
 * gn_fwd_ex and gn_bwd_ex are gn_fwd and gn_bwd on views whose elements lie
 * at
 *     GN_LAYOUT_NCHW: base + n*sn + c*sr + hw       (each channel plane contiguous)
 *     GN_LAYOUT_NHWC: base + n*sn + hw*sr + c       (each spatial row contiguous)
 * with strides in elements, one (sn, sr) pair per tensor -- for example a
 * slice of the channels of a wider tensor, or planes padded to a row pitch.
 * The dense strides are (C*HW, HW) for NCHW and (HW*C, C) for NHWC; with those
 * the calls are gn_fwd / gn_bwd exactly.  A stride may be anything when its
 * extent is 1 (sn when N == 1; sr when C == 1 for NCHW, HW == 1 for NHWC);
 * otherwise the strides must keep elements apart -- planes (rows) laid out
 * sample-major (sn >= count*sr, sr >= run) or plane(row)-major (sr >= N*sn,
 * sn >= run), with run = HW (NCHW) or C (NHWC) -- else GN_ERR_INVALID.
 * Outputs may be their input in place only with identical strides; an output
 * whose address span meets an input's span is otherwise rejected, even when
 * the views interleave without sharing an element.  Views that are not dense
 * run on the two-kernel path; they take 16-byte vectors when every base and
 * every stride (times the element size) is a multiple of 16 bytes, the scalar
 * path otherwise.  Workspace, statistics, parameters, errors and execution
 * are as for gn_fwd / gn_bwd; gn_workspace_size covers these calls too. */
GN_API int gn_fwd_ex(const void* x, int64_t x_sn, int64_t x_sr, int64_t N, int64_t C, int64_t HW,
                     int64_t G, int layout, int dtype, const float* gamma, const float* beta,
                     float eps, void* y, int64_t y_sn, int64_t y_sr, float* mean, float* rstd,
                     void* workspace, size_t workspace_bytes, void* stream);
GN_API int gn_bwd_ex(const void* dy, int64_t dy_sn, int64_t dy_sr, const void* x, int64_t x_sn,
                     int64_t x_sr, const float* mean, const float* rstd, const float* gamma,
                     int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype, void* dx,
                     int64_t dx_sn, int64_t dx_sr, float* dgamma, float* dbeta, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Size of the device scratch area that gn_fwd_static_ws uses (per device). */
#define GN_STATIC_WS_BYTES ((size_t)4 << 20)

/* gn_fwd for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this entry point exists for the library's users.)  Some callers
 * have no way to provide the workspace gn_fwd asks for: serving code that runs
 * under a fixed memory budget and must not allocate once it has started,
 * plugins whose host framework gives them no allocator, and code running where
 * calling cudaMalloc is not permitted.  This call takes the same arguments as
 * gn_fwd without the workspace, and computes the same results with the same
 * kernels, using instead a scratch area that the library holds in a statically
 * sized device array of GN_STATIC_WS_BYTES bytes.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *  - The array is reserved on every device that loads the library and stays
 *    reserved until the process exits.
 *  - A problem whose gn_workspace_size(GN_OP_FWD, ...) exceeds
 *    GN_STATIC_WS_BYTES is rejected with GN_ERR_WORKSPACE before anything is
 *    enqueued.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Each call clears the part of the array it uses (cudaMemsetAsync on
 *    `stream`) before its kernels run.
 *  - All calls share the one array: calls that overlap on the GPU (on two
 *    streams, or from two host threads) race and must not be made. */
GN_API int gn_fwd_static_ws(const void* x, int64_t N, int64_t C, int64_t HW, int64_t G,
                            int layout, int dtype, const float* gamma, const float* beta,
                            float eps, void* y, float* mean, float* rstd, void* stream);

/* Outcome of the kernels of the last gn_fwd / gn_bwd / gn_fwd_static_ws call
 * that ran on `workspace` (enqueued on `stream`): waits for `stream`, reads
 * the workspace's error word (offset 0) and returns GN_OK when every bounded
 * wait of those kernels completed, GN_ERR_TIMEOUT when one ran out (the
 * call's outputs are then not valid; the next call on the workspace clears
 * the word again), GN_ERR_WORKSPACE for a NULL or misaligned workspace, or
 * GN_ERR_CUDA.  Kernels that wait on other CTAs bound every wait (in time,
 * about 0.2 s, or in polls); a wait that runs out sets the word instead of
 * hanging, and the kernel then returns. */
GN_API int gn_workspace_status(const void* workspace, void* stream);

/* Fault injection, a test hook (process-wide).
 *   GN_FAULT_NONE   normal operation (the default).
 *   GN_FAULT_LAUNCH every gn_fwd / gn_bwd returns GN_ERR_CUDA after validating
 *                   its arguments and before enqueuing anything, as a failed
 *                   launch would (gn_last_cuda_error() reports
 *                   cudaErrorLaunchFailure); setting the environment variable
 *                   GN_FAULT_INJECT=launch before the first call does the same.
 *   GN_FAULT_STALL  the next gn_fwd / gn_bwd that runs on the wave regime
 *                   withholds the arrival of one piece of unit 0, so the waits
 *                   on that unit run out: that call's outputs for unit 0 are
 *                   not valid and gn_workspace_status reports GN_ERR_TIMEOUT.
 *                   On the flat regime it withholds CTA 0's first copy: the
 *                   call's outputs are not valid and the status is the same.
 *                   The mode then returns to GN_FAULT_NONE by itself.
 * Nothing here faults the GPU: every injected failure is made on the host, or
 * is a wait that nothing satisfies and that gives up within its bound.
 * Returns a gn_status. */
#define GN_FAULT_NONE 0
#define GN_FAULT_LAUNCH 1
#define GN_FAULT_STALL 2
GN_API int gn_set_fault_injection(int mode);

/* Static, human-readable name of a status code. */
GN_API const char* gn_status_string(int status);

/* The cudaError_t behind the last GN_ERR_CUDA returned on this thread. */
GN_API int gn_last_cuda_error(void);

/* Timing hook for benchmarks.  After this call, every gn_fwd/gn_bwd made by
 * the same host thread records, on its stream, ev_begin before its first
 * kernel, ev_mid between its two kernels and ev_end after its last kernel
 * (each a cudaEvent_t created by the caller; NULL skips that record).  Pass
 * three NULLs to stop.  Returns a gn_status. */
GN_API int gn_set_timing_events(void* ev_begin, void* ev_mid, void* ev_end);

/* Kernel families ("regimes").  GN_REGIME_TWO_KERNEL runs any shape: a
 * reduction kernel (statistics, or the backward group sums) and an
 * elementwise kernel (y, or dx).  GN_REGIME_RESIDENT runs one kernel in which
 * a thread-block cluster of up to 16 CTAs owns a whole reduction unit -- one
 * (n, group) span for NCHW (at most 16 channels per group), one (sample,
 * block of whole groups of at most 128 channels where possible) for NHWC --
 * streaming it through shared memory; it is taken for 16-byte aligned fp32 /
 * fp16 / bf16 inputs whose unit holds at most 16 MiB of input (x, or x and dy).
 * GN_REGIME_PIPELINED runs one
 * persistent kernel (a cooperative launch, NCHW with HW >= 2048 and 16-byte
 * aligned data): every CTA takes one piece of every (n, group) unit, unit
 * after unit, the second pass of a unit trailing its first by a few units so
 * that it finds the input still in L2; data arrives through bulk copies into
 * shared memory.  GN_REGIME_WAVE runs one persistent kernel (a cooperative
 * launch; 16-byte aligned fp32 / fp16 / bf16 data) that cuts every reduction
 * unit -- one (n, group) span for NCHW, one (sample, block of whole groups)
 * for NHWC -- into pieces held on chip by several CTAs at once: each CTA
 * reduces its piece, publishes per-channel partial sums, waits (bounded) for
 * the unit's other pieces and writes its output from the copy it holds
 * (in tensor memory where the piece fits there twice, with the reduce and
 * the output on separate warps), so the input is read from HBM once; it is
 * taken where every unit fits on the co-resident CTAs, and chosen
 * automatically for NCHW problems of at least 32 MiB whose units hold at least
 * 64 KiB.  GN_REGIME_FLAT
 * runs one cooperative kernel for dense, 16-byte aligned channels-last fp32 /
 * fp16 / bf16 data of at most 512 16-byte vectors per row: the N*HW rows are
 * cut into equal runs, one per SM, each read by bulk copies into shared
 * memory; every CTA writes per-group (forward) or per-channel (backward)
 * partial sums for the samples its run touches, one grid-wide barrier
 * separates that from the merge, and the output is written from the chunks
 * still held (the others are read again, from L2); it is chosen
 * automatically for channels-last backwards whose x and dy hold 10-48 MiB
 * together.  Every regime gives
 * results within the same tolerances of the definition, each bit-identical
 * from run to run. */
#define GN_REGIME_AUTO (-1)
#define GN_REGIME_TWO_KERNEL 0
#define GN_REGIME_RESIDENT 1
#define GN_REGIME_PIPELINED 2
#define GN_REGIME_WAVE 3
#define GN_REGIME_FLAT 4

/* Test hook, process-wide: GN_REGIME_AUTO (default) lets each call choose
 * the faster family for its shape; GN_REGIME_TWO_KERNEL forces the two-kernel
 * path; GN_REGIME_RESIDENT, GN_REGIME_PIPELINED, GN_REGIME_WAVE and GN_REGIME_FLAT force that regime wherever
 * the problem fits it (else the two-kernel path runs).  Not thread-safe with respect to
 * calls in flight on other threads.  Returns a gn_status. */
GN_API int gn_set_regime(int regime);

/* What a call would run, for tests and reports (host-only, no launch). */
typedef struct gn_plan_desc {
  int regime;            /* GN_REGIME_TWO_KERNEL, _RESIDENT, _PIPELINED, _WAVE or _FLAT */
  int launches;          /* kernels one call enqueues, the workspace clear included */
  int vector_width;      /* elements per access: 16-byte vectors, or 1 (scalar path) */
  int threads;           /* threads per CTA */
  int64_t ctas;          /* CTAs per kernel */
  int64_t partials;      /* fp32 partial-sum records written per call */
  size_t workspace_bytes;
  int cluster_ctas;      /* CTAs per thread-block cluster of the first (or only) kernel */
  int max_clusters;      /* such clusters that fit on the device at once (0: unknown) */
  size_t smem_bytes;     /* dynamic shared memory per CTA of that kernel */
  size_t err_offset;     /* workspace byte offset of the uint32 error word (0) */
  int finalise_second;   /* two-kernel path: 1 when every CTA of the second kernel
                            derives its groups' statistics (or dx coefficients)
                            from the partial records itself, 0 when the last
                            arrival of a sample does it in the first kernel */
  int level1_items;      /* items merged per level-1 record (1: none) */
  size_t clear_bytes;    /* bytes at the start of the workspace (error word and
                            counters) that the call zero-fills before its kernels */
  int64_t piece_elems;   /* wave regime: elements (NCHW) or rows (NHWC) per piece;
                            flat regime: rows per chunk */
  int64_t pieces_per_unit; /* wave regime: pieces of one reduction unit; flat
                            regime: chunks of the longest run */
  int slots;             /* resident / pipelined / wave / flat regimes: shared-memory slots per CTA */
  int hold_buffers;      /* wave regime: tensor-memory buffers holding reduced pieces
                            (0: a piece waits for its unit's statistics in its slot) */
} gn_plan_desc;

/* Fills *out with the plan of gn_fwd/gn_bwd for this problem, assuming every
 * data pointer is 16-byte aligned when `aligned` is nonzero.  Returns a
 * gn_status. */
GN_API int gn_plan_info(int op, int64_t N, int64_t C, int64_t HW, int64_t G, int layout, int dtype,
                 int aligned, gn_plan_desc* out);

#ifdef __cplusplus
}
#endif

#endif /* GN_H_ */
