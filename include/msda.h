/*
 * msda.h -- C ABI of the GB300 (sm_103a) multi-scale deformable attention
 * sampling core.
 *
 * The operation (msda-triton README, "The operator"): for every batch b,
 * query q and head m, the bracketed term of
 *
 *     MSDA(q) = sum_m W_m [ sum_l sum_k A_mlqk * x_l(phi_l(p_q) + dp_mlqk) ]
 *
 * i.e. out[b,q,m,:] = sum_{l,k} A[b,q,m,l,k] * bilinear_l(value[b,:,m,:], loc[b,q,m,l,k]).
 * The projections W_m, the offset/weight linears and the softmax are not part
 * of it.
 *
 * Sampling convention (README, "Kernel design", last paragraph; course ch. 4,
 * "Bilinear sampling"): x_im = x * W_l - 0.5, y_im = y * H_l - 0.5 (the
 * grid_sample align_corners=False convention); x0 = floor(x_im),
 * lx = x_im - x0 and likewise for y; the four corners (y0+i, x0+j) get the
 * weights (i ? ly : 1-ly) * (j ? lx : 1-lx); a corner outside
 * [0, W_l) x [0, H_l) contributes nothing and receives no gradient (zero
 * padding).  The cell decision floor(x_im) is taken on x_im computed in
 * binary32 as the single rounding of x * W_l - 0.5; everything is accumulated
 * in fp32 and rounded once (round to nearest even) to the I/O dtype.
 *
 * Layouts (README, "Quickstart"; course ch. 4, "Setup" and "The main loop").
 * All tensors are dense, row-major, in device memory owned by the caller:
 *
 *   value                    [B, S, M, D]        S = sum_l H_l * W_l
 *   spatial_shapes           [L, 2] int64        rows (H_l, W_l)
 *   level_start_index        [L]    int64        first pyramid row of level l
 *   sampling_locations       [B, Q, M, L, K, 2]  (x, y), normalised to [0, 1]
 *   attention_weights        [B, Q, M, L, K]
 *   out                      [B, Q, M * D]
 *   grad_out                 [B, Q, M * D]
 *   grad_value               [B, S, M, D]
 *   grad_sampling_locations  [B, Q, M, L, K, 2]
 *   grad_attention_weights   [B, Q, M, L, K]
 *
 * One dtype (msda_dtype) applies to every floating-point tensor of a call.
 * Index arithmetic is 64-bit (course ch. 4, "The int64 casts are
 * load-bearing").
 *
 * Calls are asynchronous on `stream`: they validate their arguments on the
 * host, enqueue kernels and return.  They never synchronise, never allocate
 * device memory and never read device memory from the host, so they can be
 * enqueued while a stream is being captured into a CUDA graph (README,
 * "Caveats": the operator is graph capturable).  A status other than MSDA_OK
 * means nothing was enqueued, except MSDA_ERR_CUDA, which reports a failed
 * launch.  Pointers are not retained after the call returns.
 *
 * Device-resident spatial shapes cannot be checked on the host without a
 * synchronisation.  The kernels therefore check every level themselves
 * (H_l, W_l in [1, 2^24], start >= 0, start + H_l*W_l <= S); a level that
 * fails is treated as empty (its samples read nothing and receive zero
 * gradient) and sets a bit that msda_device_errors() reports.
 */
#ifndef MSDA_H
#define MSDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (binary-compatible with cudaStream_t / CUstream); NULL is the
 * legacy default stream. */
typedef struct CUstream_st* msda_stream_t;

typedef enum { MSDA_F32 = 0, MSDA_F16 = 1, MSDA_BF16 = 2 } msda_dtype;

/* Accumulator of grad_value for fp16 / bf16 (course ch. 5, "The fix:
 * accumulate in FP32, downcast at the end"; README, "Kernel design" item 3).
 * NATIVE: relaxed 16-bit vector atomic adds straight into grad_value.
 * FP32:   relaxed fp32 vector atomic adds into a caller-provided fp32
 *         workspace, then one rounding pass into grad_value.
 * AUTO:   the choice msda_resolve_accum() returns.
 * For MSDA_F32, AUTO / NATIVE / FP32 are the same path (fp32 atomics, no
 * workspace).
 * DETERMINISTIC (any dtype): grad_value bit-identical from run to run (the
 * pages' atomics make it order-dependent; course ch. 5, "Atomics make
 * gradients nondeterministic").  Each contribution A*w*g, computed in fp32,
 * is scaled by 2^F and rounded once to a 64-bit integer; the integers are
 * summed with relaxed 64-bit integer atomic adds, which are exact and
 * therefore independent of order, then scaled back and rounded once to the
 * dtype.  F = 61 - ceil(log2(Q*L*K * max|A| * max|g|)) is chosen on the
 * device per call, so no sum can overflow.  Workspace: 256 + B*S*M*D*8
 * bytes. */
typedef enum {
    MSDA_ACCUM_AUTO = 0,
    MSDA_ACCUM_NATIVE = 1,
    MSDA_ACCUM_FP32 = 2,
    MSDA_ACCUM_DETERMINISTIC = 3
} msda_accum;

typedef enum {
    MSDA_OK = 0,
    MSDA_ERR_INVALID_ARG = 1,  /* negative or inconsistent sizes, NULL pointer, unknown enum or flag */
    MSDA_ERR_UNSUPPORTED = 2,  /* L, K, L*K or D above the compiled limits below */
    MSDA_ERR_MISALIGNED = 3,   /* a pointer not aligned to its element size */
    MSDA_ERR_WORKSPACE = 4,    /* FP32 accumulation without a large enough 16-byte aligned workspace */
    MSDA_ERR_CUDA = 5          /* a CUDA runtime call or launch failed; see msda_last_error() */
} msda_status;

/* Compiled limits. */
#define MSDA_MAX_LEVELS 16
#define MSDA_MAX_POINTS 64      /* K */
#define MSDA_MAX_SAMPLES 256    /* L * K */
#define MSDA_MAX_CHANNELS 1024  /* D */

/* Flags of msda_backward. */
#define MSDA_BWD_ACCUMULATE 1u  /* add this call's gradient to grad_value instead of overwriting it */
/* The FP32 accumulator's workspace holds zeros on entry: the call does not
 * clear it, and its rounding pass writes zeros back over every part of it
 * that it found non-zero, so the workspace again holds zeros on return.
 * For a caller that allocates the workspace once, clears it once and passes
 * it to every call (one call at a time): the separate clearing pass over the
 * whole workspace is saved.  Ignored unless the resolved accumulator is FP32
 * for fp16 / bf16 I/O. */
#define MSDA_BWD_WORKSPACE_ZEROED 2u

/*
 * Forward (course ch. 4, "The forward kernel, line by line"; README,
 * "Kernel design" item 1).  Writes out[B, Q, M*D].  B == 0, Q == 0, M == 0 or
 * D == 0 enqueue nothing and return MSDA_OK (course ch. 4, "The wrapper":
 * empty inputs are handled without launching).
 *
 * Requirements: B, S, M, D, Q >= 0; 1 <= L <= MSDA_MAX_LEVELS;
 * 1 <= K <= MSDA_MAX_POINTS; L*K <= MSDA_MAX_SAMPLES; D <= MSDA_MAX_CHANNELS;
 * every non-empty tensor pointer non-NULL and aligned to its element size.
 * Rows of 16-byte multiples with 16-byte aligned value/out take the vector
 * path; anything else takes the element-wise path, with identical results.
 * The kernel may be launched as a programmatic dependent of the work ahead of
 * it on `stream`; it waits for that work before reading anything.
 */
msda_status msda_forward(msda_dtype dt, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K,
                         int64_t Q, const void* value, const int64_t* spatial_shapes,
                         const int64_t* level_start_index, const void* sampling_locations,
                         const void* attention_weights, void* out, msda_stream_t stream);

/* Workspace bytes msda_backward needs for (dt, mode) and the value size:
 * when the resolved accumulator is FP32 for fp16/bf16, the fp32 sums
 * (B*S*M*D*4, rounded up to 16) followed by the touch classes of their rows
 * (2 bits per (b, pixel, head) row: (B*S*M + 63)/64*16 bytes); less with the
 * on-chip accumulator that MSDA_TUNE=tiled selects.  256 + B*S*M*D*8 for
 * DETERMINISTIC, else 0. */
size_t msda_backward_workspace_size(msda_dtype dt, msda_accum mode, int64_t B, int64_t S, int64_t M, int64_t D,
                                    int64_t L, int64_t K, int64_t Q);

/* The accumulator AUTO resolves to for this problem (NATIVE or FP32; a
 * NATIVE, FP32 or DETERMINISTIC request is returned unchanged, except that
 * MSDA_F32 returns NATIVE for AUTO / NATIVE / FP32). */
msda_accum msda_resolve_accum(msda_dtype dt, msda_accum mode, int64_t B, int64_t S, int64_t M, int64_t D,
                              int64_t L, int64_t K, int64_t Q);

/*
 * Backward (course ch. 5, "What the backward pass must produce", "Scatter
 * needs atomics", "sem=relaxed"; README, "Kernel design" items 2 and 3).
 *
 *   grad_attention_weights[p]     = <g, sampled_p>
 *   grad_sampling_locations[p][0] = A_p * W_l * <g, d sampled_p / d x_im>
 *   grad_sampling_locations[p][1] = A_p * H_l * <g, d sampled_p / d y_im>
 *   grad_value[b, corner, m, :]  += A_p * w_corner * g       (inside corners only)
 *
 * with g = grad_out[b, q, m*D:(m+1)*D] and the location derivative that of the
 * zero-padded bilinear interpolant inside the cell chosen by floor.
 * grad_sampling_locations and grad_attention_weights are overwritten.
 * grad_value is zeroed on `stream` first, unless `flags` has
 * MSDA_BWD_ACCUMULATE, in which case the gradient is added to its contents.
 * grad_value is summed by relaxed atomic adds, so its bits may differ between
 * runs (course ch. 5, "Atomics make gradients nondeterministic"), except with
 * MSDA_ACCUM_DETERMINISTIC.  When samples are dense on the pyramid, the
 * coefficients of a unit's samples that share corner rows are added before
 * the reduction: this changes only the order of the additions.
 *
 * Like msda_forward, the kernels may be launched as programmatic dependents
 * of the work ahead of them on `stream`; each waits for that work before
 * reading or writing memory, so stream order holds for the caller.
 *
 * `workspace` (device, 16-byte aligned, >= msda_backward_workspace_size()
 * bytes) is used only by the FP32 and DETERMINISTIC accumulators and may be
 * NULL otherwise; its contents on entry are irrelevant and are clobbered,
 * except with MSDA_BWD_WORKSPACE_ZEROED (FP32 accumulator: zeros on entry and
 * on return).  The FP32 accumulator also runs with a workspace of the fp32
 * sums alone (B*S*M*D*4 bytes); with the touch classes' bytes after them, a
 * backward run one pass per level (large problems) first counts the corner
 * contributions to the rows of the levels that take few of them, writes a row
 * taking exactly one straight to grad_value (the one-term sum, rounded once)
 * and reads back from the sums only the rows taking several.
 * B == 0, Q == 0, M == 0 or D == 0: nothing is sampled and every gradient
 * is zero (grad_value keeps its contents with MSDA_BWD_ACCUMULATE).
 * Requirements as msda_forward.
 */
msda_status msda_backward(msda_dtype dt, msda_accum mode, unsigned flags, int64_t B, int64_t S, int64_t M,
                          int64_t D, int64_t L, int64_t K, int64_t Q, const void* value,
                          const int64_t* spatial_shapes, const int64_t* level_start_index,
                          const void* sampling_locations, const void* attention_weights, const void* grad_out,
                          void* grad_value, void* grad_sampling_locations, void* grad_attention_weights,
                          void* workspace, size_t workspace_bytes, msda_stream_t stream);

/*
 * Fused operator (msda-triton README, "The operator": the weights A are
 * softmax-normalised over the L*K (level, point) pairs of a query and head,
 * and the sampling location is the reference point mapped to level l plus a
 * learned offset).  The steps on either side of the core are taken inside the
 * kernels, so sampling_locations and attention_weights never exist in memory:
 *
 *   A[b,q,m,l,k]   = softmax over the L*K entries of attention_logits[b,q,m,:]   (fp32)
 *   loc[b,q,m,l,k] = reference_points[b,q,l] + sampling_offsets[b,q,m,l,k] / (W_l, H_l)
 *                    (x by W, y by H; offsets are in pixels of level l; fp32, one
 *                    rounding per operation)
 *   out            = the core of msda_forward on (loc, A)
 *
 * Layouts: reference_points [B, Q, L, 2] (x, y); sampling_offsets
 * [B, Q, M, L, K, 2]; attention_logits [B, Q, M, L*K]; out [B, Q, M*D].
 * Needs rows of whole 16-byte vectors (D*esize in {64, 128, 192, 256} bytes:
 * D = 32/64/96/128 for bf16/fp16, 16/32/48/64 for fp32) and 16-byte aligned value /
 * out / grad pointers; otherwise MSDA_ERR_UNSUPPORTED.  Other requirements
 * and errors as msda_forward.
 */
msda_status msda_forward_fused(msda_dtype dt, int64_t B, int64_t S, int64_t M, int64_t D, int64_t L, int64_t K,
                               int64_t Q, const void* value, const int64_t* spatial_shapes,
                               const int64_t* level_start_index, const void* reference_points,
                               const void* sampling_offsets, const void* attention_logits, void* out,
                               msda_stream_t stream);

/*
 * Backward of the fused operator:
 *
 *   grad_sampling_offsets[p] = grad_loc[p] / (W_l, H_l)  =  A_p * <g, d sampled_p / d (x_im, y_im)>
 *   grad_reference_points[b,q,l] = sum over (m, k) of grad_loc[b,q,m,l,k]
 *   grad_attention_logits[b,q,m,s] = A_s * (gA_s - sum_j A_j gA_j),  gA_s = <g, sampled_s>
 *   grad_value as msda_backward
 *
 * All outputs are overwritten (grad_value accumulates with
 * MSDA_BWD_ACCUMULATE).  Accumulators, workspace and requirements as
 * msda_backward and msda_forward_fused.
 */
msda_status msda_backward_fused(msda_dtype dt, msda_accum mode, unsigned flags, int64_t B, int64_t S, int64_t M,
                                int64_t D, int64_t L, int64_t K, int64_t Q, const void* value,
                                const int64_t* spatial_shapes, const int64_t* level_start_index,
                                const void* reference_points, const void* sampling_offsets,
                                const void* attention_logits, const void* grad_out, void* grad_value,
                                void* grad_reference_points, void* grad_sampling_offsets,
                                void* grad_attention_logits, void* workspace, size_t workspace_bytes,
                                msda_stream_t stream);

/*
 * Backward with the FP32 accumulator whose scratch lives in a fixed device
 * array inside the library instead of a caller-provided workspace; it
 * allocates nothing.  The pages have no counterpart: this is for callers that
 * can pass input and output buffers but cannot allocate device memory when
 * they call (an engine plugin handed only its tensors, a loop that forbids
 * allocation after start-up).  Results equal msda_backward(dt,
 * MSDA_ACCUM_FP32, flags, ...) up to the summation order of grad_value.
 *
 * Limit: the FP32 accumulator's sums, B*S*M*D*4 bytes (what
 * msda_backward_workspace_size(dt, MSDA_ACCUM_FP32, ...) reports without the
 * touch classes, which are used when they fit as well), must fit in
 * MSDA_STATIC_WORKSPACE_BYTES, else MSDA_ERR_WORKSPACE before anything is
 * enqueued.  The limit applies only to
 * calls that need scratch: fp32 I/O, and calls with nothing to sample
 * (B*Q*M*D == 0), need none and have no limit.  Arguments are checked as
 * msda_backward checks them, and give its errors.
 *
 * The array occupies MSDA_STATIC_WORKSPACE_BYTES on every device where the
 * translation unit that holds it is loaded, until the process exits: with
 * lazy module loading (the CUDA default) a device on which this entry point
 * has looked the array up, with CUDA_MODULE_LOADING=EAGER every device the
 * process creates a context on, whether or not this entry point is called.  Its device
 * address is looked up on every call made outside stream capture; a call
 * made while `stream` is being captured uses the address found by the last
 * uncaptured call on that device, so make one such call first.  All calls
 * share the one array: calls that can overlap on the GPU race and must be
 * serialised by the caller.  MSDA_BWD_WORKSPACE_ZEROED is rejected
 * (MSDA_ERR_INVALID_ARG): every call clears the array itself.  Other
 * arguments and errors as msda_backward.
 */
#define MSDA_STATIC_WORKSPACE_BYTES (64u << 20)
msda_status msda_backward_static_workspace(msda_dtype dt, unsigned flags, int64_t B, int64_t S, int64_t M, int64_t D,
                                           int64_t L, int64_t K, int64_t Q, const void* value,
                                           const int64_t* spatial_shapes, const int64_t* level_start_index,
                                           const void* sampling_locations, const void* attention_weights,
                                           const void* grad_out, void* grad_value, void* grad_sampling_locations,
                                           void* grad_attention_weights, msda_stream_t stream);

/* Message for the last non-OK status returned on the calling thread ("" if none). */
const char* msda_last_error(void);

/* Short name of a status code. */
const char* msda_status_string(msda_status s);

/* Device-side error bits raised by kernels on the current device since the
 * last clear (bit 0: a level failed its shape check).  Synchronises the
 * device.  clear != 0 resets the bits. */
msda_status msda_device_errors(uint32_t* bits, int clear);

/* Library version: major * 10000 + minor * 100 + patch. */
int msda_version(void);

/*
 * Measurement utility (not part of the operator): the L2's throughput for
 * the backward's kind of reduction traffic on the current device.  The
 * backward adds every in-level corner row into grad_value (or its fp32
 * workspace) with relaxed 16-byte vector reductions, the row's row_bytes
 * taken by row_bytes / 16 adjacent lanes, at rows scattered over the tensor
 * (ch. 5, "Scatter needs atomics", "sem=relaxed").  This runs that pattern
 * alone: rows of `row_bytes` (16, 32, 64, 128, 256 or 512) at random places of
 * `scratch`, each taken by row_bytes / 16 lanes with one 16-byte reduction of
 * `kind` (0 bf16x2, 1 f16x2, 2 f32) each, with `blocks_per_sm` blocks of 256
 * threads per SM, and reports 32-byte sectors per second in
 * *sectors_per_second (best of `repeats` launches of 256 reductions per
 * thread, after one warm-up).
 *
 * scratch: device buffer of scratch_bytes (>= 1 MiB, 16-byte aligned); its
 * contents are overwritten.  Keep it inside the L2 (e.g. 64 MiB) to measure
 * the L2's reduction rate rather than DRAM's.  Unlike the operator calls
 * this one synchronises `stream` (it times with CUDA events) and is meant
 * for roofline reporting, not for the hot path.  Errors: NULL or small or
 * misaligned scratch, kind outside 0..2, row_bytes not listed above,
 * blocks_per_sm outside 1..16 or repeats outside 1..100 ->
 * MSDA_ERR_INVALID_ARG; a CUDA failure -> MSDA_ERR_CUDA.
 */
msda_status msda_reduction_ceiling(int kind, int row_bytes, int blocks_per_sm, int repeats, void* scratch,
                                   size_t scratch_bytes, double* sectors_per_second, msda_stream_t stream);

/*
 * Kernel trace.  While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on its own stream (no
 * synchronisation).  msda_trace_read() waits for the recorded events and
 * returns one record per launch, oldest first, then forgets them.  Launches
 * beyond `capacity` are counted in `dropped` but not recorded.  Enabling
 * creates 2*capacity events on the current device; capacity 0 disables and
 * destroys them.  Not thread-safe against concurrent msda_* calls.
 */
typedef struct {
    int kernel;        /* MSDA_KERNEL_* */
    float ms;          /* elapsed time between the two events */
    int64_t work;      /* (b,q,m) units for fwd/bwd, elements for zero/convert */
} msda_trace_record;

enum { MSDA_KERNEL_FORWARD = 0, MSDA_KERNEL_BACKWARD = 1, MSDA_KERNEL_ZERO = 2, MSDA_KERNEL_CONVERT = 3,
       MSDA_KERNEL_TILE_COUNT = 4, MSDA_KERNEL_TILE_SCAN = 5, MSDA_KERNEL_TILE_PLACE = 6,
       MSDA_KERNEL_TILE_ACCUM = 7, MSDA_KERNEL_TOUCH = 8, MSDA_KERNEL_COUNT = 9 };

msda_status msda_trace_enable(int capacity);
/* Pause (paused != 0) or resume recording without destroying the events:
 * a paused trace adds no work to the streams. */
void msda_trace_pause(int paused);
int msda_trace_read(msda_trace_record* records, int max_records, int* dropped);
const char* msda_kernel_name(int kernel);

#ifdef __cplusplus
}
#endif
#endif /* MSDA_H */
