/*
 * lse.h -- C ABI of liblse, a GB300 (sm_103a) row-wise log-sum-exp.
 *
 *     out[b] = log( sum_{n<N} exp(x[b, n]) ),   b < B
 *
 * Source: "Speeding up Log-Sum-Exp: Kernel Fusion at the Memory Wall, Integer
 * Arithmetic at the Compute Wall".  The operation is the LSE primitive of the
 * TL;DR and Sec. 2; it is a drop-in replacement for torch.logsumexp over the
 * last dimension (Abstract).  Sec. 3.1 defines the method: one pass over HBM,
 * each input element read once, one scalar written per row, partial results
 * combined with the associative, commutative pairwise LSE operation.
 *
 * Conventions shared by every entry point
 *   x           device pointer (host pointer for lse_forward_host) to B rows;
 *               row b starts at element b * row_stride.  Elements are f32,
 *               bf16 or f16 (lse_dtype).  Read-only; not retained.
 *               x must be aligned to its element size (4 bytes for f32,
 *               2 for bf16 and f16).
 *   row_stride  distance between row starts, in ELEMENTS, >= N; any value.
 *               Rows are read as 16-byte vectors; a row that does not start
 *               or end on a 16-byte boundary reads the aligned 16-byte
 *               vectors that cover it and ignores the bytes outside the row
 *               (such a vector never leaves the row's memory page).
 *   out         device pointer (host pointer for lse_forward_host) to B
 *               floats, 4-byte aligned.  Written once per row; not retained.
 *   stream      CUDA stream for all work (0 = legacy default stream).  The
 *               device entry points are asynchronous and stream-ordered.
 *   Special values (torch.logsumexp semantics): a row holding a NaN gives NaN;
 *   otherwise a row holding +inf gives +inf; a row of only -inf, or N == 0,
 *   gives -inf; -inf entries next to finite ones contribute nothing.
 *   B == 0 is a no-op returning LSE_OK.  The library never aborts, never
 *   falls back to the CPU, and never synchronises a device call except
 *   lse_forward_host.
 *
 * Errors: every call returns an lse_status.  LSE_ERR_INVALID_ARG for B < 0,
 * N < 0, row_stride < N, a NULL x (N > 0) or out (B > 0), a misaligned x or out, or
 * sizes whose byte extent overflows int64; LSE_ERR_UNSUPPORTED_DTYPE for an
 * unknown dtype; LSE_ERR_ALLOC when stream-ordered scratch cannot be
 * allocated; LSE_ERR_CUDA when a CUDA call fails (lse_last_cuda_error gives
 * the cudaError_t).  On any error nothing is guaranteed about out.
 */
#ifndef LSE_H
#define LSE_H

#include <stdint.h>

/* Exported from liblse.so (built with hidden visibility by default). */
#if defined(__GNUC__)
#define LSE_API __attribute__((visibility("default")))
#else
#define LSE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA handle types, identical to cudaStream_t / cudaEvent_t. */
typedef struct CUstream_st *lse_stream_t;
typedef struct CUevent_st *lse_event_t;

typedef enum {
    LSE_F32 = 0,
    LSE_BF16 = 1,
    LSE_F16 = 2
} lse_dtype;

typedef enum {
    LSE_OK = 0,
    LSE_ERR_INVALID_ARG = 1,
    LSE_ERR_UNSUPPORTED_DTYPE = 2,
    LSE_ERR_ALLOC = 3,
    LSE_ERR_CUDA = 4
} lse_status;

/* Kernel mappings.  AUTO lets the library choose from (dtype, B, N, layout). */
typedef enum {
    LSE_PATH_AUTO = 0,
    LSE_PATH_EMPTY = 1,   /* N == 0: one fill kernel writes -inf           */
    LSE_PATH_SUBWARP = 2, /* short rows: a group of 1..32 lanes per row     */
    LSE_PATH_CTA = 3,     /* one CTA (1..8 warps) per row, online (m, s)    */
    LSE_PATH_SPLIT = 4,   /* `splits` CTAs per row write (m, s) partials;
                             a second small kernel merges them in order   */
    LSE_PATH_COLUMNS_WARP = 5, /* lse_forward_strided: one warp per column tile */
    LSE_PATH_COLUMNS_CTA = 6,  /* lse_forward_strided: 2, 4 or 8 warps share the
                                  rows of one column tile                       */
    LSE_PATH_ROWTILE = 7,      /* back-to-back rows (<= 4 KB) from a 16-byte
                                  aligned base, streamed into shared memory by
                                  bulk copies (TMA).  Rows of 16..128 bytes in
                                  multiples of 16 (slots_per_lane = vectors per
                                  row): each warp streams 4 KB chunks of 32
                                  rows, a lane per row; row value, token
                                  log-probability and 16-bit exponentials.
                                  Rows of other widths (slots_per_lane = 0):
                                  32 KB chunks per CTA, a thread per row up to
                                  128 bytes plus one element (vector_bytes =
                                  1), else a group
                                  of 4..32 lanes (lanes_per_row); row value and
                                  token log-probability with f32 exponentials */
    LSE_PATH_COLUMNS_SHORT = 8 /* lse_forward_strided, R <= 8 rows of 16-byte
                                  column vectors: one thread per vector loads
                                  all R rows at once and folds them (max,
                                  then exp-sum); no split                     */
} lse_path;

/*
 * A launch plan.  lse_plan_query fills one with the library's choice;
 * lse_forward_plan runs a caller-edited one (fields left 0 are chosen by the
 * library; a forced value outside its valid range gives LSE_ERR_INVALID_ARG).
 */
typedef struct {
    int32_t path;           /* lse_path                                              */
    int32_t vector_bytes;   /* 16: 128-bit loads (a row that does not start on a
                               16-byte boundary reads the vectors covering it and
                               masks the bytes outside it); 1: element loads only;
                               0 in a request: let the library choose              */
    int32_t lanes_per_row;  /* SUBWARP: lanes per row, a power of two 1..32;
                               column paths: warps sharing one column tile, 1/2/4/8 */
    int32_t slots_per_lane; /* SUBWARP: vectors (or elements) per lane, 1/2/3/4/6/8
                               (output)                                            */
    int32_t threads;        /* CTA / SPLIT: threads per CTA, 32/64/128/256/512      */
    int32_t launches;       /* kernels launched per call (output)                    */
    int64_t splits;         /* SPLIT: CTAs per row (>= 2); 1 otherwise               */
    int64_t segment_slots;  /* CTA / SPLIT: vectors (or elements) per CTA (output)   */
    int64_t grid;           /* CTAs launched by the main kernel (output)             */
    int64_t scratch_bytes;  /* device scratch the plan allocates (output)           */
} lse_plan;

/*
 * lse_forward -- out[b] = log sum_n exp(x[b, n]) on the GPU, one pass over x.
 * Device pointers; asynchronous on `stream`.  The split-row mapping takes
 * B * splits * 8 bytes of scratch, allocated and freed stream-ordered on
 * `stream` (so concurrent calls on different streams never share it).
 * Every kernel is launched with programmatic dependent launch: it may become
 * resident while the previous kernel in `stream` finishes, and waits on the
 * device for that kernel to complete before touching memory.
 */
LSE_API lse_status lse_forward(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                       int64_t row_stride, float *out, lse_stream_t stream);

/*
 * lse_plan_query -- the plan lse_forward would use for these arguments on the
 * current device (x is only inspected for its alignment; it may be NULL, which
 * counts as 16-byte aligned).  Launches nothing.
 */
LSE_API lse_status lse_plan_query(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                          int64_t row_stride, lse_plan *plan);

/*
 * lse_forward_plan -- lse_forward with a caller-chosen plan (NULL = automatic).
 * If ev_begin / ev_end are non-NULL they are recorded on `stream` immediately
 * before and after the main (row-reading) kernel, so the caller can time that
 * kernel alone.  On return *plan (if non-NULL) holds the plan that ran.
 */
LSE_API lse_status lse_forward_plan(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                            int64_t row_stride, float *out, lse_stream_t stream,
                            lse_plan *plan, lse_event_t ev_begin, lse_event_t ev_end);

/*
 * lse_forward16 -- lse_forward with reduced-bit exponentials, the paper's
 * 16-bit compute variant ("Speeding up Log-Sum-Exp ...", Sec. 4.3 and Fig. 5:
 * FuseLSE16, faster on V100 at a mean absolute error below 3e-3).  The same
 * single pass, mappings and plans (plan as for lse_forward_plan, NULL =
 * automatic), except for the terms exp(x - max): each base-2 argument
 * a = (x - max) log2 e is formed in f32 plus a constant d = 0.00407 (below),
 * rounded to bf16, and two of them are exponentiated by one packed bf16 SFU
 * instruction; sums, merges and the final log stay in f32, and special values
 * follow lse_forward exactly.  The SFU rounds its bf16 result toward zero,
 * half a bf16 ulp low on average (2^-8 / (2 ln 2) of the value); d scales every
 * term up by that much first, so terms are unbiased on average, while the
 * maximum's own term (2^d = 1.0028) still truncates to exactly 1.
 * Accuracy: the argument moves by d plus at most (|a| + d) 2^-8 in rounding, and
 * truncation takes off less than a factor (1 - 2^-7), so each term is within a
 * relative r_n = 2^(d + (|a_n| + d) 2^-8) - 1 + 2^-7 of exp(x_n - max), and
 *     |result - lse| <= -log(1 - e),  e = sum_n p_n r_n
 * (p_n the row's softmax) plus the f32 rounding of lse_forward.  To first
 * order e <= 2^-7 + 2^-8 ln N + 0.003, since sum_n p_n |a_n| ln 2 <= ln N; far
 * less in practice, as rounding errors of different terms do not line up.
 * It halves the SFU operations per element; the f32 path is already bound by
 * HBM bandwidth on this GPU at full clocks, so the gain is SFU headroom (at
 * lower clocks, with 16-bit input).  The pages do not give FuseLSE16's kernel:
 * this is the plain reading of a 16-bit exponent evaluation with f32 sums.
 */
LSE_API lse_status lse_forward16(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                                 int64_t row_stride, float *out, lse_stream_t stream,
                                 lse_plan *plan);

/*
 * lse_forward_host -- the same result from HOST buffers, synchronising
 * `stream` before returning.  A page-locked x (cudaHostAlloc'ed or registered)
 * is read in place by the kernel over the host link (zero copy; the bytes
 * still cross the link once), and a page-locked out is written in place.
 * Pageable buffers are copied through stream-ordered device buffers from the
 * library pool (cudaMemcpyAsync), freed before return.
 */
LSE_API lse_status lse_forward_host(const void *x_host, lse_dtype dtype, int64_t B, int64_t N,
                            int64_t row_stride, float *out_host, lse_stream_t stream);

/*
 * lse_token_logprob -- fused token log-probability, the consumer the paper
 * benchmarks in RLHF (Sec. 5.1, Fig. 6: per-token log-probabilities over
 * vocabularies of 32K-256K):
 *
 *     logprob[b] = x[b, target[b]] - log sum_n exp(x[b, n])
 *
 * in the same single pass over x as lse_forward (x[b, target[b]] is taken
 * from registers or from the row staged in shared memory on short rows, and
 * gathered once per row on long ones).
 *   target   device pointer to B int64 column indices, 8-byte aligned; a
 *            target outside [0, N) gives logprob NaN (it is never read).
 *   logprob  device pointer to B floats, 4-byte aligned.
 *   lse_out  device pointer to B floats for the row values, or NULL.
 * Special values follow IEEE arithmetic on x[b, t] - lse[b] with lse[b] as in
 * lse_forward (e.g. a row holding NaN gives NaN; an all -inf row gives NaN).
 * Split rows take B * (splits * 8 + 4) bytes of stream-ordered scratch.
 */
LSE_API lse_status lse_token_logprob(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                                     int64_t row_stride, const int64_t *target, float *logprob,
                                     float *lse_out, lse_stream_t stream);

/* lse_token_logprob with a caller-chosen plan (NULL = automatic); on return
 * *plan (if non-NULL) holds the plan that ran. */
LSE_API lse_status lse_token_logprob_plan(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                                          int64_t row_stride, const int64_t *target,
                                          float *logprob, float *lse_out, lse_stream_t stream,
                                          lse_plan *plan);

/*
 * lse_backward -- gradient of the row value with respect to x:
 *
 *     dx[b, n] = grad[b] * exp(x[b, n] - lse[b])
 *
 * (d lse / d x is the row's softmax; the paper lists backward support among
 * its kernel variants, Table 3).  One pass: x read once, dx written once.
 *   lse      device pointer to B floats: the saved forward values.
 *   grad     device pointer to B floats: the upstream gradient of each row value.
 *   dx       device pointer, same element type as x, row b at b * dx_row_stride
 *            (elements, >= N); computed in f32, rounded to nearest-even on store.
 *            dx may be x itself (same row_stride); other overlaps are undefined.
 *            dx must be aligned to its element size (LSE_ERR_INVALID_ARG).
 * Loads and stores are 16-byte vectors when each x row and its dx row sit at
 * the same offset from a 16-byte boundary (rows off a boundary move their head
 * and tail element by element, or, back to back, as one flat array of
 * vectors); element by element otherwise.
 * Special values follow IEEE arithmetic on that formula (an all -inf row, whose
 * lse is -inf, gives NaN).  Asynchronous on `stream`; allocates nothing.
 */
LSE_API lse_status lse_backward(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                                int64_t row_stride, const float *lse, const float *grad,
                                void *dx, int64_t dx_row_stride, lse_stream_t stream);

/*
 * lse_forward_strided -- the same value over a non-last dimension:
 *
 *     out[a * C + c] = log sum_{r < R} exp(x[a * stride_a + r * stride_r + c])
 *
 * for a < A, c < C (element strides; c is the contiguous index).  This is the
 * reduction of a probabilistic-circuit sum layer over each node's children
 * (Sec. 5.2), or a column LSE of a matrix (A = 1).  One pass over x.
 *   out      device pointer to A * C floats (row-major [A, C]); must not
 *            overlap x.
 *   plan     NULL (automatic) or an lse_plan: path 0, LSE_PATH_COLUMNS_WARP
 *            (one warp per 32-lane column tile walks all its rows),
 *            LSE_PATH_COLUMNS_CTA (lanes_per_row = 2, 4 or 8 warps interleave
 *            the rows of one tile, merged in shared memory; 0 = 8) or
 *            LSE_PATH_COLUMNS_SHORT (R <= 8 and a 16-byte vector layout, no
 *            split; the automatic choice there);
 *            splits 0 (automatic) or k >= 1 (<= R, <= 65535) row splits
 *            across CTAs -- with k > 1 the call takes A * C * k * 8 bytes of
 *            stream-ordered scratch and a merge kernel; vector_bytes as for
 *            lse_forward_plan.  On return *plan holds the plan that ran.
 * R == 0 gives -inf; A == 0 or C == 0 is a no-op.  Special values as in
 * lse_forward, per (a, c).  16-byte aligned layouts with C a multiple of the
 * elements per 16 bytes take vector loads; others element loads.
 */
LSE_API lse_status lse_forward_strided(const void *x, lse_dtype dtype, int64_t A, int64_t R,
                                       int64_t C, int64_t stride_a, int64_t stride_r, float *out,
                                       lse_stream_t stream, lse_plan *plan);

/*
 * lse_backward_strided -- gradient of lse_forward_strided's value:
 *
 *     dx[a, r, c] = grad[a, c] * exp(x[a * stride_a + r * stride_r + c] - lse[a, c])
 *
 * (d out[a, c] / d x[a, r, c] is the softmax over r; the backward of the
 * value over a non-last dimension, as lse_backward is for rows).  One pass:
 * x read once, dx written once; lse and grad are read once per column tile.
 *   x        as for lse_forward_strided (element strides stride_a, stride_r;
 *            c contiguous).
 *   lse      device pointer to A * C floats ([A, C]): the saved forward values.
 *   grad     device pointer to A * C floats ([A, C]): upstream gradients.
 *   dx       device pointer, x's element type, element (a, r, c) at
 *            a * dx_stride_a + r * dx_stride_r + c; computed in f32 and
 *            rounded to nearest-even on store.  dx may be x itself (same
 *            strides); other overlaps are undefined.
 * A, R or C == 0 is a no-op.  Special values follow IEEE arithmetic on the
 * formula.  16-byte aligned layouts (x, dx, every stride) with C a multiple of
 * the elements per 16 bytes take vector loads; others element loads.
 * Asynchronous on `stream`; allocates nothing.
 */
LSE_API lse_status lse_backward_strided(const void *x, lse_dtype dtype, int64_t A, int64_t R,
                                        int64_t C, int64_t stride_a, int64_t stride_r,
                                        const float *lse, const float *grad, void *dx,
                                        int64_t dx_stride_a, int64_t dx_stride_r,
                                        lse_stream_t stream);

/*
 * lse_trim_memory -- return the current device's cached stream-ordered memory
 * to the system.  Split-row scratch and lse_forward_host's staging buffers come
 * from a library-owned memory pool that keeps freed blocks mapped for reuse by
 * later calls (while a stream is being captured into a CUDA graph, the
 * device's default pool is used instead).  Call after synchronising every
 * stream that used the library on this device.
 */
LSE_API lse_status lse_trim_memory(void);

/*
 * lse_wait_timeouts -- number of bounded device-side waits that gave up since
 * the library was loaded, on the current device (synchronous read).  Kernels
 * that wait for their own asynchronous copies (LSE_PATH_ROWTILE) stop and
 * count here instead of waiting forever; a non-zero count means results of
 * such a launch are incomplete.  Zero in correct operation.  A launch whose
 * wait gave up has still returned LSE_OK from its entry point (the wait runs
 * on the device after the call returned): this counter is the only report.
 */
LSE_API lse_status lse_wait_timeouts(unsigned long long *count);

/* Poll limit of the LSE_PATH_ROWTILE stage waits unless changed below. */
#define LSE_DEFAULT_WAIT_POLLS (1u << 26)

/*
 * lse_set_wait_limit -- testing aid: the number of mbarrier polls after which
 * a LSE_PATH_ROWTILE stage wait gives up, for every launch that follows in
 * this process (all devices).  LSE_DEFAULT_WAIT_POLLS restores the default;
 * 0 makes every stage wait give up at once.  A wait that gives up stops its
 * warp (or CTA): the rows it had not finished are left unwritten, the warp
 * first waits, with the default limit, for the bulk copies it already issued
 * so that none is in flight when it exits, lse_wait_timeouts counts one, and
 * the entry point that launched it has returned LSE_OK.  Not for production
 * use: it exists so that tests can run the give-up path without a hang.
 */
LSE_API lse_status lse_set_wait_limit(uint32_t polls);

/* Short English description of a status code (static storage). */
LSE_API const char *lse_status_string(lse_status status);

/*
 * The cudaError_t behind the calling thread's most recent LSE_ERR_CUDA or
 * LSE_ERR_ALLOC (0 if none).  Returns LSE_OK, or LSE_ERR_INVALID_ARG if
 * cuda_err is NULL.
 */
LSE_API lse_status lse_last_cuda_error(int *cuda_err);

/* Size of the fixed device scratch array of lse_forward_split_static:
 * 1 MiB, i.e. 131072 (m, s) partials of 8 bytes. */
#define LSE_STATIC_SCRATCH_BYTES (1 << 20)

/*
 * lse_forward_split_static -- the same result as lse_forward, through the
 * split-row mapping, without allocating any device memory.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * while they run (a memory budget reserved up front, real-time loops where an
 * allocator call and the synchronisation or page mapping it may trigger are not
 * allowed, allocators owned by another runtime).  It calls no cudaMalloc,
 * cudaFree, stream-ordered allocator or allocating library routine.
 *
 * The per-row partials live in a file-scope __device__ array of
 * LSE_STATIC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits.  The first call on a device (with that device current) looks
 * up the array's device address with cudaGetSymbolAddress and caches it; make
 * that first call before any stream capture.  All calls share the array, so
 * calls whose kernels overlap on the GPU (different streams, or unordered host
 * threads) race; calls on one stream are ordered and safe.  Nothing needs
 * clearing between calls: each call writes every partial it reads.
 *
 * Same arguments and conventions as lse_forward.  Extra limits, reported as
 * LSE_ERR_INVALID_ARG: B <= LSE_STATIC_SCRATCH_BYTES / 16 (65536 rows, two
 * partials per row at least), and rows long enough to split (N >= 2 vectors of
 * 16 bytes when rows are 16-byte aligned, N >= 2 otherwise).  The number of
 * splits per row is chosen to fill the GPU and capped so B * splits partials
 * fit the array.
 */
LSE_API lse_status lse_forward_split_static(const void *x, lse_dtype dtype, int64_t B, int64_t N,
                                            int64_t row_stride, float *out, lse_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LSE_H */
