/*
 * libsoftmax: numerically stable row-wise softmax for NVIDIA GB300 (sm_103a).
 *
 * The operation, for each row r and column j < n_cols:
 *
 *     y[r][j] = exp(x[r][j] - m_r) / l_r,
 *     m_r = max_k x[r][k],   l_r = sum_k exp(x[r][k] - m_r)
 *
 * as stated in "Lecture 6: GPU Kernel programming and Triton" (xwysyy.cn,
 * cs336 lecture 6 notes), section "Level 1: Softmax", display formula, and
 * computed as in the fused softmax of "Triton: write CUDA-grade GPU operators
 * in Python" (f.mffb.com.cn), example 2 "Fused Softmax": one read of the row,
 * max, subtract, exp, sum, divide, one write.  Positions past n_cols are
 * neither read nor written.  Rows longer than one multiprocessor can hold are
 * combined with the running (m, l) rescale of "Triton GPU programming deep
 * dive" (ybb.press), section 3.3.  Arithmetic is fp32 for both dtypes
 * (page 1's tuning checklist: fp32 accumulators for fp16/bf16 data).
 *
 * Conventions shared by every entry point:
 *  - Layout: row-major rows with unit column stride.  Row r of the input
 *    starts at element r * in_row_stride of `in`, row r of the output at
 *    element r * out_row_stride of `out`.  Strides count ELEMENTS, not bytes
 *    (example 2's wrapper passes x.stride(0) and out.stride(0)).
 *  - dtype: SOFTMAX_F32 (binary32 in and out), SOFTMAX_BF16 (bfloat16 in
 *    and out) or SOFTMAX_F16 (IEEE binary16 in and out); 16-bit outputs
 *    are rounded to nearest even.  The arithmetic is fp32 for every dtype
 *    ("Triton: write CUDA-grade GPU operators in Python", tuning checklist:
 *    fp32 accumulators for float16/bfloat16 data).
 *  - Ownership: every buffer belongs to the caller.  The library never
 *    allocates device or host memory and keeps no workspace.
 *  - Asynchrony: device work is queued on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) and the call returns without synchronising.
 *    The return value reports argument and launch errors only.
 *  - Errors: a status code (softmax_status_t), never an exception, never
 *    an abort.  Nothing is launched when the status is not SOFTMAX_OK.
 *  - Degenerate rows follow IEEE arithmetic of the formula: a row containing
 *    NaN or +inf, or made only of -inf, becomes all NaN.  -inf entries in an
 *    otherwise finite row give exact +0.
 *  - In place (in == out with equal strides) is allowed.  Any other overlap
 *    between the input and output elements is rejected; with unequal
 *    strides, intersecting address ranges are rejected.
 *  - Thread safety: calls may be made concurrently from several host threads.
 */
#ifndef LIBSOFTMAX_SOFTMAX_H
#define LIBSOFTMAX_SOFTMAX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SOFTMAX_ABI_VERSION 2

typedef enum {
    SOFTMAX_F32 = 0,
    SOFTMAX_BF16 = 1,
    SOFTMAX_F16 = 2
} softmax_dtype_t;

typedef enum {
    SOFTMAX_OK = 0,
    SOFTMAX_ERR_INVALID_ARG = 1,     /* bad pointer, size, stride, dtype or overlap */
    SOFTMAX_ERR_UNSUPPORTED = 2,     /* no device, wrong architecture, or a forced
                                        path that cannot take this shape */
    SOFTMAX_ERR_CUDA = 3,            /* a CUDA runtime call or launch failed */
    SOFTMAX_ERR_DEVICE_TIMEOUT = 4   /* a kernel gave up a bounded wait (see
                                        softmax_device_status) */
} softmax_status_t;

/* Execution paths chosen by the row-to-CTA scheduler. */
typedef enum {
    SOFTMAX_PATH_AUTO = -1,
    SOFTMAX_PATH_WARP = 0,      /* a warp owns whole rows, held in registers */
    SOFTMAX_PATH_CTA = 1,       /* a CTA owns a row, staged in shared memory */
    SOFTMAX_PATH_CLUSTER = 2,   /* a thread-block cluster owns a row; slices in
                                   shared memory, (m, l) partials exchanged
                                   through distributed shared memory */
    SOFTMAX_PATH_TWOPASS = 3    /* a cluster streams the row twice from HBM:
                                   online (m, l) pass, then normalise pass */
} softmax_path_t;

/*
 * softmax_rows: y = softmax(x) along each row (the operation above).
 *
 *   in, out          device pointers (or any pointer the device can access),
 *                    aligned to the element size.  May be NULL only when
 *                    n_rows == 0 or n_cols == 0.
 *   n_rows, n_cols   matrix shape; 0 in either is a no-op returning OK.
 *   in_row_stride    elements between consecutive input rows;
 *   out_row_stride   elements between consecutive output rows.  Each must be
 *                    >= n_cols when n_rows > 1.
 *   dtype            softmax_dtype_t.
 *   stream           cudaStream_t to queue the work on (NULL: legacy default).
 *
 * Returns SOFTMAX_OK once the work is queued; SOFTMAX_ERR_INVALID_ARG for a
 * negative size, a short stride, an unknown dtype, a NULL or misaligned
 * pointer, or overlapping (not identical) input and output;
 * SOFTMAX_ERR_UNSUPPORTED when the current device is not sm_103;
 * SOFTMAX_ERR_CUDA when the launch fails.  Pointers not aligned to 16 bytes,
 * or strides that break 16-byte row alignment, take slower scalar access,
 * not an error.
 */
int softmax_rows(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                 int64_t in_row_stride, int64_t out_row_stride, int dtype,
                 void* stream);

/*
 * softmax_rows_path: softmax_rows with the execution path forced (tests and
 * benchmarks).  path = SOFTMAX_PATH_AUTO behaves exactly like softmax_rows.
 * A forced path that cannot take the shape (e.g. WARP with n_cols > 1024)
 * returns SOFTMAX_ERR_UNSUPPORTED and launches nothing.
 */
int softmax_rows_path(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                      int64_t in_row_stride, int64_t out_row_stride, int dtype,
                      void* stream, int path);

/*
 * Options of softmax_rows_ex: a scaled, causally masked softmax, the form
 * attention scores take.  "Triton GPU programming deep dive", section 3.1,
 * divides the scores Q K^T by sqrt(d) before the softmax; its section 3.3
 * sets a score to -inf unless the key index is at most the query index.
 * Here the mask is computed from indices instead of -inf written into the
 * input.
 *
 *   scale          the softmax is taken over z = scale * x; 0 < scale <=
 *                  2^127 (1.0f: none).  The result is that of the exact
 *                  product scale * x (the kernels fold the scale into the
 *                  exponent).
 *   causal         0: no mask.  1: column c of row r takes part iff
 *                  c <= (r mod causal_period) + causal_offset; every other
 *                  column counts as -inf: its input is never read and its
 *                  output is exactly +0 (NaN when the row's result is NaN).
 *                  A row with no column taking part is all NaN (the formula
 *                  over only -inf).
 *   causal_period  rows per masked block (e.g. the query length when rows
 *                  are (batch, head, query) triples); <= 0 means n_rows (as
 *                  does any period of n_rows or more).
 *   causal_offset  shift of the diagonal (e.g. key length minus query
 *                  length for a bottom-right aligned mask); |offset| < 2^62.
 */
typedef struct {
    float scale;
    int32_t causal;
    int64_t causal_period;
    int64_t causal_offset;
} softmax_options_t;

/*
 * softmax_rows_ex: softmax_rows with softmax_options_t (NULL options: the
 * same as softmax_rows) and a path choice as in softmax_rows_path
 * (SOFTMAX_PATH_AUTO: the planner's).  Arguments, layout, ownership and
 * errors as for softmax_rows_path; invalid options (scale NaN, <= 0 or
 * > 2^127, causal not 0/1, |causal_offset| >= 2^62) return
 * SOFTMAX_ERR_INVALID_ARG.  softmax_rows and softmax_rows_path are this call
 * with NULL options.
 */
int softmax_rows_ex(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                    int64_t in_row_stride, int64_t out_row_stride, int dtype,
                    const softmax_options_t* options, int path, void* stream);

/*
 * softmax_visible_cols: how many leading columns of row `row` take part in
 * its softmax under `options` (NULL: no mask) for an n_rows x n_cols matrix,
 * computed on the host with the same arithmetic the kernels use; every
 * later column of that row is masked (output +0).  Returns -1 for invalid
 * options or arguments (row outside [0, n_rows), negative sizes, n_rows
 * above 2^62).
 */
int64_t softmax_visible_cols(const softmax_options_t* options, int64_t n_rows, int64_t n_cols,
                             int64_t row);

/*
 * Attention with the row softmax inside it ("Triton GPU programming deep
 * dive", section 3.1: softmax(Q K^T / sqrt(d)) V; section 3.3: the same one
 * tile of keys at a time with a running max and sum, keys past the query
 * masked).  The scores never reach memory.
 *
 *   scale          multiplies Q K^T before the softmax; 0 < scale <= 2^127.
 *                  Without options: 1/sqrt(head_dim).
 *   causal         0: every key.  1: key j is visible to query i iff
 *                  j <= i + causal_offset (0: the pages' mask; n_k - n_q: a
 *                  bottom-right aligned mask).  |causal_offset| < 2^62.
 *   impl           0: the library's choice (the ping-pong kernel, the
 *                  fastest on GB300; the single-tile tcgen05 kernel where
 *                  the ping-pong one cannot run); 1: the warp-level mma.sync
 *                  kernel; 2: the tcgen05 kernel, one 128-query tile per
 *                  CTA; 3: the ping-pong tcgen05 kernel, two 128-query
 *                  tiles per CTA, one tile's softmax overlapping the other's
 *                  products, operands by tensor-map copies
 *                  (SOFTMAX_ERR_UNSUPPORTED if batch_heads, n_q or n_k is
 *                  2^31 or more).
 */
typedef struct {
    float scale;
    int32_t causal;
    int64_t causal_offset;
    int32_t impl;
} softmax_attention_options_t;

/*
 * softmax_attention_forward: O = softmax(scale Q K^T, mask) V for every
 * (batch, head) pair.
 *
 *   q, o   [batch_heads][n_q][head_dim], k, v  [batch_heads][n_k][head_dim],
 *          dense, device memory, 16-byte aligned, dtype SOFTMAX_BF16 or
 *          SOFTMAX_F16 (16-bit operands on the tensor cores, fp32 scores,
 *          softmax and accumulators; the probabilities are rounded to the
 *          operand type for the P V product).
 *   lse    optional [batch_heads][n_q] floats: the natural-log logsumexp of
 *          each query's masked, scaled scores (NULL: not written).
 *   head_dim 64 or 128.  A query with no visible key (or n_k == 0) gives NaN
 *          outputs (the softmax of only -inf) and lse = -inf.  n_k == 0 is
 *          served by the single-tile tcgen05 kernel whatever impl asks for;
 *          k and v may then be NULL.
 *   Ownership and asynchrony as for softmax_rows.  o may be q itself; it must
 *   not otherwise overlap q, k or v; lse must overlap none of q, k, v, o.
 *   Errors: SOFTMAX_ERR_INVALID_ARG (null or misaligned pointers, negative
 *   sizes, bad options, overlap), SOFTMAX_ERR_UNSUPPORTED (fp32, another
 *   head_dim, no usable device, impl 3 outside its limits, a grid of more
 *   than 2^31 - 1 CTAs: batch_heads x the query tiles of the chosen kernel,
 *   64, 128 or 256 queries each), SOFTMAX_ERR_CUDA (launch failure).
 *   batch_heads == 0 or n_q == 0: no-op.
 */
int softmax_attention_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                              int64_t batch_heads, int64_t n_q, int64_t n_k, int64_t head_dim,
                              int dtype, const softmax_attention_options_t* options,
                              void* stream);

/*
 * softmax_strided: the softmax of rows whose elements are not contiguous.
 * Element c of row r is in[r * in_row_stride + c * in_col_stride] and its
 * result goes to out[r * out_row_stride + c * out_col_stride] (ELEMENTS).
 * The cs336 lecture 6 notes ("Lecture 6: GPU Kernel programming and Triton",
 * section "Level 1: Softmax", and its section on strides) take a column-wise
 * softmax by changing only the strides: the softmax down the columns of a
 * row-major R x C matrix is n_rows = C, n_cols = R, row strides 1, column
 * strides C.
 *
 *   Unit column strides: the same as softmax_rows.  Unit row strides with a
 *   16-byte aligned input and memory-row pitch: the tensor-copy columns
 *   kernel (tiles of 128 or 256 bytes of adjacent rows streamed twice in
 *   16 KB boxes, the second read mostly from L2; clusters of up to 8 CTAs
 *   split long rows).  Other unit-row-stride layouts: the staged-tile
 *   columns kernel (128-byte tiles staged in shared memory, one HBM read
 *   and one write per element; rows up to 16 x 512 columns per cluster of
 *   CTAs, longer ones while the tile fits in shared memory).  Other
 *   strides, or longer rows: a general gather kernel (correct for any
 *   layout, two reads per element).
 *   Strides must be >= 0; the output elements must be distinct (its rows
 *   nested within its columns or the reverse); in and out may be the same
 *   buffer with the same strides, and must not otherwise share bytes.
 *   Ownership, asynchrony and errors as for softmax_rows.
 */
int softmax_strided(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                    int64_t in_row_stride, int64_t in_col_stride, int64_t out_row_stride,
                    int64_t out_col_stride, int dtype, void* stream);

/*
 * softmax_backward_rows: the gradient through the row softmax.  Given the
 * forward output y (n_rows x n_cols) and the gradient dy of a loss with
 * respect to y, writes
 *     dx_i = y_i * (dy_i - sum_j y_j dy_j)        for every row,
 * the chain rule through y = softmax(x), whose Jacobian is
 * dy_j/dx_i = y_j (delta_ij - y_i).  ("Triton: write CUDA-grade GPU operators
 * in Python" names fused forward-backward operators among what custom
 * kernels are for; the formula is the derivative of the softmax above.)
 *
 *   y, dy, dx    device pointers, rows starting every y_row_stride,
 *                dy_row_stride and dx_row_stride ELEMENTS; contiguous
 *                columns; the same dtype for all three; fp32 arithmetic.
 *   Ownership and asynchrony as for softmax_rows.  dx may be dy or y itself
 *   (same stride); other overlaps of dx with y or dy are rejected.
 *   Errors: SOFTMAX_ERR_INVALID_ARG for a null pointer with work to do,
 *   negative sizes, a stride below n_cols (n_rows > 1), an unknown dtype or
 *   a partial overlap; SOFTMAX_ERR_UNSUPPORTED without a usable device;
 *   SOFTMAX_ERR_CUDA if the launch fails.  n_rows == 0 or n_cols == 0: no-op.
 */
int softmax_backward_rows(const void* y, const void* dy, void* dx, int64_t n_rows,
                          int64_t n_cols, int64_t y_row_stride, int64_t dy_row_stride,
                          int64_t dx_row_stride, int dtype, void* stream);

/*
 * softmax_rows_host: the same operation on HOST buffers.  Two modes:
 *
 *  staged  (d_in and d_out given): queues on `stream` a copy of the strided
 *          host input into d_in (dense, row stride n_cols), the softmax from
 *          d_in into d_out (dense), and a copy of d_out into the strided host
 *          output.
 *  direct  (d_in == d_out == NULL): h_in and h_out must be host memory the
 *          device can access (pinned / registered with the CUDA runtime, or
 *          managed); the kernel reads the input rows and writes the output
 *          rows in host memory over the host link, with no device buffers and
 *          no separate copies.  Pageable (unregistered) memory returns
 *          SOFTMAX_ERR_INVALID_ARG in this mode.
 *
 * Returns once queued; the caller synchronises `stream` before reading h_out.
 *
 *   h_in, h_out      host pointers.  Staged: pinned memory gives asynchronous
 *                    full-bandwidth copies, pageable memory works but the
 *                    copies then block the calling thread.
 *   d_in, d_out      staged: device buffers of at least n_rows * n_cols
 *                    elements each (d_in == d_out is allowed: in place on the
 *                    device); both NULL selects the direct mode; exactly one
 *                    NULL is SOFTMAX_ERR_INVALID_ARG.
 *   other arguments  as for softmax_rows (strides describe the host buffers).
 *
 * Errors as for softmax_rows; a failed copy returns SOFTMAX_ERR_CUDA.
 */
int softmax_rows_host(const void* h_in, void* h_out, int64_t n_rows, int64_t n_cols,
                      int64_t in_row_stride, int64_t out_row_stride, int dtype,
                      void* d_in, void* d_out, void* stream);

/* Static description of a status code (never NULL). */
const char* softmax_status_string(int status);

/* Device description used by the scheduler.  Fields are what
 * cudaDeviceGetAttribute reports for the device. */
typedef struct {
    int sm_count;                 /* multiprocessors */
    int max_threads_per_sm;
    int max_smem_per_sm;          /* bytes */
    int max_smem_per_block_optin; /* bytes */
    int regs_per_sm;
    int cc_major, cc_minor;       /* compute capability; this build runs on 10.3 */
    int max_cluster;              /* largest thread-block cluster (CTAs) the
                                     row-slice kernel can be co-scheduled with */
} softmax_device_desc_t;

/* The scheduler's decision for one call. */
typedef struct {
    int path;            /* softmax_path_t chosen */
    int dtype;
    int vec;             /* elements per global vector access (1 = scalar) */
    int out_vec;         /* elements per global vector store */
    int bulk_copy;       /* 1: rows staged by cp.async.bulk into shared memory */
    int threads;         /* threads per CTA (TWOPASS staged: consumer threads;
                            the CTA also has one producer warp) */
    int cluster;         /* CTAs per cluster (1: no cluster) */
    int rows_per_warp;   /* WARP path: rows a warp holds at once */
    int chunks;          /* vectors per thread (WARP: per lane per row; CTA and
                            CLUSTER: 16-byte vectors of the slice; TWOPASS
                            staged: 16-byte vectors per thread per ring chunk) */
    int64_t slice_cols;  /* CTA/CLUSTER/TWOPASS: columns owned by one CTA */
    int stages;          /* CTA/CLUSTER: slices in flight per CTA; TWOPASS
                            staged: chunks in the ring (ring depth) */
    int smem_bytes;      /* dynamic shared memory per CTA */
    int64_t grid;        /* CTAs launched; 0 = sized at launch from occupancy
                            in waves of resident CTAs: CTA path up to ten
                            (4-byte elements) or two (2-byte), at least 1.5
                            rows per CTA; WARP path up to four; cluster
                            path one persistent wave; two-pass path one,
                            or two when each CTA owns whole rows and two
                            CTAs fit on an SM */
    int lanes_per_row;   /* WARP path, rows in registers (bulk_copy 0): lanes
                            that share one row, a power of two; below 32 a
                            warp holds 32 / lanes_per_row rows side by side
                            (short rows, chunks 1).  0 is read as 32. */
} softmax_plan_t;

/*
 * softmax_plan: run the row-to-CTA scheduler without launching anything.
 * dev == NULL queries the current CUDA device (needs a GPU); a non-NULL dev
 * makes this a pure host computation, usable without a GPU.  Pointers are
 * only inspected for alignment (they may be fake addresses).  Validation and
 * return codes are those of softmax_rows_path.
 */
int softmax_plan(const softmax_device_desc_t* dev, const void* in, const void* out,
                 int64_t n_rows, int64_t n_cols, int64_t in_row_stride,
                 int64_t out_row_stride, int dtype, int path, softmax_plan_t* plan);

/*
 * softmax_plan_check: the checks softmax_rows_planned applies to *plan before
 * it launches, without launching: SOFTMAX_OK when the plan describes this
 * problem and fits the device, else the code softmax_rows_planned would
 * return (SOFTMAX_ERR_INVALID_ARG for a plan that could read or write outside
 * the rows).  dev == NULL checks against the current CUDA device (needs a
 * GPU); a non-NULL dev makes this a pure host computation.  Pointers are
 * only inspected for alignment and overlap.
 */
int softmax_plan_check(const softmax_device_desc_t* dev, const void* in, const void* out,
                       int64_t n_rows, int64_t n_cols, int64_t in_row_stride,
                       int64_t out_row_stride, int dtype, const softmax_plan_t* plan);

/*
 * softmax_rows_planned: launch with an explicit scheduler decision (tuning
 * sweeps and tests).  *plan must describe this problem: typically the result
 * of softmax_plan with some launch-shape fields changed.  The plan is checked
 * before anything is launched (path and dtype, vector widths against pointer
 * and stride alignment, slice coverage of the row, threads x vectors
 * covering the slice, stage count and shared memory against the device,
 * cluster size); a plan that could read or write outside the rows returns
 * SOFTMAX_ERR_INVALID_ARG.  Otherwise behaves like softmax_rows.
 */
int softmax_rows_planned(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                         int64_t in_row_stride, int64_t out_row_stride, int dtype,
                         const softmax_plan_t* plan, void* stream);

/* Writes a one-line text form of *plan into buf (always NUL-terminated when
 * len > 0).  Returns the number of characters the full text needs. */
int softmax_plan_format(const softmax_plan_t* plan, char* buf, size_t len);

/*
 * softmax_plan_describe: the scheduler's decision, as text, for softmax_rows
 * on n_rows contiguous rows of n_cols elements (strides n_cols, 16-byte
 * aligned device buffers) on the current device.  The launch wrapper of
 * "Triton: write CUDA-grade GPU operators in Python", Example 2 (Fused
 * Softmax), fixes one program per row; this call reports how this library
 * maps the same rows instead (path, threads, cluster, slices, stages, grid).
 *
 *   buf, len  receives the one-line text of softmax_plan_format, truncated
 *             to len - 1 characters and NUL-terminated (len == 0: nothing is
 *             written; buf may then be NULL).
 *   Returns SOFTMAX_OK, SOFTMAX_ERR_INVALID_ARG (bad sizes or dtype, or
 *   buf == NULL with len > 0), SOFTMAX_ERR_UNSUPPORTED (no usable device).
 *   Launches nothing.  A composition of softmax_plan and
 *   softmax_plan_format, which also take other strides and alignments, and
 *   a device description in place of the current device.
 */
int softmax_plan_describe(int64_t n_rows, int64_t n_cols, int dtype, char* buf, size_t len);

/*
 * softmax_device_status: synchronises the current device, then reports
 * whether any kernel of this library gave up a bounded wait (an mbarrier that
 * never completed) since the last clear.  Returns SOFTMAX_OK or
 * SOFTMAX_ERR_DEVICE_TIMEOUT (SOFTMAX_ERR_CUDA if synchronisation fails).
 * clear != 0 resets the flag.
 */
int softmax_device_status(int clear);

/*
 * softmax_selftest_wait_timeout: test hook for the bounded waits.  Queues on
 * `stream` one single-thread kernel that initialises an mbarrier nobody will
 * signal and waits on it with the same bounded wait the CTA/CLUSTER kernels
 * use for their bulk copies (about two seconds).  The wait runs out, the
 * kernel records the timeout and returns normally, so the next
 * softmax_device_status() reports SOFTMAX_ERR_DEVICE_TIMEOUT while the CUDA
 * context stays usable.  No copy is in flight and nothing faults.  Returns
 * the launch status.
 */
int softmax_selftest_wait_timeout(void* stream);

/* Number of kernels this library has launched in this process. */
uint64_t softmax_launch_count(void);

/* SOFTMAX_ABI_VERSION of the loaded library. */
int softmax_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBSOFTMAX_SOFTMAX_H */
