/*
 * Row-wise softmax oracle: plain, slow, single-threaded CPU code in double.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is
 * compared against.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load or call it.  It shares no code,
 * header, table or helper with the CUDA path (row_wise_softmax_gb300/csrc)
 * and includes nothing from it.
 *
 * What it computes, and where the pages define it:
 *  - softmax of each row, y_j = exp(x_j - max x) / sum_k exp(x_k - max x):
 *    "Lecture 6: GPU Kernel programming and Triton" (xwysyy.cn, cs336 lec06),
 *    section "Level 1: Softmax", display formula; the steps (row max, subtract,
 *    exp, row sum, divide) follow the fused softmax kernel of "Triton: write
 *    CUDA-grade GPU operators in Python" (f.mffb.com.cn), example 2
 *    "Fused Softmax".  Positions past n_cols are never read (mask); the
 *    input and the output each have their own row stride, in elements
 *    (example 2's launch wrapper passes x.stride(0) and out.stride(0)).
 *  - the online (m, l) recurrence over column tiles: "Triton GPU programming
 *    deep dive" (ybb.press), section 3.3 "Triton Flash Attention core
 *    implementation" (running max m_i, running sum l_i rescaled by
 *    exp(m_i - m_ij)), with the reading that a tile whose running max is
 *    still -inf contributes nothing (the page does not say what happens when
 *    a whole tile is masked).
 *  - the scaled, causally masked softmax of attention scores: "Triton GPU
 *    programming deep dive", section 3.1 (the scores are divided by sqrt(d)
 *    before the softmax: here a general factor `scale`) and section 3.3 (a
 *    score whose key index exceeds its query index is replaced by -inf
 *    before the running max).  Reading: row r of the matrix is query
 *    (r mod period) of its block of `period` rows, column c is key c, and
 *    an offset shifts the diagonal; so column c takes part iff
 *    c <= (r mod period) + offset.  A masked column is never read.  A row
 *    with no column taking part is the formula over only -inf: all NaN.
 *  - softmax over strided rows (column-wise softmax): lec06 "Level 1"
 *    and its section on strides; see oracle_softmax_strided.
 *  - the softmax backward (the gradient through the row softmax, by the
 *    chain rule; the pages name forward-backward fused operators among the
 *    custom kernels Triton is for, without the formula): see below.
 *  - the tiled row sum with one accumulator per lane: lec06 section
 *    "Level 2: Row Sum (tiling)", worked example of 12 elements, BLOCK 4.
 *  - bf16 and fp16 decoding (exact) and rounding of a double to bf16 or
 *    fp16 with round-to-nearest-even, for the 16-bit comparisons (fp16 I/O
 *    with fp32 arithmetic: the pages' tuning checklist keeps accumulators in
 *    fp32 for float16/bfloat16 inputs).
 *
 * Pins: each function here is checked by tests/test_oracle_pins.py against
 * closed forms, invariants, high-precision brute force (mpmath), a library
 * softmax (torch CPU, double) and the pages' worked example.  No function
 * here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- fp16 (IEEE 754 binary16) <-> double ------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 stored mantissa bits.
 * Exponent field 0: subnormal, m * 2^-24; field 31: infinity (m = 0) or NaN. */
double oracle_f16_to_double(uint16_t bits)
{
    const int neg = (bits >> 15) & 1;
    const int e = (bits >> 10) & 0x1F;
    const int m = bits & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return neg ? -v : v;
}

/*
 * Round a double to the nearest binary16, ties to even, directly from the
 * double.  As for bf16 below: the spacing q of binary16 values around |v| is
 * 2^(e-10) for 2^e <= |v| < 2^(e+1), and 2^-24 below 2^-14; rint(|v|/q) * q
 * is the rounded value (a carry to the next power of two is still exact).
 * Values from (2 - 2^-11) * 2^15 = 65520 up round to infinity.
 */
uint16_t oracle_double_to_f16(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFE00u : 0x7E00u);
    const uint16_t sign = signbit(v) ? 0x8000u : 0u;
    const double a = fabs(v);
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                   /* 2^(e-1) <= a < 2^e */
    int q_exp = (e - 1) - 10;
    if (q_exp < -24)
        q_exp = -24;                /* subnormal spacing */
    const double r = ldexp(rint(ldexp(a, -q_exp)), q_exp);
    if (r < ldexp(1.0, -14))        /* subnormal (or zero): field 0 */
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
    int e2;
    frexp(r, &e2);                  /* 2^(e2-1) <= r < 2^e2 */
    const int biased = (e2 - 1) + 15;
    const int mant = (int)(ldexp(r, -(e2 - 1 - 10)) - 1024.0);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)mant);
}

void oracle_double_to_f16_array(const double* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_double_to_f16(v[i]);
}

void oracle_f16_to_double_array(const uint16_t* b, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f16_to_double(b[i]);
}

/* ---- bf16 <-> double ------------------------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16 (8 exponent bits, 7 stored mantissa
 * bits), ties to even, directly from the double (no intermediate binary32,
 * so no double rounding).
 *
 * Method: for |v| in the normal bf16 range the spacing of bf16 values is
 * q = 2^(e-7) where 2^e <= |v| < 2^(e+1); below 2^-126 it is the subnormal
 * spacing 2^-133.  |v|/q is exact (q is a power of two), rint() rounds it to
 * an integer with ties to even (default rounding mode), and the product with
 * q is a bf16 value, exactly representable in binary32.
 */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    const int neg = signbit(v) ? 1 : 0;
    const double a = fabs(v);
    /* Halfway between the largest finite bf16, (2 - 2^-7) * 2^127, and
     * 2^128; the largest finite bf16 has an odd mantissa, so the tie goes up. */
    const double overflow_at = ldexp(2.0 - ldexp(1.0, -8), 127);
    float r;
    if (a >= overflow_at) {
        r = INFINITY;
    } else if (a == 0.0) {
        r = 0.0f;
    } else {
        int e;
        frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1) */
        int q_exp = (e - 1) - 7;    /* 2^(e-1) <= a < 2^e */
        if (q_exp < -133)
            q_exp = -133;           /* subnormal spacing */
        const double n = rint(ldexp(a, -q_exp));
        r = (float)ldexp(n, q_exp); /* exact: n < 2^9, result is a bf16 */
    }
    uint32_t u;
    memcpy(&u, &r, sizeof u);
    uint16_t b = (uint16_t)(u >> 16);
    if (neg)
        b |= 0x8000u;
    return b;
}

void oracle_double_to_bf16_array(const double* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_double_to_bf16(v[i]);
}

void oracle_bf16_to_double_array(const uint16_t* b, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_double(b[i]);
}

/* ---- softmax of one row, from its exact values ------------------------ */

/*
 * y_j = exp(x_j - m) / l with m = max_j x_j and l = sum_j exp(x_j - m),
 * summed left to right.  IEEE semantics decide the degenerate rows without
 * special cases: a NaN anywhere makes l NaN; +inf makes inf - inf = NaN;
 * a row of only -inf has m = -inf and -inf - (-inf) = NaN.  In each case the
 * whole row is NaN, which is what the formula gives.
 */
static void softmax_row(const double* x, int64_t n, double* y)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (x[j] > m)
            m = x[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        y[j] = exp(x[j] - m);
        l += y[j];
    }
    for (int64_t j = 0; j < n; ++j)
        y[j] = y[j] / l;
}

/*
 * The same row via the online recurrence, one tile of `tile` columns at a
 * time: m_new = max(m, max(tile)), l = l * exp(m - m_new) + sum exp(x - m_new).
 * While m_new is still -inf (every value so far is -inf) the tile adds
 * nothing and (m, l) stays (-inf, 0); a NaN in such a tile still makes l NaN.
 * The final division uses the last m and l.
 */
static void online_softmax_row(const double* x, int64_t n, int64_t tile, double* y)
{
    double m = -INFINITY, l = 0.0;
    for (int64_t t0 = 0; t0 < n; t0 += tile) {
        const int64_t t1 = (t0 + tile < n) ? t0 + tile : n;
        double bm = -INFINITY;
        int has_nan = 0;
        for (int64_t j = t0; j < t1; ++j) {
            if (isnan(x[j]))
                has_nan = 1;
            else if (x[j] > bm)
                bm = x[j];
        }
        const double m_new = (bm > m) ? bm : m;
        if (m_new == -INFINITY) {
            if (has_nan)
                l = NAN;
            continue;
        }
        double s = 0.0;
        for (int64_t j = t0; j < t1; ++j)
            s += exp(x[j] - m_new);
        l = l * exp(m - m_new) + s;
        m = m_new;
    }
    for (int64_t j = 0; j < n; ++j)
        y[j] = exp(x[j] - m) / l;
}

/* ---- row-matrix entry points ----------------------------------------- */
/*
 * The number of leading columns of row r that take part in its softmax:
 * n_cols without a mask; with one, the columns c <= (r mod period) + offset,
 * i.e. (r mod period) + offset + 1 of them, clamped to [0, n_cols].
 */
static int64_t visible_cols(int64_t r, int64_t n_cols, int causal, int64_t period, int64_t offset)
{
    if (!causal)
        return n_cols;
    const int64_t last = r % period + offset;       /* last column taking part */
    if (last < 0)
        return 0;
    return last + 1 < n_cols ? last + 1 : n_cols;
}

/*
 * dtype 0: `in` is binary32; dtype 1: `in` is bf16 bit patterns (uint16);
 * dtype 2: `in` is binary16 bit patterns (uint16).
 * Row r of the input starts at element r * in_row_stride; row r of the
 * output (double) at element r * out_row_stride.  Only columns [0, n_cols)
 * are written, and only the columns taking part are read.  The softmax is
 * taken over z_c = scale * x_c (exact in double: both factors have at most
 * 24 significant bits) for the columns taking part, and z_c = -inf for the
 * masked ones.  `tile` <= 0 selects the plain definition, > 0 the online
 * recurrence with that tile width.  causal != 0 enables the mask; period
 * <= 0 means n_rows.  Returns 0, or -1 on a bad argument.
 */
int oracle_softmax_rows_ex(const void* in, double* out, int64_t n_rows, int64_t n_cols,
                           int64_t in_row_stride, int64_t out_row_stride, int dtype,
                           int64_t tile, double scale, int causal, int64_t period,
                           int64_t offset)
{
    if (n_rows < 0 || n_cols < 0 || dtype < 0 || dtype > 2 || !(scale > 0.0))
        return -1;
    if (n_rows == 0 || n_cols == 0)
        return 0;
    if (!in || !out)
        return -1;
    if (period <= 0)
        period = n_rows;
    double* x = (double*)malloc((size_t)n_cols * sizeof(double));
    if (!x)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t vis = visible_cols(r, n_cols, causal, period, offset);
        if (dtype == 0) {
            const float* src = (const float*)in + r * in_row_stride;
            for (int64_t j = 0; j < vis; ++j)
                x[j] = scale * (double)src[j];
        } else if (dtype == 1) {
            const uint16_t* src = (const uint16_t*)in + r * in_row_stride;
            for (int64_t j = 0; j < vis; ++j)
                x[j] = scale * oracle_bf16_to_double(src[j]);
        } else {
            const uint16_t* src = (const uint16_t*)in + r * in_row_stride;
            for (int64_t j = 0; j < vis; ++j)
                x[j] = scale * oracle_f16_to_double(src[j]);
        }
        for (int64_t j = vis; j < n_cols; ++j)
            x[j] = -INFINITY;
        double* y = out + r * out_row_stride;
        if (tile > 0)
            online_softmax_row(x, n_cols, tile, y);
        else
            softmax_row(x, n_cols, y);
    }
    free(x);
    return 0;
}

/*
 * Softmax over arbitrarily strided rows: element c of row r is
 * in[r * in_row_stride + c * in_col_stride] (elements).  Column-wise softmax
 * of a row-major matrix is the case in_row_stride = 1, in_col_stride = its
 * row length: "Lecture 6: GPU Kernel programming and Triton", section
 * "Level 1: Softmax", notes that only the strides change to take the softmax
 * along columns, and its section on strides writes the address of element
 * [row, col] as ptr + row * stride_row + col * stride_col.  The output is
 * dense double [n_rows][n_cols]; each row is gathered and then reduced by the
 * plain definition.  Returns 0, or -1 on a bad argument.
 */
int oracle_softmax_strided(const void* in, double* out, int64_t n_rows, int64_t n_cols,
                           int64_t in_row_stride, int64_t in_col_stride, int dtype)
{
    if (n_rows < 0 || n_cols < 0 || dtype < 0 || dtype > 2)
        return -1;
    if (n_rows == 0 || n_cols == 0)
        return 0;
    if (!in || !out)
        return -1;
    double* x = (double*)malloc((size_t)n_cols * sizeof(double));
    if (!x)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t c = 0; c < n_cols; ++c) {
            const int64_t idx = r * in_row_stride + c * in_col_stride;
            if (dtype == 0)
                x[c] = (double)((const float*)in)[idx];
            else if (dtype == 1)
                x[c] = oracle_bf16_to_double(((const uint16_t*)in)[idx]);
            else
                x[c] = oracle_f16_to_double(((const uint16_t*)in)[idx]);
        }
        softmax_row(x, n_cols, out + r * n_cols);
    }
    free(x);
    return 0;
}

/* The plain softmax of each row: no scale, no mask. */
int oracle_softmax_rows(const void* in, double* out, int64_t n_rows, int64_t n_cols,
                        int64_t in_row_stride, int64_t out_row_stride, int dtype,
                        int64_t tile)
{
    return oracle_softmax_rows_ex(in, out, n_rows, n_cols, in_row_stride, out_row_stride,
                                  dtype, tile, 1.0, 0, 0, 0);
}

/*
 * Tiled row sum with one accumulator per lane (lec06 "Level 2"): lane i adds
 * x[t * block + i] for every tile t, then the lanes are summed.  Writes the
 * lane accumulators after `snapshot_tiles` tiles into acc_out[block] (all of
 * them when snapshot_tiles >= number of tiles) and returns the row sum.
 */
double oracle_tiled_row_sum(const double* x, int64_t n, int64_t block,
                            int64_t snapshot_tiles, double* acc_out)
{
    double* acc = (double*)calloc((size_t)block, sizeof(double));
    if (!acc)
        return NAN;
    int64_t tiles_done = 0;
    for (int64_t t0 = 0; t0 < n; t0 += block) {
        if (tiles_done == snapshot_tiles && acc_out)
            memcpy(acc_out, acc, (size_t)block * sizeof(double));
        for (int64_t i = 0; i < block; ++i)
            if (t0 + i < n)         /* masked lanes load 0 */
                acc[i] += x[t0 + i];
        ++tiles_done;
    }
    if (tiles_done <= snapshot_tiles && acc_out)
        memcpy(acc_out, acc, (size_t)block * sizeof(double));
    double s = 0.0;
    for (int64_t i = 0; i < block; ++i)
        s += acc[i];
    free(acc);
    return s;
}

/* ---- softmax backward --------------------------------------------------- */

/* Element j of row r of a 16-bit or binary32 buffer, exactly, as a double. */
static double load_elem(const void* base, int64_t idx, int dtype)
{
    if (dtype == 0)
        return (double)((const float*)base)[idx];
    const uint16_t b = ((const uint16_t*)base)[idx];
    return dtype == 1 ? oracle_bf16_to_double(b) : oracle_f16_to_double(b);
}

/*
 * The gradient of the row softmax y = softmax(x) with respect to x, given y
 * and the gradient dy of a loss with respect to y.  The Jacobian of the
 * softmax is dy_j/dx_i = y_j (delta_ij - y_i), so by the chain rule
 *     dx_i = sum_j dy_j y_j (delta_ij - y_i) = y_i (dy_i - sum_j y_j dy_j).
 * Computed in double from the exact values of y and dy, the dot product
 * summed left to right.  Row r of y, dy and dx starts at r times its own
 * stride (elements); dx is double.  Returns 0, or -1 on a bad argument.
 */
int oracle_softmax_backward_rows(const void* y, const void* dy, double* dx, int64_t n_rows,
                                 int64_t n_cols, int64_t y_row_stride, int64_t dy_row_stride,
                                 int64_t dx_row_stride, int dtype)
{
    if (n_rows < 0 || n_cols < 0 || dtype < 0 || dtype > 2)
        return -1;
    if (n_rows == 0 || n_cols == 0)
        return 0;
    if (!y || !dy || !dx)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        double dot = 0.0;
        for (int64_t j = 0; j < n_cols; ++j)
            dot += load_elem(y, r * y_row_stride + j, dtype) *
                   load_elem(dy, r * dy_row_stride + j, dtype);
        for (int64_t j = 0; j < n_cols; ++j) {
            const double yj = load_elem(y, r * y_row_stride + j, dtype);
            const double gj = load_elem(dy, r * dy_row_stride + j, dtype);
            dx[r * dx_row_stride + j] = yj * (gj - dot);
        }
    }
    return 0;
}
