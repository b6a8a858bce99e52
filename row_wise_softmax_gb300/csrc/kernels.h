// Internal interface between the C ABI (softmax_abi.cu), the scheduler
// (plan.cpp) and the kernel translation units.  Not installed; the public
// interface is include/softmax.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "softmax.h"

namespace rwsm {

struct Problem {
    const void* in;
    void* out;
    int64_t n_rows, n_cols, ld_in, ld_out;
    int dtype;
    bool no_bulk = false;   // rows live in host memory: no cp.async.bulk staging
    // Logit transform (softmax_rows_ex): z = scale * x, optional causal mask.
    float scale = 1.0f;
    int causal = 0;
    int64_t causal_period = 0;   // > 0 when causal
    int64_t causal_offset = 0;
};

// Logit transform passed to every kernel.  The softmax is taken over
// z = scale * x (scale > 0, default 1) with an optional causal mask: column c
// of row r takes part iff c <= (r mod period) + offset; every other column is
// -inf.  Because scale > 0, max z = scale * max x and z - max z =
// scale * (x - max x), so the scale only changes the exponent multiplier
// k = scale * log2 e: e^(z - max z) = 2^((x - max x) * k).  Masked columns are
// never loaded: a row's loads stop at logits_valid(row).
struct LogitsArg {
    float k;             // scale * log2(e)
    int causal;          // 0: no mask
    int64_t period;      // > 0
    int64_t offset;
    // row mod period without a 64-bit division: q = floor(row / period) is
    // SRL(t + SRL(row - t, sh1), sh2) with t = MULUH(mul, row), the unsigned
    // division by an invariant integer of Granlund and Montgomery, "Division
    // by invariant integers using multiplication" (PLDI 1994), figure 4.1,
    // for 64-bit words (exact for every row in [0, 2^64)).
    uint64_t mul;
    int sh1, sh2;
};

__host__ __device__ __forceinline__ uint64_t mulhi_u64(uint64_t a, uint64_t b)
{
#ifdef __CUDA_ARCH__
    return __umul64hi(a, b);
#else
    return static_cast<uint64_t>((static_cast<unsigned __int128>(a) * b) >> 64);
#endif
}

// Columns [0, valid) of `row` take part in its softmax: all of them, or with
// the causal mask those c <= (row mod period) + offset.
// row mod period: the row's position in the mask period.
__host__ __device__ __forceinline__ uint64_t logits_period_pos(const LogitsArg& lg, int64_t row)
{
    const uint64_t n = static_cast<uint64_t>(row);
    const uint64_t t = mulhi_u64(lg.mul, n);
    const uint64_t q = (t + ((n - t) >> lg.sh1)) >> lg.sh2;
    return n - q * static_cast<uint64_t>(lg.period);
}

// Kept columns of a causally masked row at position `pos` of the period.
__host__ __device__ __forceinline__ int64_t logits_lim(const LogitsArg& lg, uint64_t pos,
                                                       int64_t n_cols)
{
    const int64_t lim = static_cast<int64_t>(pos) + lg.offset + 1;
    return lim < 0 ? 0 : (lim > n_cols ? n_cols : lim);
}

__host__ __device__ __forceinline__ int64_t logits_valid(const LogitsArg& lg, int64_t row,
                                                         int64_t n_cols)
{
    if (!lg.causal)
        return n_cols;
    return logits_lim(lg, logits_period_pos(lg, row), n_cols);
}

// Kernels are compiled twice: OPTS = false for the plain softmax (scale 1, no
// mask: the multiplier is the constant log2 e and every column takes part,
// with no per-row arithmetic), OPTS = true for any softmax_options_t.
inline bool has_options(const Problem& p)
{
    return p.causal != 0 || p.scale != 1.0f;
}

// logits_valid for either compilation.
template <bool OPTS>
__host__ __device__ __forceinline__ int64_t kept_cols(const LogitsArg& lg, int64_t row,
                                                      int64_t n_cols)
{
    if constexpr (OPTS)
        return logits_valid(lg, row, n_cols);
    else
        return n_cols;
}

// Multiplier and shifts of the division by d >= 1 (figure 4.1 above, N = 64):
// l = ceil(log2 d), mul = floor(2^64 (2^l - d) / d) + 1, sh1 = min(l, 1),
// sh2 = max(l - 1, 0).
inline void divisor_magic(uint64_t d, uint64_t* mul, int* sh1, int* sh2)
{
    int l = 0;
    while (l < 64 && (static_cast<unsigned __int128>(1) << l) < d)
        ++l;
    const unsigned __int128 two64 = static_cast<unsigned __int128>(1) << 64;
    const unsigned __int128 num = two64 * ((static_cast<unsigned __int128>(1) << l) - d);
    *mul = static_cast<uint64_t>(num / d + 1);
    *sh1 = l < 1 ? l : 1;
    *sh2 = l - 1 > 0 ? l - 1 : 0;
}

inline LogitsArg logits_of(const Problem& p)
{
    const float log2e = 1.4426950408889634f;
    LogitsArg a;
    a.k = p.scale == 1.0f ? log2e : static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    a.causal = p.causal;
    a.period = p.causal_period > 0 ? p.causal_period : 1;
    a.offset = p.causal_offset;
    divisor_magic(static_cast<uint64_t>(a.period), &a.mul, &a.sh1, &a.sh2);
    return a;
}

// Scheduler (plan.cpp): validation and the path / launch-shape decision.
int validate(const void* in, const void* out, int64_t n_rows, int64_t n_cols,
             int64_t ld_in, int64_t ld_out, int dtype);
int make_plan(const softmax_device_desc_t& dev, const Problem& p, int path,
              softmax_plan_t* plan);
// Validate softmax_options_t into the problem (softmax_abi.cu).
int apply_options(const softmax_options_t* o, Problem* p);
// Is a caller-supplied plan safe and complete for this problem?
int check_plan(const softmax_device_desc_t& dev, const Problem& p, const softmax_plan_t& plan);

// Softmax backward (backward_rows.cu): dx = y * (dy - sum(y * dy)) per row.
struct BackwardProblem {
    const void* y;
    const void* dy;
    void* dx;
    int64_t n_rows, n_cols;
    int64_t ld_y, ld_dy, ld_dx;
    int dtype;
};
constexpr int64_t kBackwardWarpMaxCols = 1024;      // warp per row up to here
// `vec`: y, dy and dx rows all 16-byte aligned (vector access).
cudaError_t launch_backward_rows(const BackwardProblem& p, bool vec, cudaStream_t s);

// Softmax over strided rows (columns.cu): element c of row r at
// r * row_stride + c * col_stride, in and out each with their own strides.
struct StridedProblem {
    const void* in;
    void* out;
    int64_t n_rows, n_cols;
    int64_t in_row_stride, in_col_stride, out_row_stride, out_col_stride;
    int dtype;
};
// Launch shape of the columns kernel (unit row strides): a cluster of
// `cluster` CTAs per tile of 128 bytes of adjacent rows, `rows_per_cta`
// memory rows (softmax columns) staged per CTA.  ok = false: use the gather
// kernel.
struct ColumnsShape {
    bool ok;
    bool stream;            // the staged (tensor-copy) columns kernel
    int row_bytes;          // staged kernel: tile width in bytes of a memory row
    int cluster, rows_per_cta, smem_bytes, stages;
    int64_t tiles;
    bool vec_in, vec_out;
};
constexpr int64_t kColumnsRowsPerCta = 512;
constexpr int64_t kColumnsMaxCluster = 16;
ColumnsShape columns_shape(const StridedProblem& p, int max_smem_per_block);
cudaError_t launch_strided(const StridedProblem& p, const ColumnsShape& sh, cudaStream_t s);
// Staged columns kernel (columns_stream.cu): 16 KB boxes of a tile's memory
// row segments by the tensor memory accelerator, two passes, clusters split
// the memory rows.  ok = false when the input layout does not allow it.
ColumnsShape columns_stream_shape(const StridedProblem& p, int sm_count, int max_smem_per_sm);
cudaError_t launch_columns_stream(const StridedProblem& p, const ColumnsShape& sh, cudaStream_t s);
unsigned read_error_columns_stream(bool clear);

// Attention forward (attention_mma.cu): O = softmax(scale Q K^T, mask) V per
// (batch, head); q, o [bh][n_q][head_dim], k, v [bh][n_k][head_dim], 16-bit.
struct AttentionProblem {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;                 // [bh][n_q] natural-log logsumexp, or null
    int64_t bh, n_q, n_k, head_dim;
    int dtype;
    float scale;
    int causal;
    int64_t offset;             // key j visible to query i iff j <= i + offset
};
cudaError_t launch_attention_mma(const AttentionProblem& p, cudaStream_t s);   // mma.sync
cudaError_t launch_attention_tc(const AttentionProblem& p, cudaStream_t s);    // tcgen05
unsigned read_error_attention_tc(bool clear);

// Launchers, one per path (each in its own translation unit).
cudaError_t launch_warp_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_tile_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_row_slices(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_row_slices_options(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_twopass(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);
cudaError_t launch_stream_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s);

// Largest cluster the row-slice kernel can launch with on the current device.
int max_cluster_size_row_slices();

// Error words of the translation units that wait on mbarriers: read and
// optionally clear (host side, after the device has been synchronised).
unsigned read_error_row_slices(bool clear);
unsigned read_error_row_slices_options(bool clear);
unsigned read_error_tile_rows(bool clear);
unsigned read_error_stream_rows(bool clear);
cudaError_t launch_selftest_wait(cudaStream_t s);

// Launch attributes shared by every kernel launch: a cluster dimension when
// cs > 1, and programmatic stream serialisation (the kernels begin with
// griddepcontrol.wait).  Returns the number of attributes written (<= 2).
inline int launch_attrs(cudaLaunchAttribute* a, int cs)
{
    int n = 0;
    if (cs > 1) {
        a[n].id = cudaLaunchAttributeClusterDimension;
        a[n].val.clusterDim.x = static_cast<unsigned>(cs);
        a[n].val.clusterDim.y = 1;
        a[n].val.clusterDim.z = 1;
        ++n;
    }
    a[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    return n;
}

// Persistent grid size for `work` equal units (rows, tiles, row groups)
// dealt round-robin to at most `max_active` resident CTAs (or clusters):
// the last round should be as full as possible (the tail effect of the cs336
// lecture 6 notes, "Block Occupancy", applied to units per CTA).  Among
// g in [max_active/2, max_active], take those whose idle share of the last
// round, (g * ceil(work/g) - work) / (g * ceil(work/g)), is within 1% of the
// best; prefer a multiple of `sm_count`, then the largest.
inline int64_t balanced_grid(int64_t work, int64_t max_active, int64_t sm_count)
{
    if (work <= 0 || max_active <= 0)
        return 1;
    if (work <= max_active)
        return work;
    const int64_t lo = (max_active + 1) / 2;
    double best = 1.0;
    for (int64_t g = lo; g <= max_active; ++g) {
        const int64_t slots = g * ((work + g - 1) / g);
        const double idle = static_cast<double>(slots - work) / static_cast<double>(slots);
        if (idle < best)
            best = idle;
    }
    int64_t pick = -1, pick_mult = -1;
    for (int64_t g = lo; g <= max_active; ++g) {
        const int64_t slots = g * ((work + g - 1) / g);
        const double idle = static_cast<double>(slots - work) / static_cast<double>(slots);
        if (idle > best + 0.01)
            continue;
        pick = g;
        if (sm_count > 0 && g % sm_count == 0)
            pick_mult = g;
    }
    return pick_mult > 0 ? pick_mult : pick;
}

// Helpers implemented in softmax_abi.cu.
int resident_ctas(const void* kernel, int threads, int smem_bytes);  // whole-GPU CTA slots
int sm_count_current();
void note_launch();

}  // namespace rwsm
