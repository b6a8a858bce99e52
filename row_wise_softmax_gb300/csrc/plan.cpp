// Row-to-CTA scheduler: argument validation and the choice of execution path
// and launch shape.  Pure host code: it reads a device description and the
// pointers' alignment, never the device, so it runs without a GPU.
//
// Paths by row length (n_cols, element size esz):
//   WARP     n_cols <= 1024: a warp owns rows in registers (short rows).
//   CTA      row <= 64 KB: one CTA per row, the row staged in shared memory.
//   CLUSTER  row <= max_cluster slices of <= 96 KB: a cluster per row, each
//            CTA holding a slice in shared memory (long rows, single HBM pass).
//   TWOPASS  anything longer: a cluster streams the row twice.
// The 64 KB / 96 KB slice caps keep two or three CTAs resident per SM
// (228 KB of shared memory each on GB300), so the copy engine has several
// slices in flight per SM while others are being reduced or stored.
//
// Whole waves (the "Block Occupancy: tail effect" rule of the cs336 lecture
// 6 notes): the WARP and TWOPASS grids are persistent, sized at launch to the
// number of CTAs (clusters) the device can hold at once; the CTA and CLUSTER
// grids launch one CTA (cluster) per row and rely on many resident CTAs per
// SM and the hardware block scheduler to balance the tail.
#include "kernels.h"

#include <stdint.h>

namespace rwsm {

namespace {

constexpr int64_t kWarpMaxCols = 1024;
constexpr int64_t kCtaMaxBytes = 64 * 1024;
constexpr int64_t kSliceBytesSmallCluster = 64 * 1024;   // cluster <= 8
constexpr int64_t kSliceBytesLargeCluster = 96 * 1024;   // cluster 16
constexpr int kSmemReserve = 2048;                        // static smem + slack

int esize(int dtype) { return dtype == SOFTMAX_F32 ? 4 : 2; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

int64_t pow2_ceil(int64_t v)
{
    int64_t p = 1;
    while (p < v)
        p <<= 1;
    return p;
}

int64_t pow2_floor(int64_t v)
{
    int64_t p = 1;
    while (p * 2 <= v)
        p <<= 1;
    return p;
}

bool aligned16(const void* ptr, int64_t n_rows, int64_t ld, int esz)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    return (a % 16 == 0) && (n_rows <= 1 || (ld * esz) % 16 == 0);
}

// Rows held in flight per warp on the WARP path (must match warp_rows.cu).
int warp_rows_for(int e)
{
    return e >= 16 ? 1 : (16 / e > 8 ? 8 : 16 / e);
}

// Threads for a shared-memory slice of nv 16-byte vectors: about four
// vectors per thread, between 128 and 512 threads.
int slice_threads(int64_t nv)
{
    int64_t t = pow2_floor(ceil_div(nv, 4) > 0 ? ceil_div(nv, 4) : 1);
    if (t < 128)
        t = 128;
    if (t > 512)
        t = 512;
    return static_cast<int>(t);
}

// Does [a_lo, a_hi) intersect [b_lo, b_hi)?
bool ranges_intersect(uintptr_t a_lo, uintptr_t a_hi, uintptr_t b_lo, uintptr_t b_hi)
{
    return a_lo < b_hi && b_lo < a_hi;
}

}  // namespace

int validate(const void* in, const void* out, int64_t n_rows, int64_t n_cols,
             int64_t ld_in, int64_t ld_out, int dtype)
{
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16)
        return SOFTMAX_ERR_INVALID_ARG;
    if (n_rows < 0 || n_cols < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    if (!in || !out)
        return SOFTMAX_ERR_INVALID_ARG;
    const int esz = esize(dtype);
    if (reinterpret_cast<uintptr_t>(in) % esz || reinterpret_cast<uintptr_t>(out) % esz)
        return SOFTMAX_ERR_INVALID_ARG;
    if (n_cols > 0x7fffffff)
        return SOFTMAX_ERR_INVALID_ARG;
    if (n_rows > 1 && (ld_in < n_cols || ld_out < n_cols))
        return SOFTMAX_ERR_INVALID_ARG;
    // Extents in elements must fit in int64 and in the address space.
    const int64_t lim = INT64_MAX / 4;
    const int64_t li = n_rows > 1 ? ld_in : 0, lo = n_rows > 1 ? ld_out : 0;
    if ((li > 0 && n_rows - 1 > (lim - n_cols) / li) || (lo > 0 && n_rows - 1 > (lim - n_cols) / lo))
        return SOFTMAX_ERR_INVALID_ARG;
    const uintptr_t in_lo = reinterpret_cast<uintptr_t>(in);
    const uintptr_t out_lo = reinterpret_cast<uintptr_t>(out);
    const uintptr_t in_hi = in_lo + static_cast<uintptr_t>(((n_rows - 1) * li + n_cols) * esz);
    const uintptr_t out_hi = out_lo + static_cast<uintptr_t>(((n_rows - 1) * lo + n_cols) * esz);
    if (in_hi < in_lo || out_hi < out_lo)
        return SOFTMAX_ERR_INVALID_ARG;
    if (!ranges_intersect(in_lo, in_hi, out_lo, out_hi))
        return SOFTMAX_OK;
    if (in == out && (n_rows == 1 || ld_in == ld_out))
        return SOFTMAX_OK;                              // in place
    if (n_rows > 1 && ld_in != ld_out)
        return SOFTMAX_ERR_INVALID_ARG;                 // conservative
    // Equal strides (or one row): element sets overlap iff some row shift k
    // puts out row r+k within n_cols elements of in row r.
    const int64_t diff = static_cast<int64_t>(out_lo - in_lo);
    if (diff % esz)
        return SOFTMAX_ERR_INVALID_ARG;
    const int64_t d = diff / esz;
    if (n_rows == 1)
        return (d > -n_cols && d < n_cols) ? SOFTMAX_ERR_INVALID_ARG : SOFTMAX_OK;
    const int64_t ld = ld_in;
    // Shifts near -d/ld are the only candidates (|d + k*ld| < n_cols <= ld).
    int64_t k0 = -d / ld;
    for (int64_t k = k0 - 1; k <= k0 + 1; ++k) {
        if (k <= -n_rows || k >= n_rows)
            continue;
        const int64_t off = d + k * ld;
        if (off > -n_cols && off < n_cols)
            return SOFTMAX_ERR_INVALID_ARG;
    }
    return SOFTMAX_OK;
}

int make_plan(const softmax_device_desc_t& dev, const Problem& p, int path, softmax_plan_t* plan)
{
    if (!plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const int st = validate(p.in, p.out, p.n_rows, p.n_cols, p.ld_in, p.ld_out, p.dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (path < SOFTMAX_PATH_AUTO || path > SOFTMAX_PATH_TWOPASS)
        return SOFTMAX_ERR_INVALID_ARG;
    if (dev.cc_major != 10 || dev.cc_minor != 3)
        return SOFTMAX_ERR_UNSUPPORTED;

    const int esz = esize(p.dtype);
    const int vmax = 16 / esz;
    const bool in_al = aligned16(p.in, p.n_rows, p.ld_in, esz);
    const bool out_al = aligned16(p.out, p.n_rows, p.ld_out, esz);
    const int64_t row_bytes = p.n_cols * esz;
    const int64_t smem_cap = static_cast<int64_t>(dev.max_smem_per_block_optin) - kSmemReserve;
    const int max_cluster = dev.max_cluster < 1 ? 1 : (dev.max_cluster > 16 ? 16 : dev.max_cluster);

    // Smallest cluster (>= 2) whose slices fit the per-slice cap.
    auto cluster_for = [&](int64_t cap_small, int64_t cap_large) -> int {
        for (int cs = 2; cs <= max_cluster; cs *= 2) {
            const int64_t slice_bytes = round_up(ceil_div(p.n_cols, cs), vmax) * esz;
            const int64_t cap = cs <= 8 ? cap_small : cap_large;
            if (slice_bytes <= cap && slice_bytes <= smem_cap)
                return cs;
        }
        return 0;
    };

    if (path == SOFTMAX_PATH_AUTO) {
        if (p.n_cols <= kWarpMaxCols)
            path = SOFTMAX_PATH_WARP;
        else if (row_bytes <= kCtaMaxBytes && row_bytes <= smem_cap)
            path = SOFTMAX_PATH_CTA;
        else if (cluster_for(kSliceBytesSmallCluster, kSliceBytesLargeCluster))
            path = SOFTMAX_PATH_CLUSTER;
        else
            path = SOFTMAX_PATH_TWOPASS;
    }

    softmax_plan_t q = {};
    q.path = path;
    q.dtype = p.dtype;
    q.cluster = 1;
    switch (path) {
    case SOFTMAX_PATH_WARP: {
        if (p.n_cols > kWarpMaxCols)
            return SOFTMAX_ERR_UNSUPPORTED;
        q.vec = (in_al && out_al) ? vmax : 1;
        q.out_vec = q.vec;
        q.chunks = static_cast<int>(pow2_ceil(ceil_div(p.n_cols, 32 * q.vec)));
        q.rows_per_warp = warp_rows_for(q.vec * q.chunks);
        q.threads = 128;
        q.slice_cols = p.n_cols;
        q.grid = 0;
        break;
    }
    case SOFTMAX_PATH_CTA:
    case SOFTMAX_PATH_CLUSTER: {
        int cs = 1;
        if (path == SOFTMAX_PATH_CLUSTER) {
            // Forced or automatic: prefer the regular caps, else anything
            // that fits shared memory.
            cs = cluster_for(kSliceBytesSmallCluster, kSliceBytesLargeCluster);
            if (!cs)
                cs = cluster_for(smem_cap, smem_cap);
            if (!cs)
                return SOFTMAX_ERR_UNSUPPORTED;
        }
        const int64_t slice = round_up(ceil_div(p.n_cols, cs), vmax);
        if (slice * esz > smem_cap)
            return SOFTMAX_ERR_UNSUPPORTED;
        q.cluster = cs;
        q.slice_cols = slice;
        q.smem_bytes = static_cast<int>(slice * esz);
        q.vec = vmax;
        q.out_vec = out_al ? vmax : 1;
        q.bulk_copy = in_al ? 1 : 0;
        q.threads = slice_threads(slice / vmax);
        q.grid = p.n_rows * cs;
        break;
    }
    case SOFTMAX_PATH_TWOPASS: {
        int64_t cs = pow2_floor(p.n_cols / 8192 > 0 ? p.n_cols / 8192 : 1);
        if (cs > max_cluster)
            cs = pow2_floor(max_cluster);
        q.cluster = static_cast<int>(cs);
        q.vec = (in_al && out_al) ? vmax : 1;
        q.out_vec = q.vec;
        q.slice_cols = round_up(ceil_div(p.n_cols, cs), vmax);
        q.threads = 512;
        q.grid = 0;
        break;
    }
    default:
        return SOFTMAX_ERR_INVALID_ARG;
    }
    *plan = q;
    return SOFTMAX_OK;
}

}  // namespace rwsm
