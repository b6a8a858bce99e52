// Row-to-CTA scheduler: argument validation and the choice of execution path
// and launch shape.  Pure host code: it reads a device description and the
// pointers' alignment, never the device, so it runs without a GPU.
//
// Paths by row length (n_cols, element size esz), chosen from measured
// GB300 sweeps over row lengths:
//   WARP     n_cols <= 1024: a warp owns rows.  fp32 rows stay in registers
//            (software-pipelined loads); bf16 rows with 16-byte aligned input
//            go through the staged tile kernel (cp.async.bulk ring of rows).
//   CTA      row <= 32 KB: a persistent CTA per row at a time, the row staged
//            by cp.async.bulk and held in registers (one ring stage: the
//            register copy is the second buffer).
//   CLUSTER  rows of 32..64 KB whose input is not 16-byte aligned: one HBM
//            pass, a cluster of CTAs holding <= 32 KB slices, max and sum
//            exchanged through distributed shared memory.  (When forced:
//            slices up to 128 KB fp32 / 64 KB bf16.)
//   TWOPASS  longer rows (every row beyond 32 KB when the input is 16-byte
//            aligned): a cluster of 1..4 CTAs (about 256 KB of fp32 row or
//            1 MB of 16-bit row per CTA) streams the row twice through a
//            cp.async.bulk chunk ring fed by a producer warp; the second read
//            mostly hits L2.  Unaligned input: the register two-pass kernel
//            (about 256 KB per CTA, clusters of up to 8).
//
// Whole waves (the "Block Occupancy: tail effect" rule of the cs336 lecture
// 6 notes): every grid is persistent, sized at launch to the number of CTAs
// (clusters) the device holds at once, so the last wave is never a small
// fraction of the machine; rows are dealt round-robin to CTAs (clusters).
#include "kernels.h"

#include <stdint.h>

namespace rwsm {

namespace {

constexpr int64_t kWarpMaxCols = 1024;
constexpr int64_t kSliceTargetBytes = 32 * 1024;   // preferred slice (CTA path: whole row)
constexpr int kSliceStages = 2;                    // ring stages of the slice kernel
constexpr int64_t kTileRingBudgetBytes = 16 * 1024; // shared memory for the tile ring, per CTA
constexpr int64_t kClusterMaxRowBytes = 64 * 1024;  // longer rows take TWOPASS
constexpr int64_t kTwoPassBytesPerCta = 256 * 1024;      // register two-pass
// Staged two-pass (measured on GB300 over rows of 128 KB to 16 MB): 512
// consumer threads x 4 vectors (32 KB chunks); slices of about 256 KB fp32
// or 1 MB 16-bit; clusters of at most 4; ring stages by CTAs per SM.
constexpr int64_t kStreamSliceBytesF32 = 256 * 1024;
constexpr int64_t kStreamSliceBytes16 = 1024 * 1024;
constexpr int kStreamThreads = 512;
constexpr int kStreamVectors = 4;
constexpr int kStreamStagesOneCta = 6;       // 192 KB: one CTA per SM
constexpr int kStreamStagesTwoCtas = 3;      // 96 KB: two CTAs per SM
constexpr int kStreamStagesLongSlice = 4;    // fp32 slices beyond 256 KB
// A row under 96 KB on one CTA: 256 threads x 4 vectors (16 KB chunks), six
// stages (96 KB: two CTAs per SM, launched as two waves).  Measured on GB300
// against 32 KB chunks and one CTA per SM: 2730 x 12288 fp32 4832 -> 6576
// GB/s, 3947 x 8500 fp32 3440 -> 4861, 4096 x 32768 bf16 5512 -> 5863, 2048
// x 32768 bf16 5141 -> 5301 (4096 x 16384 fp32 6778 -> 6479); 96 KB rows and
// longer keep 32 KB chunks (1365 x 24576 fp32: 6626 against 5909).
constexpr int64_t kStreamShortSliceBytes = 96 * 1024;
constexpr int kStreamThreadsShort = 256;
constexpr int kStreamStagesShort = 6;
constexpr int64_t kStreamMaxClusterAuto = 4;
constexpr int64_t kTwoPassMaxCluster = 8;
constexpr int64_t kTwoPassMinSliceBytes = 64 * 1024;     // when clusters grow for few rows
constexpr int kMaxStages = 8;                       // must match row_slices.cu
constexpr int kMaxSliceThreads = 1024;
constexpr int kMinSliceThreads = 64;
constexpr int kSmemReserve = 2048;                  // static smem + slack
constexpr int64_t kTileStageBytes = 8 * 1024;      // WARP path (staged): rows per stage
constexpr int64_t kTileMaxRowsPerWarp = 16;

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

// Rows a lane holds at once in the sub-warp kernel, one vector each (must
// match warp_rows.cu).
int sub_rows_for(int vec) { return vec >= 8 ? 4 : (vec == 4 ? 8 : 16); }

// Rows held in flight per warp on the WARP path (must match warp_rows.cu).
int warp_rows_for(int e)
{
    return e >= 16 ? 1 : (16 / e > 8 ? 8 : 16 / e);
}

// 16-byte vectors a thread of the slice kernel holds at most (32 floats).
int max_vectors_per_thread(int esz) { return esz == 4 ? 8 : 4; }

// Columns one CTA of the slice kernel can hold in registers.
int64_t slice_capacity(int esz) { return int64_t{kMaxSliceThreads} * max_vectors_per_thread(esz) * (16 / esz); }

// Threads and vectors per thread for a slice of nvec 16-byte vectors: about
// 32 elements per thread (more only when 1024 threads do not suffice), at
// least 64 threads, then the smallest power-of-two vectors per thread that
// covers the slice.  Rows of 8 KB and less on 64 threads rather than 128
// (more rows in flight per SM): 43690 x 1536 bf16 4389 -> 5258 GB/s, 32768 x
// 2048 bf16 5539 -> 6453, 21845 x 1536 fp32 6165 -> 6931 on GB300.
void slice_shape(int64_t nvec, int esz, int* threads, int* nv)
{
    const int nv_target = esz == 4 ? 8 : 4;
    int64_t t = pow2_ceil(ceil_div(nvec, nv_target));
    if (t < kMinSliceThreads)
        t = kMinSliceThreads;
    if (t > kMaxSliceThreads)
        t = kMaxSliceThreads;
    int64_t v = pow2_ceil(ceil_div(nvec, t));
    if (v < 1)
        v = 1;
    *threads = static_cast<int>(t);
    *nv = static_cast<int>(v);
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
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16 && dtype != SOFTMAX_F16)
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
    const int path_in = path;
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
    const bool in_vec = aligned16(p.in, p.n_rows, p.ld_in, esz);   // 16-byte input rows
    const bool in_al = in_vec && !p.no_bulk;                        // ... and staging allowed
    const bool out_al = aligned16(p.out, p.n_rows, p.ld_out, esz);
    const int64_t row_bytes = p.n_cols * esz;
    const int64_t smem_cap = static_cast<int64_t>(dev.max_smem_per_block_optin) - kSmemReserve;
    const int max_cluster = dev.max_cluster < 1 ? 1 : (dev.max_cluster > 16 ? 16 : dev.max_cluster);

    const int64_t cap = slice_capacity(esz);
    auto slice_cols_for = [&](int cs) { return round_up(ceil_div(p.n_cols, cs), vmax); };
    // Smallest cluster (>= 2) whose slices fit the preferred size; when
    // forced, else the largest cluster if its slices fit a CTA's registers.
    auto cluster_for = [&](bool allow_big) -> int {
        for (int cs = 2; cs <= max_cluster; cs *= 2)
            if (slice_cols_for(cs) * esz <= kSliceTargetBytes)
                return cs;
        const int big = static_cast<int>(pow2_floor(max_cluster));
        if (allow_big && big >= 2 && slice_cols_for(big) <= cap &&
            slice_cols_for(big) * esz <= smem_cap)
            return big;
        return 0;
    };

    // Rows beyond 32 KB go to the staged two-pass kernel when the input
    // allows bulk copies: its deep ring and producer warp measured faster than
    // a cluster holding the row on chip from 48 KB up (e.g. 64 KB fp32 rows
    // 6.2 against 5.0 TB/s), while the second pass re-reads the row mostly
    // from L2.  Unaligned input keeps the cluster kernel up to 64 KB rows.
    if (path == SOFTMAX_PATH_AUTO) {
        if (p.n_cols <= kWarpMaxCols)
            path = SOFTMAX_PATH_WARP;
        else if (row_bytes <= kSliceTargetBytes)
            path = SOFTMAX_PATH_CTA;
        else if (!in_al && cluster_for(false) && row_bytes <= kClusterMaxRowBytes)
            path = SOFTMAX_PATH_CLUSTER;
        else
            path = SOFTMAX_PATH_TWOPASS;
    }
    const bool automatic = path_in == SOFTMAX_PATH_AUTO;

    softmax_plan_t q = {};
    q.path = path;
    q.dtype = p.dtype;
    q.cluster = 1;
    switch (path) {
    case SOFTMAX_PATH_WARP: {
        if (p.n_cols > kWarpMaxCols)
            return SOFTMAX_ERR_UNSUPPORTED;
        q.threads = 128;
        q.grid = 0;
        // 16-bit rows go through the staged tile kernel; fp32 rows measured
        // faster in the register kernel (its loads are all in flight at once).
        // 16-bit rows of at most 16 vectors take the register kernel too,
        // several rows to a warp (on GB300: 64 bf16 columns 1565 -> 3778
        // GB/s, 128 columns 2924 -> 3676; from 200 columns the tile kernel
        // is faster).
        const bool short16 = p.dtype != SOFTMAX_F32 && automatic && in_vec && out_al &&
                             p.n_cols <= 16 * vmax;
        if (in_al && (p.dtype != SOFTMAX_F32 || !automatic) && !short16) {
            // Staged tile kernel: stages of 4 * rows_per_warp rows of
            // row_pad elements (about 16 KB), about 64 KB of ring per CTA.
            const int64_t row_pad = round_up(p.n_cols, vmax);
            const int64_t row_bytes_pad = row_pad * esz;
            int64_t rpw = pow2_floor(kTileStageBytes / (4 * row_bytes_pad) > 0
                                         ? kTileStageBytes / (4 * row_bytes_pad) : 1);
            if (rpw > kTileMaxRowsPerWarp)
                rpw = kTileMaxRowsPerWarp;
            const int64_t stage_bytes = 4 * rpw * row_bytes_pad;
            int64_t stages = kTileRingBudgetBytes / stage_bytes;
            stages = stages < 1 ? 1 : (stages > kMaxStages ? kMaxStages : stages);
            q.bulk_copy = 1;
            q.vec = out_al ? vmax : 1;
            q.out_vec = q.vec;
            q.chunks = static_cast<int>(pow2_ceil(ceil_div(p.n_cols, 32 * q.vec)));
            q.rows_per_warp = static_cast<int>(rpw);
            q.lanes_per_row = 32;
            q.slice_cols = row_pad;
            q.stages = static_cast<int>(stages);
            q.smem_bytes = static_cast<int>(stages * stage_bytes);
        } else {
            q.vec = (in_vec && out_al) ? vmax : 1;
            q.out_vec = q.vec;
            q.chunks = static_cast<int>(pow2_ceil(ceil_div(p.n_cols, 32 * q.vec)));
            q.rows_per_warp = warp_rows_for(q.vec * q.chunks);
            q.lanes_per_row = 32;
            if (q.chunks == 1) {
                // Rows of at most 16 vectors: several rows side by side in a
                // warp, each on the smallest power-of-two group of lanes.
                const int64_t lanes = pow2_ceil(ceil_div(p.n_cols, q.vec));
                if (lanes < 32) {
                    q.lanes_per_row = static_cast<int>(lanes);
                    q.rows_per_warp = (32 / q.lanes_per_row) * sub_rows_for(q.vec);
                }
            }
            q.slice_cols = p.n_cols;
        }
        break;
    }
    case SOFTMAX_PATH_CTA:
    case SOFTMAX_PATH_CLUSTER: {
        int cs = 1;
        if (path == SOFTMAX_PATH_CLUSTER) {
            cs = cluster_for(true);
            if (!cs)
                return SOFTMAX_ERR_UNSUPPORTED;
        }
        const int64_t slice = slice_cols_for(cs);
        const int64_t stage_bytes = slice * esz;
        if (slice > cap || stage_bytes > smem_cap)
            return SOFTMAX_ERR_UNSUPPORTED;
        int threads = 0, nv = 0;
        slice_shape(slice / vmax, esz, &threads, &nv);
        int64_t stages = kSliceStages;
        while (stages > 1 && stages * stage_bytes > smem_cap)
            --stages;
        q.cluster = cs;
        q.slice_cols = slice;
        q.vec = in_vec ? vmax : 1;        // global input loads (staged: always 16 bytes)
        q.out_vec = out_al ? vmax : 1;
        q.bulk_copy = in_al ? 1 : 0;
        q.threads = threads;
        q.chunks = nv;
        q.stages = in_al ? static_cast<int>(stages) : 0;
        q.smem_bytes = in_al ? static_cast<int>(stages * stage_bytes) : 0;
        q.grid = 0;
        break;
    }
    case SOFTMAX_PATH_TWOPASS: {
        // Staged: 512 consumer threads stream 32 KB chunks; slices of about
        // 256 KB (fp32) or 1 MB (16-bit) on clusters of up to 4 CTAs, with a
        // 192 KB ring when one CTA holds the SM and 96-128 KB for two; rows
        // under 96 KB on one CTA stream 16 KB chunks, two CTAs per SM.  The
        // register kernel (unaligned input): about 256 KB and at least two
        // CTAs.  A single CTA when forced on short rows.
        const int64_t per_cta = in_al ? (esz == 4 ? kStreamSliceBytesF32 : kStreamSliceBytes16)
                                      : kTwoPassBytesPerCta;
        int64_t cs = pow2_ceil(ceil_div(row_bytes, per_cta));
        if (automatic && !in_al && cs < 2)
            cs = 2;
        if (automatic && cs > (in_al ? kStreamMaxClusterAuto : kTwoPassMaxCluster))
            cs = in_al ? kStreamMaxClusterAuto : kTwoPassMaxCluster;
        // Few rows: larger clusters (up to 8, slices of at least 64 KB) so
        // that more SMs take part.
        while (automatic && cs < kTwoPassMaxCluster && p.n_rows * cs < dev.sm_count &&
               row_bytes / (2 * cs) >= kTwoPassMinSliceBytes)
            cs *= 2;
        if (cs > max_cluster)
            cs = pow2_floor(max_cluster);
        q.cluster = static_cast<int>(cs);
        q.slice_cols = round_up(ceil_div(p.n_cols, cs), vmax);
        q.grid = 0;
        if (in_al) {
            // Staged: the slice streams twice through a ring of 32 KB chunks.
            q.bulk_copy = 1;
            q.vec = vmax;
            q.out_vec = out_al ? vmax : 1;
            const int64_t slice_bytes = q.slice_cols * esz;
            const bool short_slice = cs == 1 && slice_bytes < kStreamShortSliceBytes;
            q.threads = short_slice ? kStreamThreadsShort : kStreamThreads;
            q.chunks = kStreamVectors;
            int stages = short_slice ? kStreamStagesShort
                         : (esz != 4 || cs == 1) ? kStreamStagesOneCta
                         : (slice_bytes > kStreamSliceBytesF32 ? kStreamStagesLongSlice
                                                               : kStreamStagesTwoCtas);
            const int64_t chunk_bytes = int64_t{q.threads} * q.chunks * 16;
            while (stages > 1 && stages * chunk_bytes > smem_cap)
                --stages;
            q.stages = stages;
            q.smem_bytes = static_cast<int>(stages * chunk_bytes);
        } else {
            q.vec = (in_vec && out_al) ? vmax : 1;
            q.out_vec = q.vec;
            q.threads = 512;
        }
        break;
    }
    default:
        return SOFTMAX_ERR_INVALID_ARG;
    }
    *plan = q;
    return SOFTMAX_OK;
}

int check_plan(const softmax_device_desc_t& dev, const Problem& p, const softmax_plan_t& q)
{
    const int st = validate(p.in, p.out, p.n_rows, p.n_cols, p.ld_in, p.ld_out, p.dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (dev.cc_major != 10 || dev.cc_minor != 3)
        return SOFTMAX_ERR_UNSUPPORTED;
    if (q.dtype != p.dtype || q.grid < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    const int esz = esize(p.dtype);
    const int vmax = 16 / esz;
    const bool in_vec = aligned16(p.in, p.n_rows, p.ld_in, esz);
    const bool in_al = in_vec && !p.no_bulk;
    const bool out_al = aligned16(p.out, p.n_rows, p.ld_out, esz);
    const int64_t smem_cap = static_cast<int64_t>(dev.max_smem_per_block_optin) - kSmemReserve;
    const int max_cluster = dev.max_cluster < 1 ? 1 : (dev.max_cluster > 16 ? 16 : dev.max_cluster);
    auto pow2_in = [](int64_t v, int64_t lo, int64_t hi) {
        return v >= lo && v <= hi && (v & (v - 1)) == 0;
    };
    auto vec_ok = [&](int v, bool aligned) { return v == 1 || (v == vmax && aligned); };
    switch (q.path) {
    case SOFTMAX_PATH_WARP: {
        if (p.n_cols > kWarpMaxCols || q.out_vec != q.vec || q.grid > 0x7fffffff)
            return SOFTMAX_ERR_INVALID_ARG;
        if (!pow2_in(q.chunks, 1, 32) || q.vec * q.chunks > 32 ||
            int64_t{32} * q.vec * q.chunks < p.n_cols)
            return SOFTMAX_ERR_INVALID_ARG;
        const int lanes = q.lanes_per_row ? q.lanes_per_row : 32;
        if (!pow2_in(lanes, 1, 32) ||
            (lanes < 32 && (q.bulk_copy != 0 || q.chunks != 1 || int64_t{lanes} * q.vec < p.n_cols)))
            return SOFTMAX_ERR_INVALID_ARG;
        if (q.bulk_copy == 0)
            return vec_ok(q.vec, in_vec && out_al) ? SOFTMAX_OK : SOFTMAX_ERR_INVALID_ARG;
        // Staged tile kernel.
        const int64_t row_pad = round_up(p.n_cols, vmax);
        if (q.bulk_copy != 1 || !in_al || !vec_ok(q.vec, out_al) || q.slice_cols != row_pad ||
            q.rows_per_warp < 1 || q.rows_per_warp > kTileMaxRowsPerWarp ||
            q.stages < 1 || q.stages > kMaxStages || q.threads != 128)
            return SOFTMAX_ERR_INVALID_ARG;
        const int64_t stage_bytes = 4 * int64_t{q.rows_per_warp} * row_pad * esz;
        if (stage_bytes >= (1 << 20) || q.smem_bytes != q.stages * stage_bytes ||
            q.smem_bytes > smem_cap)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    }
    case SOFTMAX_PATH_CTA:
    case SOFTMAX_PATH_CLUSTER: {
        const int cs = q.cluster;
        if (q.path == SOFTMAX_PATH_CTA ? cs != 1 : !pow2_in(cs, 2, max_cluster))
            return SOFTMAX_ERR_INVALID_ARG;
        if (q.slice_cols <= 0 || q.slice_cols % vmax || q.slice_cols * cs < p.n_cols)
            return SOFTMAX_ERR_INVALID_ARG;
        if (q.bulk_copy ? q.vec != vmax : !vec_ok(q.vec, in_vec))
            return SOFTMAX_ERR_INVALID_ARG;
        if (!pow2_in(q.threads, kMinSliceThreads, kMaxSliceThreads) ||
            !pow2_in(q.chunks, 1, max_vectors_per_thread(esz)) ||
            int64_t{q.threads} * q.chunks * vmax < q.slice_cols)
            return SOFTMAX_ERR_INVALID_ARG;
        if (!vec_ok(q.out_vec, out_al) || (q.bulk_copy && !in_al) ||
            (q.bulk_copy != 0 && q.bulk_copy != 1))
            return SOFTMAX_ERR_INVALID_ARG;
        if (q.bulk_copy) {
            if (q.stages < 1 || q.stages > kMaxStages ||
                q.smem_bytes != q.stages * q.slice_cols * esz || q.smem_bytes > smem_cap)
                return SOFTMAX_ERR_INVALID_ARG;
        } else if (q.smem_bytes != 0) {
            return SOFTMAX_ERR_INVALID_ARG;
        }
        if (q.grid % cs || q.grid > 0x7fffffff)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    }
    case SOFTMAX_PATH_TWOPASS: {
        const int cs = q.cluster;
        if (!pow2_in(cs, 1, max_cluster) || q.grid % cs || q.grid > 0x7fffffff)
            return SOFTMAX_ERR_INVALID_ARG;
        if (q.slice_cols <= 0 || q.slice_cols % vmax || q.slice_cols * cs < p.n_cols ||
            (q.threads != 256 && q.threads != 512))
            return SOFTMAX_ERR_INVALID_ARG;
        if (q.bulk_copy == 0)
            return (vec_ok(q.vec, in_vec && out_al) && q.out_vec == q.vec) ? SOFTMAX_OK
                                                                             : SOFTMAX_ERR_INVALID_ARG;
        // Staged two-pass (ring of chunks of threads * chunks * 16 bytes).
        if (q.bulk_copy != 1 || !in_al || q.vec != vmax || !vec_ok(q.out_vec, out_al) ||
            (q.chunks != 2 && q.chunks != 4 && !(q.chunks == 8 && esz == 4)) ||
            q.stages < 1 || q.stages > kMaxStages ||
            q.smem_bytes != q.stages * q.threads * q.chunks * 16 || q.smem_bytes > smem_cap)
            return SOFTMAX_ERR_INVALID_ARG;
        return SOFTMAX_OK;
    }
    default:
        return SOFTMAX_ERR_INVALID_ARG;
    }
}

}  // namespace rwsm
