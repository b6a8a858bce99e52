// WARP path: one warp owns whole rows of up to 1024 columns, held in
// registers.  Each lane loads VEC-wide vectors at columns (c*32 + lane)*VEC,
// so every load and store instruction of the warp covers 32*VEC consecutive
// elements of a row (coalesced).  A warp works on a group of ROWS rows at a
// time and is software-pipelined: the loads of its next group are issued
// before the current group is reduced and stored, so each warp keeps a group
// of rows in flight from HBM while it computes.
//
// Per row: m = max (lanes, then __shfl_xor tree), e = exp(x - m) in place,
// l = sum (lanes, then tree), y = e * (1/l).  This is the fused softmax of
// "Triton: write CUDA-grade GPU operators in Python", example 2, with one row
// per warp instead of one row per program, and the "-inf padding contributes
// 0" rule of the cs336 lecture 6 notes, "Level 1: Softmax", for the masked
// tail.
//
// The grid holds up to four times the resident CTAs, each warp striding over
// row groups: a CTA that finishes early is replaced by a fresh one, so the
// last rows are spread over every SM instead of a few finishing alone
// (lecture 6 notes, "Block Occupancy: tail effect").
//
// Rows of at most 16 vectors leave most lanes of a warp idle, so the sub-warp
// kernel gives each row LPR lanes (a power of two) and a warp 32 / LPR rows
// side by side: lane l takes row l / LPR of a slot and the vector at column
// (l % LPR) * VEC, the maximum and the sum reduce with __shfl_xor within
// those LPR lanes, and consecutive slots of rows sit in the same registers
// (ROWS rows a lane) so that their loads are in flight together.
#include "common.cuh"
#include "kernels.h"

namespace rwsm {

constexpr int kWarpPathThreads = 128;
constexpr int kWarpGridWaves = 4;       // CTAs launched per resident CTA (at most)

template <typename T, int VEC, int CHUNKS, int ROWS, bool OPTS>
__device__ __forceinline__ void load_group(const T* in, int64_t g, int64_t n_rows, int n_cols,
                                           int64_t ld_in, const LogitsArg lg, int lane,
                                           float (&v)[ROWS][VEC * CHUNKS])
{
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int64_t row = g * ROWS + r;
        if (row < n_rows) {
            const T* src = in + row * ld_in;
            const int64_t lim = kept_cols<OPTS>(lg, row, n_cols);   // masked columns: not read
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c)
                load_vec_masked<T, VEC, OPTS && (VEC > 1)>(src, (c * 32 + lane) * VEC, lim,
                                                          &v[r][c * VEC]);
        } else {
#pragma unroll
            for (int k = 0; k < VEC * CHUNKS; ++k)
                v[r][k] = kNegInf;
        }
    }
}

template <typename T, int VEC, int CHUNKS, int ROWS>
__device__ __forceinline__ void softmax_group(T* out, int64_t g, int64_t n_rows, int n_cols,
                                              int64_t ld_out, float k, int lane,
                                              float (&v)[ROWS][VEC * CHUNKS])
{
    constexpr int E = VEC * CHUNKS;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int64_t row = g * ROWS + r;
        float m = kNegInf;
#pragma unroll
        for (int e = 0; e < E; ++e)
            m = fmaxf(m, v[r][e]);
        m = warp_max_redux(m);
        float l = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            v[r][e] = exp_biased(v[r][e] - m, k);
            l += v[r][e];
        }
        l = warp_sum(l);
        const float inv = 1.0f / l;
        if (row < n_rows) {
            T* dst = out + row * ld_out;
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c)
                store_vec_masked<T, VEC>(dst, (c * 32 + lane) * VEC, n_cols, &v[r][c * VEC], inv);
        }
    }
}

template <typename T, int VEC, int CHUNKS, int ROWS, bool OPTS>
__global__ void __launch_bounds__(kWarpPathThreads)
warp_rows_kernel(const T* in, T* out, int64_t n_rows, int n_cols,
                 int64_t ld_in, int64_t ld_out, int64_t prefetch_ctas, LogitsArg lg)
{
    constexpr int E = VEC * CHUNKS;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t n_groups = (n_rows + ROWS - 1) / ROWS;
    pdl_launch_dependents();
    // CTAs of the first wave (resident before the preceding grid ends) bring
    // their first group's rows into L2 while it drains: the loads after
    // griddepcontrol.wait still see its writes (L2 is the point of
    // coherence).  prefetch_ctas is 0 unless the rows are 16-byte aligned
    // device memory.
    if (lane == 0 && static_cast<int64_t>(blockIdx.x) < prefetch_ctas && warp0 < n_groups) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int64_t row = warp0 * ROWS + r;
            if (row < n_rows) {
                const uint32_t bytes =
                    static_cast<uint32_t>(kept_cols<OPTS>(lg, row, n_cols) * sizeof(T)) & ~15u;
                if (bytes)
                    bulk_prefetch_l2(in + row * ld_in, bytes);
            }
        }
    }
    pdl_wait();
    if (warp0 >= n_groups)
        return;

    // Two register buffers, A and B, alternate: while one group is reduced
    // and stored, the loads of the next group are already in flight.
    float a[ROWS][E], b[ROWS][E];
    int64_t g = warp0;
    load_group<T, VEC, CHUNKS, ROWS, OPTS>(in, g, n_rows, n_cols, ld_in, lg, lane, a);
    while (true) {
        const int64_t gb = g + n_warps;
        if (gb < n_groups)
            load_group<T, VEC, CHUNKS, ROWS, OPTS>(in, gb, n_rows, n_cols, ld_in, lg, lane, b);
        softmax_group<T, VEC, CHUNKS, ROWS>(out, g, n_rows, n_cols, ld_out, (OPTS ? lg.k : kLog2e), lane, a);
        if (gb >= n_groups)
            break;
        const int64_t ga = gb + n_warps;
        if (ga < n_groups)
            load_group<T, VEC, CHUNKS, ROWS, OPTS>(in, ga, n_rows, n_cols, ld_in, lg, lane, a);
        softmax_group<T, VEC, CHUNKS, ROWS>(out, gb, n_rows, n_cols, ld_out, (OPTS ? lg.k : kLog2e), lane, b);
        if (ga >= n_groups)
            break;
        g = ga;
    }
}

// Maximum and sum over the LPR lanes of a row group (aligned groups: every
// xor offset below LPR stays inside the group).
template <int LPR>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int LPR>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T, int VEC, int LPR, int ROWS, bool OPTS>
__global__ void __launch_bounds__(kWarpPathThreads)
warp_sub_rows_kernel(const T* in, T* out, int64_t n_rows, int n_cols, int64_t ld_in,
                     int64_t ld_out, int64_t prefetch_ctas, LogitsArg lg)
{
    constexpr int RPS = 32 / LPR;                         // rows side by side in a warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;                           // this lane's row of a slot
    const int col = (lane % LPR) * VEC;                   // this lane's first column
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t group_rows = int64_t{RPS} * ROWS;
    const int64_t n_groups = (n_rows + group_rows - 1) / group_rows;
    pdl_launch_dependents();
    // First wave: the first group's rows into L2 while the preceding grid
    // drains (prefetch_ctas is 0 unless the rows are packed, 16-byte aligned
    // device memory, so the group is one span).
    if (lane == 0 && static_cast<int64_t>(blockIdx.x) < prefetch_ctas && warp0 < n_groups) {
        const int64_t r0 = warp0 * group_rows;
        const int64_t nr = n_rows - r0 < group_rows ? n_rows - r0 : group_rows;
        const int64_t bytes = (nr * ld_in * static_cast<int64_t>(sizeof(T))) & ~int64_t{15};
        for (int64_t off = 0; off < bytes; off += 32768)
            bulk_prefetch_l2(reinterpret_cast<const char*>(in + r0 * ld_in) + off,
                             static_cast<uint32_t>(bytes - off < 32768 ? bytes - off : 32768));
    }
    pdl_wait();
    const float k = OPTS ? lg.k : kLog2e;
    for (int64_t g = warp0; g < n_groups; g += n_warps) {
        float v[ROWS][VEC];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int64_t row = g * group_rows + r * RPS + sub;
            if (row < n_rows) {
                const int64_t lim = kept_cols<OPTS>(lg, row, n_cols);   // masked columns: not read
                load_vec_masked<T, VEC, OPTS && (VEC > 1)>(in + row * ld_in, col, lim, v[r]);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    v[r][j] = kNegInf;
            }
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int64_t row = g * group_rows + r * RPS + sub;
            float m = kNegInf;
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                m = fmaxf(m, v[r][j]);
            m = group_max<LPR>(m);
            float l = 0.0f;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                v[r][j] = exp_biased(v[r][j] - m, k);
                l += v[r][j];
            }
            l = group_sum<LPR>(l);
            const float inv = 1.0f / l;
            if (row < n_rows)
                store_vec_masked<T, VEC>(out + row * ld_out, col, n_cols, v[r], inv);
        }
    }
}

// Rows kept in flight per warp: about 16 elements per lane in total.
template <int E>
constexpr int rows_for()
{
    return E >= 16 ? 1 : (16 / E > 8 ? 8 : 16 / E);
}

template <typename T, int VEC, int CHUNKS, bool OPTS>
static cudaError_t launch_opts(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    constexpr int ROWS = rows_for<VEC * CHUNKS>();
    auto* k = warp_rows_kernel<T, VEC, CHUNKS, ROWS, OPTS>;
    const int64_t groups = (p.n_rows + ROWS - 1) / ROWS;
    const int warps_per_cta = kWarpPathThreads / 32;
    int64_t want = (groups + warps_per_cta - 1) / warps_per_cta;
    int64_t grid = plan.grid;
    const int resident = resident_ctas(reinterpret_cast<const void*>(k), kWarpPathThreads, 0);
    const size_t esz = p.dtype == SOFTMAX_F32 ? 4 : 2;
    const bool aligned_device = !p.no_bulk && reinterpret_cast<uintptr_t>(p.in) % 16 == 0 &&
                                (static_cast<size_t>(p.ld_in) * esz) % 16 == 0;
    if (grid <= 0) {
        // Four times the resident CTAs (at most one row group per warp): CTAs
        // that finish early are replaced by fresh ones whose loads start at
        // once, so the last rows are spread over every SM.  Measured on
        // GB300 against one resident wave: 262144 x 127 fp32 5935 -> 6547,
        // 65536 x 512 5941 -> 6717, 32768 x 1000 5902 -> 6697 GB/s.
        const int64_t cap = int64_t{kWarpGridWaves} * resident;
        grid = want < cap ? want : cap;
    }
    if (grid < 1)
        grid = 1;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kWarpPathThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, 1));
    const cudaError_t err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in),
                                               static_cast<T*>(p.out), p.n_rows,
                                               static_cast<int>(p.n_cols), p.ld_in, p.ld_out,
                                               aligned_device ? int64_t{resident} : int64_t{0},
                                               logits_of(p));
    note_launch();
    return err;
}

// Rows a lane holds in the sub-warp kernel: 32 values for 16-bit vectors, 32
// for fp32 vectors, 16 single elements (must match plan.cpp).
template <int VEC>
constexpr int sub_rows()
{
    return VEC >= 8 ? 4 : (VEC == 4 ? 8 : 16);
}

template <typename T, int VEC, int LPR, bool OPTS>
static cudaError_t launch_sub_opts(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    constexpr int ROWS = sub_rows<VEC>();
    auto* k = warp_sub_rows_kernel<T, VEC, LPR, ROWS, OPTS>;
    const int64_t group_rows = int64_t{32 / LPR} * ROWS;
    const int64_t groups = (p.n_rows + group_rows - 1) / group_rows;
    const int warps_per_cta = kWarpPathThreads / 32;
    const int64_t want = (groups + warps_per_cta - 1) / warps_per_cta;
    const int resident = resident_ctas(reinterpret_cast<const void*>(k), kWarpPathThreads, 0);
    int64_t grid = plan.grid;
    if (grid <= 0) {
        const int64_t cap = int64_t{kWarpGridWaves} * resident;    // as the full-warp kernel
        grid = want < cap ? want : cap;
    }
    if (grid < 1)
        grid = 1;
    const size_t esz = p.dtype == SOFTMAX_F32 ? 4 : 2;
    const bool packed = !p.no_bulk && !has_options(p) && p.ld_in == p.n_cols &&
                        reinterpret_cast<uintptr_t>(p.in) % 16 == 0 &&
                        (static_cast<size_t>(p.ld_in) * esz) % 16 == 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kWarpPathThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, 1));
    const cudaError_t err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in),
                                               static_cast<T*>(p.out), p.n_rows,
                                               static_cast<int>(p.n_cols), p.ld_in, p.ld_out,
                                               packed ? int64_t{resident} : int64_t{0},
                                               logits_of(p));
    note_launch();
    return err;
}

template <typename T, int VEC, int LPR>
static cudaError_t launch_sub(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    return has_options(p) ? launch_sub_opts<T, VEC, LPR, true>(p, plan, s)
                    : launch_sub_opts<T, VEC, LPR, false>(p, plan, s);
}

template <typename T, int VEC>
static cudaError_t launch_lanes(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    switch (plan.lanes_per_row) {
    case 1: return launch_sub<T, VEC, 1>(p, plan, s);
    case 2: return launch_sub<T, VEC, 2>(p, plan, s);
    case 4: return launch_sub<T, VEC, 4>(p, plan, s);
    case 8: return launch_sub<T, VEC, 8>(p, plan, s);
    case 16: return launch_sub<T, VEC, 16>(p, plan, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T, int VEC, int CHUNKS>
static cudaError_t launch_one(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    return has_options(p) ? launch_opts<T, VEC, CHUNKS, true>(p, plan, s)
                    : launch_opts<T, VEC, CHUNKS, false>(p, plan, s);
}

template <typename T, int VEC>
static cudaError_t launch_vec(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (plan.lanes_per_row > 0 && plan.lanes_per_row < 32)
        return plan.chunks == 1 ? launch_lanes<T, VEC>(p, plan, s) : cudaErrorInvalidValue;
    switch (plan.chunks) {
    case 1: return launch_one<T, VEC, 1>(p, plan, s);
    case 2: return launch_one<T, VEC, 2>(p, plan, s);
    case 4: return launch_one<T, VEC, 4>(p, plan, s);
    case 8:
        if constexpr (VEC * 8 <= 32) return launch_one<T, VEC, 8>(p, plan, s);
        break;
    case 16:
        if constexpr (VEC * 16 <= 32) return launch_one<T, VEC, 16>(p, plan, s);
        break;
    case 32:
        if constexpr (VEC * 32 <= 32) return launch_one<T, VEC, 32>(p, plan, s);
        break;
    default:
        break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_warp_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (p.dtype == SOFTMAX_F32) {
        if (plan.vec == 4) return launch_vec<float, 4>(p, plan, s);
        if (plan.vec == 1) return launch_vec<float, 1>(p, plan, s);
    } else if (p.dtype == SOFTMAX_BF16) {
        if (plan.vec == 8) return launch_vec<BF16Bits, 8>(p, plan, s);
        if (plan.vec == 1) return launch_vec<BF16Bits, 1>(p, plan, s);
    } else {
        if (plan.vec == 8) return launch_vec<F16Bits, 8>(p, plan, s);
        if (plan.vec == 1) return launch_vec<F16Bits, 1>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rwsm
