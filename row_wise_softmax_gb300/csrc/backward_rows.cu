// Softmax backward: dx = y * (dy - sum_j y_j dy_j) for every row, given the
// forward output y and the incoming gradient dy (the chain rule through the
// row softmax, whose Jacobian is y_j (delta_ij - y_i)).  Per element one read
// of y, one of dy and one write of dx: HBM-bound like the forward pass.
//
//   warp kernel   rows <= 1024 columns: one warp per row, y and dy in
//                 registers (VEC-wide loads at columns (c*32 + lane)*VEC), the
//                 dot product reduced with __shfl_xor, dx stored from the same
//                 registers.  Warps stride over rows of a grid of up to two
//                 resident waves.
//   CTA kernel    longer rows: one CTA of 512 threads per row.  A row of up
//                 to THREADS * NV * VEC = 8192 elements stays in registers
//                 (one HBM pass); a longer row is streamed twice, the first
//                 pass computing the dot product, the second reading y and
//                 dy again (mostly from L2) for dx.
//
// Both read y and dy through the same masked vector loads as the forward
// kernels (element loads when a row is not 16-byte aligned).
#include "common.cuh"
#include "kernels.h"

namespace rwsm {

namespace {

constexpr int kBwdWarpThreads = 128;
constexpr int kBwdGridWaves = 2;

// The first row's y and dy (its first n elements) into L2 while the
// preceding grid drains: CTAs of the first wave, resident before it ends,
// call this before griddepcontrol.wait; the loads after the wait still see
// the preceding grid's writes (L2 is the point of coherence).  Rows 16-byte
// aligned in device memory.
template <typename T>
__device__ __forceinline__ void prefetch_row_pair(const T* y, const T* dy, int64_t n)
{
    const int64_t bytes = (n * static_cast<int64_t>(sizeof(T))) & ~int64_t{15};
    for (int64_t off = 0; off < bytes; off += 32768) {
        const uint32_t b = static_cast<uint32_t>(bytes - off < 32768 ? bytes - off : 32768);
        bulk_prefetch_l2(reinterpret_cast<const char*>(y) + off, b);
        bulk_prefetch_l2(reinterpret_cast<const char*>(dy) + off, b);
    }
}

template <typename T, int VEC, int CHUNKS>
__global__ void __launch_bounds__(kBwdWarpThreads)
backward_warp_kernel(const T* y, const T* dy, T* dx, int64_t n_rows, int n_cols, int64_t ld_y,
                     int64_t ld_dy, int64_t ld_dx, int64_t prefetch_ctas)
{
    constexpr int E = VEC * CHUNKS;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    pdl_launch_dependents();
    if (lane == 0 && static_cast<int64_t>(blockIdx.x) < prefetch_ctas && warp0 < n_rows)
        prefetch_row_pair(y + warp0 * ld_y, dy + warp0 * ld_dy, n_cols);
    pdl_wait();
    for (int64_t row = warp0; row < n_rows; row += n_warps) {
        float a[E], g[E];
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c) {
            const int col = (c * 32 + lane) * VEC;
            load_vec_masked<T, VEC>(y + row * ld_y, col, n_cols, &a[c * VEC]);
            load_vec_masked<T, VEC>(dy + row * ld_dy, col, n_cols, &g[c * VEC]);
        }
        // Masked positions read -inf; they take no part in the dot product.
        float dot = 0.0f;
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c)
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const int e = c * VEC + j;
                if ((c * 32 + lane) * VEC + j < n_cols)
                    dot = fmaf(a[e], g[e], dot);
            }
        dot = warp_sum(dot);
#pragma unroll
        for (int e = 0; e < E; ++e)
            a[e] = a[e] * (g[e] - dot);
        T* d = dx + row * ld_dx;
#pragma unroll
        for (int c = 0; c < CHUNKS; ++c)
            store_vec_masked<T, VEC>(d, (c * 32 + lane) * VEC, n_cols, &a[c * VEC], 1.0f);
    }
}

// Sum of one float over the CTA; every thread gets the total.  `red` holds
// THREADS / 32 floats and is free again when the function returns.
template <int THREADS>
__device__ __forceinline__ float cta_sum(float v, float* red)
{
    constexpr int NW = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    v = warp_sum(lane < NW ? red[lane] : 0.0f);
    __syncthreads();
    return v;
}

template <typename T, int THREADS, int VEC, int NV>
__global__ void __launch_bounds__(THREADS)
backward_cta_kernel(const T* y, const T* dy, T* dx, int64_t n_rows, int64_t n_cols, int64_t ld_y,
                    int64_t ld_dy, int64_t ld_dx, int64_t prefetch_ctas)
{
    constexpr int E = NV * VEC;
    constexpr int64_t SPAN = int64_t{THREADS} * E;      // columns held in registers
    __shared__ float red[THREADS / 32];
    const int tid = threadIdx.x;
    pdl_launch_dependents();
    if (tid == 0 && static_cast<int64_t>(blockIdx.x) < prefetch_ctas && blockIdx.x < n_rows)
        prefetch_row_pair(y + blockIdx.x * ld_y, dy + blockIdx.x * ld_dy,
                          n_cols < SPAN ? n_cols : SPAN);
    pdl_wait();
    for (int64_t row = blockIdx.x; row < n_rows; row += gridDim.x) {
        const T* yr = y + row * ld_y;
        const T* gr = dy + row * ld_dy;
        T* dr = dx + row * ld_dx;
        if (n_cols <= SPAN) {
            // One pass: the row stays in registers.
            float a[E], g[E];
            float dot = 0.0f;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int64_t col = (tid + int64_t{k} * THREADS) * VEC;
                load_vec_masked<T, VEC>(yr, col, n_cols, &a[k * VEC]);
                load_vec_masked<T, VEC>(gr, col, n_cols, &g[k * VEC]);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (col + j < n_cols)
                        dot = fmaf(a[k * VEC + j], g[k * VEC + j], dot);
            }
            dot = cta_sum<THREADS>(dot, red);
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int64_t col = (tid + int64_t{k} * THREADS) * VEC;
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    a[k * VEC + j] = a[k * VEC + j] * (g[k * VEC + j] - dot);
                store_vec_masked<T, VEC>(dr, col, n_cols, &a[k * VEC], 1.0f);
            }
        } else {
            // Two passes over chunks of THREADS * VEC columns: the dot
            // product, then dx from a second read (served mostly by L2).
            float dot = 0.0f;
            for (int64_t c0 = 0; c0 < n_cols; c0 += int64_t{THREADS} * VEC) {
                const int64_t col = c0 + int64_t{tid} * VEC;
                float a[VEC], g[VEC];
                load_vec_masked<T, VEC>(yr, col, n_cols, a);
                load_vec_masked<T, VEC>(gr, col, n_cols, g);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (col + j < n_cols)
                        dot = fmaf(a[j], g[j], dot);
            }
            dot = cta_sum<THREADS>(dot, red);
            for (int64_t c0 = 0; c0 < n_cols; c0 += int64_t{THREADS} * VEC) {
                const int64_t col = c0 + int64_t{tid} * VEC;
                float a[VEC], g[VEC];
                load_vec_masked<T, VEC>(yr, col, n_cols, a);
                load_vec_masked<T, VEC>(gr, col, n_cols, g);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    a[j] = a[j] * (g[j] - dot);
                store_vec_masked<T, VEC>(dr, col, n_cols, a, 1.0f);
            }
        }
    }
}

// Up to `waves` times the resident CTAs, at most one unit (row or warp's
// row) each: a CTA that finishes early is replaced by a fresh one, so the
// last rows spread over every SM.  Two waves measured best on GB300: 4096 x
// 4096 fp32 5499 -> 5674 GB/s, 32768 x 1024 bf16 5450 -> 5593 (one to six
// waves tried).
template <typename K>
int64_t persistent_grid(K* k, int threads, int64_t units, int waves, int64_t* resident_out)
{
    const int resident = resident_ctas(reinterpret_cast<const void*>(k), threads, 0);
    *resident_out = resident;
    const int64_t cap = static_cast<int64_t>(waves) * resident;
    int64_t g = units < cap ? units : cap;
    return g < 1 ? 1 : g;
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K* k, int64_t grid, int threads, cudaStream_t s, Args... args)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, 1));
    const cudaError_t err = cudaLaunchKernelEx(&cfg, k, args...);
    note_launch();
    return err;
}

template <typename T, int VEC>
cudaError_t launch_warp(const BackwardProblem& p, cudaStream_t s)
{
    // CHUNKS: 32-lane vector chunks to cover the row (at most 1024 columns).
    const int64_t per_chunk = 32 * VEC;
    const int64_t chunks = (p.n_cols + per_chunk - 1) / per_chunk;
    const int64_t rows_per_cta = kBwdWarpThreads / 32;
    auto go = [&](auto* k) {
        int64_t resident = 0;
        const int64_t grid = persistent_grid(k, kBwdWarpThreads, (p.n_rows + rows_per_cta - 1) /
                                                                     rows_per_cta, kBwdGridWaves,
                                             &resident);
        return launch_pdl(k, grid, kBwdWarpThreads, s, static_cast<const T*>(p.y),
                          static_cast<const T*>(p.dy), static_cast<T*>(p.dx), p.n_rows,
                          static_cast<int>(p.n_cols), p.ld_y, p.ld_dy, p.ld_dx,
                          VEC > 1 ? resident : int64_t{0});
    };
    if (chunks <= 1) return go(backward_warp_kernel<T, VEC, 1>);
    if (chunks <= 2) return go(backward_warp_kernel<T, VEC, 2>);
    if (chunks <= 4) return go(backward_warp_kernel<T, VEC, 4>);
    if constexpr (VEC * 8 <= 32)
        if (chunks <= 8) return go(backward_warp_kernel<T, VEC, 8>);
    if constexpr (VEC * 16 <= 32)
        if (chunks <= 16) return go(backward_warp_kernel<T, VEC, 16>);
    if constexpr (VEC * 32 <= 32)
        if (chunks <= 32) return go(backward_warp_kernel<T, VEC, 32>);
    return cudaErrorInvalidValue;
}

template <typename T, int VEC>
cudaError_t launch_cta(const BackwardProblem& p, cudaStream_t s)
{
    // 512 threads x 16 elements: 4 CTAs of 16 warps per SM (a row in flight
    // per CTA, so resident warps hide the load latency).
    constexpr int THREADS = 512;
    constexpr int NV = 16 / VEC > 8 ? 8 : 16 / VEC;           // up to 16 elements a thread
    auto* k = backward_cta_kernel<T, THREADS, VEC, NV>;
    int64_t resident = 0;
    const int64_t grid = persistent_grid(k, THREADS, p.n_rows, kBwdGridWaves, &resident);
    return launch_pdl(k, grid, THREADS, s, static_cast<const T*>(p.y),
                      static_cast<const T*>(p.dy), static_cast<T*>(p.dx), p.n_rows, p.n_cols,
                      p.ld_y, p.ld_dy, p.ld_dx, VEC > 1 ? resident : int64_t{0});
}

template <typename T>
cudaError_t launch_typed(const BackwardProblem& p, bool vec, cudaStream_t s)
{
    constexpr int V = Elem<T>::kVec16;
    if (p.n_cols <= kBackwardWarpMaxCols)
        return vec ? launch_warp<T, V>(p, s) : launch_warp<T, 1>(p, s);
    return vec ? launch_cta<T, V>(p, s) : launch_cta<T, 1>(p, s);
}

}  // namespace

cudaError_t launch_backward_rows(const BackwardProblem& p, bool vec, cudaStream_t s)
{
    if (p.dtype == SOFTMAX_F32)
        return launch_typed<float>(p, vec, s);
    if (p.dtype == SOFTMAX_BF16)
        return launch_typed<BF16Bits>(p, vec, s);
    return launch_typed<F16Bits>(p, vec, s);
}

}  // namespace rwsm
