// Softmax over strided rows: element c of row r at r * row_stride +
// c * col_stride.  The cs336 lecture 6 notes ("Level 1: Softmax") take a
// column-wise softmax by changing only the strides; here the two layouts get
// kernels of their own because the memory access pattern, not the
// arithmetic, is what changes.
//
//   columns kernel   unit row stride (the softmax runs down the columns of a
//                    row-major matrix): adjacent softmax rows are adjacent in
//                    memory.  A CTA stages a tile of W adjacent softmax rows
//                    (128 bytes of every memory row) for its share of the
//                    memory rows in shared memory with cp.async, reduces each
//                    column there (max, then the sum of exp_biased), and writes
//                    the result from the same tile: one HBM read and one write
//                    per element, every access a full 128-byte segment.
//                    Longer columns are split over the CTAs of a cluster, which
//                    combine their per-column maxima and sums through
//                    distributed shared memory.
//   gather kernel    any other strides: one warp per softmax row, each lane an
//                    online (m, l) over every 32nd element, merged across the
//                    warp, then a second pass writing the outputs.  Correct for
//                    every layout, not tuned.
#include "common.cuh"
#include "kernels.h"

#include <atomic>

namespace rwsm {

namespace {

constexpr int kColThreads = 256;
constexpr int kColGroup = 8;              // lanes per 128-byte memory-row segment
constexpr int kColAlign = 128;

template <typename T>
__device__ __forceinline__ float to_f32(const T* p)
{
    if constexpr (sizeof(T) == 4)
        return *reinterpret_cast<const float*>(p);
    else
        return Elem<T>::widen(*reinterpret_cast<const unsigned short*>(p));
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Combine column c's value over the CTAs of the cluster through distributed
// shared memory (IS_MAX: maximum, else sum).  `mine` holds this CTA's values;
// the caller's cluster barrier has made every CTA's values visible.  A value
// is rewritten only after at least one more cluster barrier, which every peer
// reaches after its reads.
template <bool IS_MAX>
__device__ __forceinline__ float cluster_column(float* mine, int c, int cs)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    float r = IS_MAX ? kNegInf : 0.0f;
    for (int k = 0; k < cs; ++k) {
        const float v = *cluster.map_shared_rank(&mine[c], k);
        r = IS_MAX ? fmaxf(r, v) : r + v;
    }
    return r;
}

template <typename T>
__global__ void __launch_bounds__(kColThreads)
columns_kernel(const T* in, T* out, int64_t n_s, int64_t n_l, int64_t ld_in, int64_t ld_out,
               int lc, int cs, int vec_in, int vec_out)
{
    constexpr int VEC = Elem<T>::kVec16;
    constexpr int W = kColGroup * VEC;            // softmax rows per tile (128 bytes)
    constexpr int NSLOT = kColThreads / W;        // memory-row slots per column
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ float red[NSLOT][W];
    __shared__ float part[2][W];                  // this CTA's column max / sum
    __shared__ float col_m[W], col_inv[W];

    T* tile = reinterpret_cast<T*>((reinterpret_cast<uintptr_t>(smem_raw) + (kColAlign - 1)) &
                                   ~static_cast<uintptr_t>(kColAlign - 1));
    const int tid = threadIdx.x;
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;
    const int64_t l0 = static_cast<int64_t>(rank) * lc;
    int lv = static_cast<int>(n_l - l0 < lc ? n_l - l0 : lc);   // memory rows held here
    lv = lv < 0 ? 0 : lv;
    const int64_t n_tiles = (n_s + W - 1) / W;
    const int c = tid % W, slot = tid / W;

    if (cs == 1)
        pdl_launch_dependents();
    pdl_wait();
    for (int64_t t = cluster_id; t < n_tiles; t += n_clusters) {
        const int64_t s0 = t * W;
        // ---- stage the tile: memory row l, 16-byte group g
        for (int i = tid; i < lv * kColGroup; i += kColThreads) {
            const int l = i / kColGroup, g = i % kColGroup;
            const int64_t s = s0 + int64_t{g} * VEC;
            T* dst = tile + l * W + g * VEC;
            const T* src = in + (l0 + l) * ld_in + s;
            if (vec_in && s + VEC <= n_s) {
                cp_async16(dst, src);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    if constexpr (sizeof(T) == 4)
                        reinterpret_cast<float*>(dst)[j] = s + j < n_s ? __ldg(
                            reinterpret_cast<const float*>(src) + j) : 0.0f;
                    else
                        reinterpret_cast<unsigned short*>(dst)[j] = s + j < n_s ? __ldg(
                            reinterpret_cast<const unsigned short*>(src) + j) : 0;
                }
            }
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- column maximum: slots, then CTAs
        float m = kNegInf;
        for (int l = slot; l < lv; l += NSLOT)
            m = fmaxf(m, to_f32(tile + l * W + c));
        red[slot][c] = m;
        __syncthreads();
        if (tid < W) {
            float mm = kNegInf;
#pragma unroll
            for (int k = 0; k < NSLOT; ++k)
                mm = fmaxf(mm, red[k][tid]);
            part[0][tid] = mm;
        }
        if (cs > 1) {
            cooperative_groups::this_cluster().sync();
            if (tid < W)
                col_m[tid] = cluster_column<true>(part[0], tid, cs);
        } else {
            __syncthreads();
            if (tid < W)
                col_m[tid] = part[0][tid];
        }
        __syncthreads();

        // ---- sum of exp_biased(x - max) (the 2^64 bias cancels in the ratio)
        const float mc = col_m[c];
        float sum = 0.0f;
        for (int l = slot; l < lv; l += NSLOT)
            sum += exp_biased(to_f32(tile + l * W + c) - mc, kLog2e);
        red[slot][c] = sum;
        __syncthreads();
        if (tid < W) {
            float ss = 0.0f;
#pragma unroll
            for (int k = 0; k < NSLOT; ++k)
                ss += red[k][tid];
            part[1][tid] = ss;
        }
        if (cs > 1) {
            cooperative_groups::this_cluster().sync();
            if (tid < W)
                col_inv[tid] = 1.0f / cluster_column<false>(part[1], tid, cs);
        } else {
            __syncthreads();
            if (tid < W)
                col_inv[tid] = 1.0f / part[1][tid];
        }
        __syncthreads();

        // ---- write: the same 128-byte segments
        for (int i = tid; i < lv * kColGroup; i += kColThreads) {
            const int l = i / kColGroup, g = i % kColGroup;
            const int64_t s = s0 + int64_t{g} * VEC;
            float y[VEC];
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                y[j] = exp_biased(to_f32(tile + l * W + g * VEC + j) - col_m[g * VEC + j], kLog2e) *
                       col_inv[g * VEC + j];
            T* dst = out + (l0 + l) * ld_out + s;
            if (vec_out && s + VEC <= n_s) {
                store_vec<T, VEC>(dst, y, 1.0f);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (s + j < n_s)
                        Elem<T>::store1(dst + j, y[j]);
            }
        }
        __syncthreads();          // the tile and col_* are rewritten by the next tile
    }
    if (cs > 1) {
        pdl_launch_dependents();
        cooperative_groups::this_cluster().sync();     // peers may still read `part`
    }
}

// One warp per softmax row, any strides: per-lane online (m, l), warp merge,
// then a second pass writing exp(x - m) / l.
template <typename T>
__global__ void __launch_bounds__(128)
gather_kernel(const T* in, T* out, int64_t n_rows, int64_t n_cols, int64_t in_rs, int64_t in_cs,
              int64_t out_rs, int64_t out_cs)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t r = warp0; r < n_rows; r += n_warps) {
        const T* src = in + r * in_rs;
        float m = kNegInf, l = 0.0f;
        for (int64_t j = lane; j < n_cols; j += 32) {
            const float x = Elem<T>::load1(src + j * in_cs);
            const float mn = fmaxf(m, x);
            const float ref = (mn == kNegInf) ? 0.0f : mn;
            l = l * exp_ftz(m - ref, kLog2e) + exp_biased(x - ref, kLog2e);
            m = mn;
        }
        warp_ml_merge(m, l, kLog2e);
        const float inv = 1.0f / l;
        T* dst = out + r * out_rs;
        for (int64_t j = lane; j < n_cols; j += 32)
            Elem<T>::store1(dst + j * out_cs,
                            exp_biased(Elem<T>::load1(src + j * in_cs) - m, kLog2e) * inv);
    }
}

template <typename K, typename... Args>
cudaError_t launch(K* k, int64_t grid, int threads, int smem, int cs, cudaStream_t s,
                   Args... args)
{
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, cs));
    const cudaError_t err = cudaLaunchKernelEx(&cfg, k, args...);
    note_launch();
    return err;
}

constexpr int kMaxDevices = 64;

template <typename T>
cudaError_t launch_columns(const StridedProblem& p, const ColumnsShape& sh, cudaStream_t s)
{
    auto* k = columns_kernel<T>;
    static std::atomic<int> smem_set[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int smem = sh.smem_bytes + kColAlign;
    if (smem_set[dev].load() < smem) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess)
            return err;
        cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess)
            return err;
        smem_set[dev].store(smem);
    }
    int64_t clusters = 0;
    if (sh.cluster > 1) {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(static_cast<unsigned>(sh.cluster), 1, 1);
        q.blockDim = dim3(kColThreads, 1, 1);
        q.dynamicSmemBytes = static_cast<size_t>(smem);
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = static_cast<unsigned>(sh.cluster);
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        q.attrs = a;
        q.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, k, &q) != cudaSuccess) {
            cudaGetLastError();
            active = 0;
        }
        clusters = active;
    } else {
        clusters = resident_ctas(reinterpret_cast<const void*>(k), kColThreads, smem);
    }
    if (clusters < 1)
        clusters = 1;
    clusters = balanced_grid(sh.tiles, clusters, sh.cluster == 1 ? sm_count_current() : 0);
    return launch(k, clusters * sh.cluster, kColThreads, smem, sh.cluster, s,
                  static_cast<const T*>(p.in), static_cast<T*>(p.out), p.n_rows, p.n_cols,
                  p.in_col_stride, p.out_col_stride, sh.rows_per_cta, sh.cluster,
                  sh.vec_in ? 1 : 0, sh.vec_out ? 1 : 0);
}

template <typename T>
cudaError_t launch_gather(const StridedProblem& p, cudaStream_t s)
{
    auto* k = gather_kernel<T>;
    const int resident = resident_ctas(reinterpret_cast<const void*>(k), 128, 0);
    int64_t grid = (p.n_rows + 3) / 4;
    grid = grid < resident ? grid : resident;
    return launch(k, grid < 1 ? 1 : grid, 128, 0, 1, s, static_cast<const T*>(p.in),
                  static_cast<T*>(p.out), p.n_rows, p.n_cols, p.in_row_stride, p.in_col_stride,
                  p.out_row_stride, p.out_col_stride);
}

}  // namespace

ColumnsShape columns_shape(const StridedProblem& p, int max_smem_per_block)
{
    ColumnsShape sh{};
    const int esz = p.dtype == SOFTMAX_F32 ? 4 : 2;
    const int64_t row_bytes = 128;                      // one tile row: W elements
    const int64_t w = row_bytes / esz;
    // Memory rows per CTA: about 64 KB of tile (several CTAs per SM), more
    // CTAs per cluster for longer columns, up to 16; then larger tiles.
    int64_t cs = (p.n_cols + kColumnsRowsPerCta - 1) / kColumnsRowsPerCta;
    if (cs < 1)
        cs = 1;
    if (cs > kColumnsMaxCluster)
        cs = kColumnsMaxCluster;
    const int64_t rows = (p.n_cols + cs - 1) / cs;
    const int64_t smem = rows * row_bytes;
    if (smem + kColAlign > max_smem_per_block - 2048)
        return sh;                                       // does not fit: ok = false
    sh.ok = true;
    sh.cluster = static_cast<int>(cs);
    sh.rows_per_cta = static_cast<int>(rows);
    sh.smem_bytes = static_cast<int>(smem);
    sh.tiles = (p.n_rows + w - 1) / w;
    auto al = [&](const void* q, int64_t ld) {
        return reinterpret_cast<uintptr_t>(q) % 16 == 0 && (ld * esz) % 16 == 0;
    };
    sh.vec_in = al(p.in, p.in_col_stride);
    sh.vec_out = al(p.out, p.out_col_stride);
    return sh;
}

cudaError_t launch_strided(const StridedProblem& p, const ColumnsShape& sh, cudaStream_t s)
{
    if (sh.ok && sh.stream)
        return launch_columns_stream(p, sh, s);
    if (sh.ok) {
        if (p.dtype == SOFTMAX_F32) return launch_columns<float>(p, sh, s);
        if (p.dtype == SOFTMAX_BF16) return launch_columns<BF16Bits>(p, sh, s);
        return launch_columns<F16Bits>(p, sh, s);
    }
    if (p.dtype == SOFTMAX_F32) return launch_gather<float>(p, s);
    if (p.dtype == SOFTMAX_BF16) return launch_gather<BF16Bits>(p, s);
    return launch_gather<F16Bits>(p, s);
}

}  // namespace rwsm
