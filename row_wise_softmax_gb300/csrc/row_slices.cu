// CTA and CLUSTER paths: a row (CTA path, cs == 1) or a slice of a row
// (CLUSTER path, cs CTAs per row) is staged in shared memory, read from HBM
// exactly once.
//
//   stage   one elected thread starts cp.async.bulk copies of the CTA's slice
//           (global -> shared, completing on an mbarrier); a ragged tail of
//           fewer than 16 bytes is loaded by plain loads.  Without 16-byte
//           alignment every thread copies elements instead.
//   pass A  each thread walks its shared-memory vectors in batches and keeps
//           an online (m, l) partial: m_new = max(m, batch max),
//           l = l * e^(m - m_new) + sum e^(x - m_new) — the running-max
//           rescale of "Triton GPU programming deep dive", section 3.3, here
//           over slices of one row instead of key blocks.
//   merge   (m, l) partials are merged across the warp (__shfl_xor), the CTA
//           (shared memory) and, for cs > 1, the cluster: each CTA publishes
//           its partial, a cluster barrier orders the writes, and every warp
//           reads the cs partials through distributed shared memory.
//   pass B  y = e^(x - M) * (1/L) from shared memory, stored to HBM with
//           16-byte vector stores when the output rows are 16-byte aligned.
//
// Tiling a row too long for one block and carrying an accumulator across the
// tiles is the "Level 2: Row Sum (tiling)" pattern of the cs336 lecture 6
// notes; the slices of one row live on several SMs at once, so the row is
// read once and written once however long it is (up to the cluster's
// shared memory).  Rows are independent (lecture 6, "Level 1: Softmax"),
// so CTAs for different rows never communicate.
#include "common.cuh"
#include "kernels.h"

#include <atomic>
#include <mutex>

namespace rwsm {

__device__ unsigned g_error_row_slices = 0;

constexpr uint32_t kBulkChunkBytes = 32768;
constexpr int kBatch = 4;          // shared-memory vectors per thread per pass-A step

template <typename T>
__device__ __forceinline__ void copy_elem(T* dst, const T* src)
{
    if constexpr (sizeof(T) == 4)
        *reinterpret_cast<float*>(dst) = __ldg(reinterpret_cast<const float*>(src));
    else
        *reinterpret_cast<unsigned short*>(dst) = __ldg(reinterpret_cast<const unsigned short*>(src));
}

template <typename T>
__device__ __forceinline__ void set_neg_inf(T* dst)
{
    if constexpr (sizeof(T) == 4)
        *reinterpret_cast<float*>(dst) = kNegInf;
    else
        *reinterpret_cast<unsigned short*>(dst) = 0xff80u;   // bf16 -inf
}

template <typename T, int THREADS, bool BULK, bool OUTVEC>
__global__ void __launch_bounds__(THREADS)
row_slices_kernel(const T* in, T* out, int64_t n_rows, int64_t n_cols, int64_t ld_in,
                  int64_t ld_out, int slice_cols, int cs)
{
    constexpr int VEC = Elem<T>::kVec16;
    constexpr int NW = THREADS / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    T* buf = reinterpret_cast<T*>(smem_raw);
    __shared__ float red_m[NW], red_l[NW];
    __shared__ float2 part[2];
    __shared__ __align__(8) unsigned long long bar;

    const int tid = threadIdx.x;
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;

    const int64_t c0 = static_cast<int64_t>(rank) * slice_cols;
    int64_t len64 = n_cols - c0;
    len64 = len64 < 0 ? 0 : (len64 > slice_cols ? slice_cols : len64);
    const int len = static_cast<int>(len64);
    const int len_pad = (len + VEC - 1) / VEC * VEC;
    const int nv = len_pad / VEC;

    const uint32_t bar_a = smem_addr(&bar);
    if (BULK && tid == 0) {
        mbar_init(bar_a, 1);
        fence_mbar_init();
    }
    for (int e = len + tid; e < len_pad; e += THREADS)
        set_neg_inf(buf + e);                       // pad to whole vectors
    __syncthreads();

    bool failed = false;                            // CTA-uniform
    uint32_t failed_phase = 0;
    uint32_t phase = 0;
    int slot = 0;
    for (int64_t row = cluster_id; row < n_rows; row += n_clusters, phase ^= 1u, slot ^= 1) {
        const T* src = in + row * ld_in + c0;
        // ---- stage the slice in shared memory
        if constexpr (BULK) {
            const uint32_t bytes = static_cast<uint32_t>(len * sizeof(T)) & ~15u;
            if (tid == 0 && !failed) {
                fence_proxy_async_smem();           // earlier generic reads of buf
                if (bytes) {
                    mbar_arrive_expect_tx(bar_a, bytes);
                    const uint32_t dst = smem_addr(buf);
                    for (uint32_t off = 0; off < bytes; off += kBulkChunkBytes) {
                        const uint32_t n = bytes - off < kBulkChunkBytes ? bytes - off : kBulkChunkBytes;
                        bulk_g2s(dst + off, reinterpret_cast<const char*>(src) + off, n, bar_a);
                    }
                } else {
                    mbar_arrive(bar_a);
                }
            }
            for (int e = static_cast<int>(bytes / sizeof(T)) + tid; e < len; e += THREADS)
                copy_elem(buf + e, src + e);        // < 16-byte ragged tail
            const bool ok = failed ? true : mbar_wait_bounded(bar_a, phase);
            if (__syncthreads_or(!ok) && !failed) {
                failed = true;
                failed_phase = phase;
            }
        } else {
            for (int e = tid; e < len; e += THREADS)
                copy_elem(buf + e, src + e);
            __syncthreads();
        }

        // ---- pass A: online (m, l) over this thread's vectors
        float m = kNegInf, l = 0.0f;
        for (int v0 = tid; v0 < nv; v0 += THREADS * kBatch) {
            float x[kBatch * VEC];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int v = v0 + k * THREADS;
                if (v < nv) {
                    lds_vec<T, VEC>(buf + v * VEC, &x[k * VEC]);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        x[k * VEC + j] = kNegInf;
                }
            }
            float bm = kNegInf;
#pragma unroll
            for (int i = 0; i < kBatch * VEC; ++i)
                bm = fmaxf(bm, x[i]);
            const float mn = fmaxf(m, bm);
            const float ref = (mn == kNegInf) ? 0.0f : mn;
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < kBatch * VEC; ++i)
                s += exp_fast(x[i] - ref);
            l = l * exp_fast(m - ref) + s;
            m = mn;
        }

        // ---- merge: warp, CTA, cluster
        cta_ml_reduce<THREADS>(m, l, red_m, red_l);
        if (cs > 1)
            cluster_ml_reduce(m, l, part, slot, cs);
        const float inv = 1.0f / l;

        // ---- pass B: normalise and store
        T* dst = out + row * ld_out + c0;
        for (int v = tid; v < nv; v += THREADS) {
            float x[VEC];
            lds_vec<T, VEC>(buf + v * VEC, x);
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                x[j] = exp_fast(x[j] - m);
            if constexpr (OUTVEC) {
                store_vec_masked<T, VEC>(dst, static_cast<int64_t>(v) * VEC, len, x, inv);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (v * VEC + j < len)
                        Elem<T>::store1(dst + v * VEC + j, x[j] * inv);
            }
        }
        __syncthreads();                            // buf and red_* are reused
    }
    if (cs > 1)
        cooperative_groups::this_cluster().sync();  // peers may still read `part`
    if (BULK && failed && tid == 0) {
        atomicOr(&g_error_row_slices, kErrMbarrierTimeout);
        mbar_wait_bounded(bar_a, failed_phase);     // the copy still in flight
    }
}

// A single thread waits, with the bounded wait above, on an mbarrier that
// expects one arrival nobody makes; the wait runs out and the timeout is
// recorded in the same error word the row-slice kernel uses.
__global__ void selftest_wait_kernel()
{
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t a = smem_addr(&bar);
    mbar_init(a, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(a, 0))
        atomicOr(&g_error_row_slices, kErrMbarrierTimeout);
}

cudaError_t launch_selftest_wait(cudaStream_t s)
{
    selftest_wait_kernel<<<1, 1, 0, s>>>();
    note_launch();
    return cudaGetLastError();
}

// ------------------------------------------------------------------ host side

unsigned read_error_row_slices(bool clear)
{
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_row_slices, sizeof v) != cudaSuccess)
        return 0;
    if (clear && v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_error_row_slices, &zero, sizeof zero);
    }
    return v;
}

namespace {

constexpr int kMaxDevices = 64;

// Per-device, per-instantiation attribute state (dynamic smem limit set so far).
template <typename Kernel>
struct KernelAttrs {
    std::atomic<int> smem_set[kMaxDevices];
    std::atomic<bool> cluster_set[kMaxDevices];
};

template <typename T, int THREADS, bool BULK, bool OUTVEC>
cudaError_t launch_rs(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    auto* k = row_slices_kernel<T, THREADS, BULK, OUTVEC>;
    static KernelAttrs<decltype(k)> attrs;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (attrs.smem_set[dev].load() < plan.smem_bytes) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem_bytes);
        if (err != cudaSuccess)
            return err;
        attrs.smem_set[dev].store(plan.smem_bytes);
    }
    if (!attrs.cluster_set[dev].load()) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess)
            return err;
        cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        attrs.cluster_set[dev].store(true);
    }
    const int cs = plan.cluster;
    int64_t grid = p.n_rows * cs;
    const int64_t cap = (int64_t{0x7fffffff} / cs) * cs;
    if (grid > cap)
        grid = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan.smem_bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cs > 1 ? 1 : 0;
    err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in), static_cast<T*>(p.out),
                             p.n_rows, p.n_cols, p.ld_in, p.ld_out,
                             static_cast<int>(plan.slice_cols), cs);
    note_launch();
    return err;
}

template <typename T, int THREADS>
cudaError_t launch_flags(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    const bool outvec = plan.out_vec > 1;
    if (plan.bulk_copy)
        return outvec ? launch_rs<T, THREADS, true, true>(p, plan, s)
                      : launch_rs<T, THREADS, true, false>(p, plan, s);
    return outvec ? launch_rs<T, THREADS, false, true>(p, plan, s)
                  : launch_rs<T, THREADS, false, false>(p, plan, s);
}

template <typename T>
cudaError_t launch_threads(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    switch (plan.threads) {
    case 128: return launch_flags<T, 128>(p, plan, s);
    case 256: return launch_flags<T, 256>(p, plan, s);
    case 512: return launch_flags<T, 512>(p, plan, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_row_slices(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    return p.dtype == SOFTMAX_F32 ? launch_threads<float>(p, plan, s)
                                  : launch_threads<BF16Bits>(p, plan, s);
}

int max_cluster_size_row_slices()
{
    auto* k = row_slices_kernel<float, 512, true, true>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 8;
    const int smem = 96 * 1024;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(512, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int size = 0;
    if (cudaOccupancyMaxPotentialClusterSize(&size, k, &cfg) != cudaSuccess || size < 1) {
        cudaGetLastError();
        return 8;
    }
    return size > 16 ? 16 : size;
}

}  // namespace rwsm
