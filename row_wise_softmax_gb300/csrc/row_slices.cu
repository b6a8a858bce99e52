// CTA and CLUSTER paths: a row (CTA path, cs == 1) or a slice of a row
// (CLUSTER path, cs CTAs per row) is read from HBM exactly once.
//
// Persistent CTAs (clusters) walk their rows r, r + G, r + 2G, ... with a ring
// of `stages` shared-memory buffers, one slice each:
//
//   ring    one elected thread keeps up to `stages` slices in flight with
//           cp.async.bulk copies (global -> shared, completing on one mbarrier
//           per stage).  A ragged tail of fewer than 16 bytes is read with
//           plain loads by the thread that owns it.
//   load    every thread copies its vectors of the slice from shared memory
//           into registers; after a CTA barrier the stage is refilled with the
//           slice `stages` rows ahead, so HBM reads continue while this row is
//           reduced and stored.
//   max     m: thread, warp (__shfl_xor), CTA (shared memory), and for a
//           cluster, every CTA's maximum read through distributed shared
//           memory after a cluster barrier.
//   exp/sum e = exp(x - m) kept in registers (exp_biased, one ex2 per element),
//           l = sum reduced the same way.
//   store   y = e * (1/l), 16-byte vector stores when the output rows allow.
//
// This is the fused softmax of "Triton: write CUDA-grade GPU operators in
// Python" (example 2) — one HBM read and one write per element — with the row
// split over the SMs of a cluster when it is longer than one SM can hold;
// tiling a row over several blocks and combining their partial results is the
// "Level 2: Row Sum (tiling)" pattern of the cs336 lecture 6 notes.  Without
// staging (input rows not 16-byte aligned, or rows in host memory) the kernel
// reads the slice straight into registers (no ring), with 16-byte loads when
// the rows allow.
//
// The kernel is compiled twice: here for the plain softmax, and for
// softmax_options_t (scale, causal mask) in row_slices_options.cu, which
// defines RWSM_ROW_SLICES_OPTIONS and includes this file, so that the two
// sets of instantiations build in parallel.
#include "common.cuh"
#include "kernels.h"

#include <atomic>

#ifndef RWSM_ROW_SLICES_OPTIONS
#define RWSM_ROW_SLICES_OPTIONS 0
#endif

namespace rwsm {

// Error word of this translation unit's kernels (the options unit has its own).
static __device__ unsigned g_error_row_slices = 0;
constexpr bool kOptions = RWSM_ROW_SLICES_OPTIONS != 0;

constexpr int kMaxStages = 8;
constexpr uint32_t kBulkChunkBytes = 32768;
// The ring starts at the first 128-byte boundary of dynamic shared memory;
// launches request this much slack on top of the plan's ring size.
constexpr int kRingAlign = 128;
// Waves of resident CTAs that an automatic single-CTA grid launches, by
// element size: fp32 gained up to ten waves, 16-bit rows peaked near two.
constexpr int64_t kCtaWaves4 = 10;
constexpr int64_t kCtaWaves2 = 2;

template <typename T>
__device__ __forceinline__ void set_neg_inf(T* dst)
{
    if constexpr (sizeof(T) == 4)
        *reinterpret_cast<float*>(dst) = kNegInf;
    else
        *reinterpret_cast<unsigned short*>(dst) = Elem<T>::kNegInfBits;
}

// One element from shared memory, widened to fp32.
template <typename T>
__device__ __forceinline__ float lds1(const T* p)
{
    if constexpr (sizeof(T) == 4)
        return *reinterpret_cast<const float*>(p);
    else
        return Elem<T>::widen(*reinterpret_cast<const unsigned short*>(p));
}

// Cluster-wide reduction of one float per CTA: thread 0 publishes v in its
// shared slot, a cluster barrier (release / acquire) orders the writes, then
// each warp reads the cs slots through distributed shared memory and reduces
// them.  The slot of a given kind is rewritten only one row later, after at
// least one more cluster barrier that every peer reaches only once it has
// read the previous value.
template <bool IS_MAX>
__device__ __forceinline__ float cluster_reduce(float v, float* slot, int cs)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    if (threadIdx.x == 0)
        *slot = v;
    cluster.sync();
    const int lane = threadIdx.x & 31;
    float r = IS_MAX ? kNegInf : 0.0f;
    if (lane < cs)
        r = *cluster.map_shared_rank(slot, lane);
    return IS_MAX ? warp_max(r) : warp_sum(r);
}

template <typename T, int THREADS, int NV, bool BULK, bool OUTVEC, bool OPTS>
__global__ void __launch_bounds__(THREADS)
row_slices_kernel(const T* in, T* out, int64_t n_rows, int n_cols, int64_t ld_in,
                  int64_t ld_out, int slice_cols, int cs, int stages, int in_vec, LogitsArg lg)
{
    constexpr int VEC = Elem<T>::kVec16;
    constexpr int NW = THREADS / 32;
    constexpr int E = NV * VEC;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ float red_max[NW], red_sum[NW];
    __shared__ float part[2][2];
    __shared__ __align__(8) unsigned long long full[kMaxStages];
    __shared__ unsigned issued[kMaxStages];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float kk = OPTS ? lg.k : kLog2e;       // exponent multiplier, scale * log2 e
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;
    const int c0 = rank * slice_cols;
    int len = n_cols - c0;
    len = len < 0 ? 0 : (len > slice_cols ? slice_cols : len);
    const int nv = (len + VEC - 1) / VEC;
    // Without options every row copies [0, plain_copied) of the slice; the
    // vector holding a < 16-byte ragged tail (if any) is tail_vec.
    const uint32_t plain_bytes = static_cast<uint32_t>(len * sizeof(T)) & ~15u;
    const int plain_copied = static_cast<int>(plain_bytes / sizeof(T));
    const int tail_vec = plain_copied < len ? plain_copied / VEC : -1;
    // Columns of this slice that take part in `row` (all of them unless a
    // causal mask stops the row inside or before the slice).
    auto row_lim = [&](int64_t row) -> int {
        if constexpr (!OPTS)
            return len;
        int64_t lim = logits_valid(lg, row, n_cols) - c0;
        return static_cast<int>(lim < 0 ? 0 : (lim > len ? len : lim));
    };

    T* ring = reinterpret_cast<T*>((reinterpret_cast<uintptr_t>(smem_raw) + (kRingAlign - 1)) &
                                   ~static_cast<uintptr_t>(kRingAlign - 1));
    auto stage_ptr = [&](int s) { return ring + static_cast<int64_t>(s) * slice_cols; };
    auto issue = [&](int s, int64_t row) {      // thread 0 only
        const uint32_t bar = smem_addr(&full[s]);
        const uint32_t bulk_bytes = OPTS ? span_copy_bytes<T>(row_lim(row), n_cols - c0)
                                         : plain_bytes;
        fence_proxy_async_smem();
        issued[s] += 1;
        if (bulk_bytes) {
            mbar_arrive_expect_tx(bar, bulk_bytes);
            const char* src = reinterpret_cast<const char*>(in + row * ld_in + c0);
            const uint32_t dst = smem_addr(stage_ptr(s));
            for (uint32_t off = 0; off < bulk_bytes; off += kBulkChunkBytes) {
                const uint32_t n = bulk_bytes - off < kBulkChunkBytes ? bulk_bytes - off : kBulkChunkBytes;
                bulk_g2s(dst + off, src + off, n, bar);
            }
        } else {
            mbar_arrive(bar);
        }
    };

    bool failed = false;                      // CTA-uniform
    // Cluster launches let the next grid start only after the row loop:
    // clusters of the next grid placed early into leftover slots measured
    // slower.  Single-CTA launches let it start at once.
    if (cs == 1)
        pdl_launch_dependents();
    if constexpr (BULK) {
        if (tid == 0) {
            for (int s = 0; s < stages; ++s) {
                mbar_init(smem_addr(&full[s]), 1);
                issued[s] = 0;
            }
            fence_mbar_init();
            // The first rows' bytes into L2 while the preceding grid drains
            // (a prefetch reads nothing into this CTA: the copies after
            // griddepcontrol.wait see the preceding grid's writes).  Later
            // waves prefetch too: their copies wait for the ring's set-up,
            // the prefetch does not (measured +1% against the first wave
            // alone on 4096x4096 fp32).
            for (int s = 0; s < stages; ++s) {
                const int64_t row = cluster_id + s * n_clusters;
                if (row >= n_rows)
                    break;
                const uint32_t bytes = OPTS ? span_copy_bytes<T>(row_lim(row), n_cols - c0) : plain_bytes;
                const char* src = reinterpret_cast<const char*>(in + row * ld_in + c0);
                for (uint32_t off = 0; off < bytes; off += kBulkChunkBytes)
                    bulk_prefetch_l2(src + off, bytes - off < kBulkChunkBytes ? bytes - off : kBulkChunkBytes);
            }
        }
        if constexpr (!OPTS) {
            // Every row copies the same span: positions of the last vector
            // that the copies never write read as -inf.
            for (int s = 0; s < stages; ++s)
                for (int e = plain_copied + tid; e < nv * VEC; e += THREADS)
                    set_neg_inf(stage_ptr(s) + e);
        }
        __syncthreads();
        pdl_wait();
        if (tid == 0)
            for (int s = 0; s < stages; ++s) {
                const int64_t row = cluster_id + s * n_clusters;
                if (row < n_rows)
                    issue(s, row);
            }
    } else {
        pdl_wait();
    }

    int64_t i = 0;
    for (int64_t row = cluster_id; row < n_rows; row += n_clusters, ++i) {
        float x[E];
        const T* src = in + row * ld_in + c0;
        const int lim = row_lim(row);
        if constexpr (BULK) {
            const int s = static_cast<int>(i % stages);
            const uint32_t parity = static_cast<uint32_t>((i / stages) & 1);
            const bool ok = failed ? true : mbar_wait_bounded(smem_addr(&full[s]), parity);
            const T* st = stage_ptr(s);
            if constexpr (!OPTS) {
                // [0, plain_copied) was copied, the rest of its last vector
                // is -inf in the ring; a < 16-byte ragged tail of the row is
                // patched in from HBM.
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int v = tid + k * THREADS;
                    if (v < nv) {
                        lds_vec<T, VEC>(st + v * VEC, &x[k * VEC]);
                        if (v == tail_vec) {
#pragma unroll
                            for (int j = 0; j < VEC; ++j) {
                                const int e = v * VEC + j;
                                if (e >= plain_copied)
                                    x[k * VEC + j] = e < len ? Elem<T>::load1(src + e) : kNegInf;
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            x[k * VEC + j] = kNegInf;
                    }
                }
            } else {
                // [0, copied) was copied; [copied, lim) is a < 16-byte tail read
                // from HBM; from lim on the slice is masked or past the row (-inf).
                int copied = static_cast<int>(span_copy_bytes<T>(lim, n_cols - c0) / sizeof(T));
                copied = copied < lim ? copied : lim;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int e0 = (tid + k * THREADS) * VEC;
                    if (e0 + VEC <= copied) {
                        lds_vec<T, VEC>(st + e0, &x[k * VEC]);
                    } else if (e0 >= lim) {
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            x[k * VEC + j] = kNegInf;
                    } else {
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const int e = e0 + j;
                            x[k * VEC + j] = e < copied ? lds1(st + e)
                                                        : (e < lim ? Elem<T>::load1(src + e) : kNegInf);
                        }
                    }
                }
            }
            // Every thread has its slice in registers: the stage is free.
            if (__syncthreads_or(!ok))
                failed = true;
            if (tid == 0 && !failed) {
                const int64_t next = row + static_cast<int64_t>(stages) * n_clusters;
                if (next < n_rows)
                    issue(s, next);
            }
        } else if (in_vec) {
            // No staging (rows in host memory): 16-byte loads into registers.
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int v = tid + k * THREADS;
                if (v < nv) {
                    load_vec_masked<T, VEC, OPTS>(src, v * VEC, lim, &x[k * VEC]);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        x[k * VEC + j] = kNegInf;
                }
            }
        } else {
            // Input rows not 16-byte aligned: element loads only (same
            // register layout as the vector path).
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int v = tid + k * THREADS;
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const int e = v * VEC + j;
                    x[k * VEC + j] = (v < nv && e < lim) ? Elem<T>::load1(src + e) : kNegInf;
                }
            }
        }

        // ---- row maximum
        float m = kNegInf;
#pragma unroll
        for (int e = 0; e < E; ++e)
            m = fmaxf(m, x[e]);
        m = warp_max(m);
        if (lane == 0)
            red_max[warp] = m;
        __syncthreads();
        m = warp_max(lane < NW ? red_max[lane] : kNegInf);
        if (cs > 1)
            m = cluster_reduce<true>(m, &part[i & 1][0], cs);

        // ---- exponentials and their sum (biased by 2^64, see exp_biased)
        float l = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            x[e] = exp_biased(x[e] - m, kk);
            l += x[e];
        }
        l = warp_sum(l);
        if (lane == 0)
            red_sum[warp] = l;
        __syncthreads();
        l = warp_sum(lane < NW ? red_sum[lane] : 0.0f);
        if (cs > 1)
            l = cluster_reduce<false>(l, &part[i & 1][1], cs);
        const float inv = 1.0f / l;

        // ---- normalise and store
        T* dst = out + row * ld_out + c0;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = tid + k * THREADS;
            if (v < nv) {
                if constexpr (OUTVEC) {
                    store_vec_masked<T, VEC>(dst, v * VEC, len, &x[k * VEC], inv);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        if (v * VEC + j < len)
                            Elem<T>::store1(dst + v * VEC + j, x[k * VEC + j] * inv);
                }
            }
        }
    }
    if (cs > 1)
        pdl_launch_dependents();
    if (cs > 1)
        cooperative_groups::this_cluster().sync();  // peers may still read `part`
    if (BULK && failed && tid == 0) {
        atomicOr(&g_error_row_slices, kErrMbarrierTimeout);
        for (int s = 0; s < stages; ++s)             // copies possibly still in flight
            if (issued[s])
                mbar_wait_bounded(smem_addr(&full[s]), (issued[s] - 1) & 1u);
    }
}

static unsigned read_error_tu(bool clear)
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

#if !RWSM_ROW_SLICES_OPTIONS
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

unsigned read_error_row_slices(bool clear)
{
    return read_error_tu(clear) | read_error_row_slices_options(clear);
}
#else
unsigned read_error_row_slices_options(bool clear)
{
    return read_error_tu(clear);
}
#endif

namespace {

constexpr int kMaxDevices = 64;

struct KernelAttrs {
    std::atomic<int> smem_set[kMaxDevices];
    std::atomic<bool> flags_set[kMaxDevices];
};

template <typename T, int THREADS, int NV, bool BULK, bool OUTVEC>
cudaError_t launch_rs(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    auto* k = row_slices_kernel<T, THREADS, NV, BULK, OUTVEC, kOptions>;
    static KernelAttrs attrs;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int smem = plan.bulk_copy ? plan.smem_bytes + kRingAlign : 0;
    if (attrs.smem_set[dev].load() < smem) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess)
            return err;
        attrs.smem_set[dev].store(smem);
    }
    if (!attrs.flags_set[dev].load()) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess)
            return err;
        cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        attrs.flags_set[dev].store(true);
    }
    const int cs = plan.cluster;
    cudaLaunchAttribute attr[2];
    const int n_attr = launch_attrs(attr, cs);
    int64_t clusters = plan.grid > 0 ? plan.grid / cs : 0;
    if (clusters <= 0) {
        // Persistent: as many CTAs (clusters) as can be resident at once.
        int active = 0;
        if (cs > 1) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
            q.blockDim = dim3(THREADS, 1, 1);
            q.dynamicSmemBytes = static_cast<size_t>(smem);
            q.attrs = attr;
            q.numAttrs = 1;                   // the cluster dimension
            if (cudaOccupancyMaxActiveClusters(&active, k, &q) != cudaSuccess) {
                cudaGetLastError();
                active = 0;
            }
        } else {
            active = resident_ctas(reinterpret_cast<const void*>(k), THREADS, smem);
        }
        if (active < 1)
            active = 1;
        if (cs == 1 && plan.bulk_copy) {
            // Several waves of single CTAs: the block scheduler hands a row
            // to whichever SM frees first, which evens out SMs whose copies
            // drain slower than others (measured on 4096x4096 fp32 5509 ->
            // 6020 GB/s, 65536x1536 fp32 5387 -> 6870, 8192x8192 bf16 5470
            // -> 6200 against one resident wave).  Each CTA keeps at least
            // 1.5 rows so its ring still prefetches a next row.
            const int64_t waves = sizeof(T) == 4 ? kCtaWaves4 : kCtaWaves2;
            int64_t g = waves * active;
            if (g > p.n_rows * 2 / 3)
                g = p.n_rows * 2 / 3;
            clusters = g > active ? g : (p.n_rows < active ? p.n_rows : active);
        } else {
            clusters = balanced_grid(p.n_rows, active, cs == 1 ? sm_count_current() : 0);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n_attr);
    err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in), static_cast<T*>(p.out),
                             p.n_rows, static_cast<int>(p.n_cols), p.ld_in, p.ld_out,
                             static_cast<int>(plan.slice_cols), cs, plan.stages,
                             plan.vec > 1 ? 1 : 0, logits_of(p));
    note_launch();
    return err;
}

template <typename T, int THREADS, int NV>
cudaError_t launch_flags(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    const bool outvec = plan.out_vec > 1;
    if (plan.bulk_copy)
        return outvec ? launch_rs<T, THREADS, NV, true, true>(p, plan, s)
                      : launch_rs<T, THREADS, NV, true, false>(p, plan, s);
    return outvec ? launch_rs<T, THREADS, NV, false, true>(p, plan, s)
                  : launch_rs<T, THREADS, NV, false, false>(p, plan, s);
}

template <typename T, int THREADS>
cudaError_t launch_nv(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    switch (plan.chunks) {
    case 1: return launch_flags<T, THREADS, 1>(p, plan, s);
    case 2: return launch_flags<T, THREADS, 2>(p, plan, s);
    case 4: return launch_flags<T, THREADS, 4>(p, plan, s);
    case 8:
        if constexpr (sizeof(T) == 4) return launch_flags<T, THREADS, 8>(p, plan, s);
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_threads(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    switch (plan.threads) {
    case 64: return launch_nv<T, 64>(p, plan, s);
    case 128: return launch_nv<T, 128>(p, plan, s);
    case 256: return launch_nv<T, 256>(p, plan, s);
    case 512: return launch_nv<T, 512>(p, plan, s);
    case 1024: return launch_nv<T, 1024>(p, plan, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

#if RWSM_ROW_SLICES_OPTIONS
cudaError_t launch_row_slices_options(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (p.dtype == SOFTMAX_F32)
        return launch_threads<float>(p, plan, s);
    return p.dtype == SOFTMAX_BF16 ? launch_threads<BF16Bits>(p, plan, s)
                                   : launch_threads<F16Bits>(p, plan, s);
}
#else
cudaError_t launch_row_slices(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (plan.bulk_copy && (plan.stages < 1 || plan.stages > kMaxStages))
        return cudaErrorInvalidValue;
    if (has_options(p))
        return launch_row_slices_options(p, plan, s);
    if (p.dtype == SOFTMAX_F32)
        return launch_threads<float>(p, plan, s);
    return p.dtype == SOFTMAX_BF16 ? launch_threads<BF16Bits>(p, plan, s)
                                   : launch_threads<F16Bits>(p, plan, s);
}

int max_cluster_size_row_slices()
{
    auto* k = row_slices_kernel<float, 512, 8, true, true, false>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 8;
    const int smem = 64 * 1024 + kRingAlign;
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
#endif

}  // namespace rwsm
