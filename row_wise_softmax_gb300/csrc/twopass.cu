// TWOPASS path, for rows too long for a cluster's shared memory: the row is
// streamed from HBM twice.
//
//   pass 1  each CTA of the row's cluster walks its slice in batches of
//           vectors held in registers, keeping an online (m, l) partial per
//           thread (the running max / rescaled sum of "Triton GPU programming
//           deep dive", section 3.3, over column tiles as in the "Level 2:
//           Row Sum (tiling)" loop of the cs336 lecture 6 notes);
//   merge   warp, CTA and cluster (distributed shared memory) merges give
//           every thread the row's (M, L);
//   pass 2  the slice is read again and y = e^(x - M) / L is written.
//
// A slice is re-read soon after its first read: the first pass reads with an
// L2 evict-last policy and the second pass (and the stores) with evict-first,
// so the second read mostly hits L2 and HBM traffic stays close to one read
// and one write per element.
// In place (in == out) is safe: every element is re-read by the thread that
// then writes it, and the cluster barrier between the passes orders every
// pass-1 read of the row before any write.
#include "common.cuh"
#include "kernels.h"

namespace rwsm {

constexpr int kTwoPassBatch = 4;

// Load the k-th batch vector of this thread: 16-byte vectors with an L2
// policy when VEC covers 16 bytes, element loads (masked) otherwise.
template <typename T, int VEC>
__device__ __forceinline__ void tp_load(const T* src, int64_t v, int64_t len, float* x,
                                        uint64_t pol)
{
    if constexpr (VEC * sizeof(T) == 16) {
        if ((v + 1) * VEC <= len) {
            load16_hint<T>(src + v * VEC, x, pol);
            return;
        }
    }
    load_vec_masked<T, VEC>(src, v * VEC, len, x);
}

// Walk this thread's batches of B vectors (v = v0 + k*THREADS, batches
// THREADS*B apart) with two register buffers: the loads of the next batch are
// issued before `body` consumes the current one, so every thread keeps one
// batch in flight while it computes.
template <typename T, int VEC, int B, int THREADS, typename Body>
__device__ __forceinline__ void pipelined_batches(const T* src, int64_t nv, int64_t len,
                                                  uint64_t pol, Body&& body)
{
    constexpr int64_t kStride = int64_t{THREADS} * B;
    auto load_batch = [&](float (&x)[B * VEC], int64_t v0) {
#pragma unroll
        for (int k = 0; k < B; ++k) {
            const int64_t v = v0 + int64_t{k} * THREADS;
            if (v < nv) {
                tp_load<T, VEC>(src, v, len, &x[k * VEC], pol);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    x[k * VEC + j] = kNegInf;
            }
        }
    };
    int64_t v0 = threadIdx.x;
    if (v0 >= nv)
        return;
    float a[B * VEC], b[B * VEC];
    load_batch(a, v0);
    while (true) {
        const int64_t v1 = v0 + kStride;
        if (v1 < nv)
            load_batch(b, v1);
        body(a, v0);
        if (v1 >= nv)
            break;
        const int64_t v2 = v1 + kStride;
        if (v2 < nv)
            load_batch(a, v2);
        body(b, v1);
        if (v2 >= nv)
            break;
        v0 = v2;
    }
}

template <typename T, int VEC, int THREADS>
__global__ void __launch_bounds__(THREADS)
twopass_kernel(const T* in, T* out, int64_t n_rows, int64_t n_cols, int64_t ld_in,
               int64_t ld_out, int64_t slice_cols, int cs, LogitsArg lg)
{
    constexpr int NW = THREADS / 32;
    constexpr int B = kTwoPassBatch;
    __shared__ float red_m[NW], red_l[NW];
    __shared__ float2 part[2];

    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;
    const int64_t c0 = static_cast<int64_t>(rank) * slice_cols;
    int64_t len = n_cols - c0;
    len = len < 0 ? 0 : (len > slice_cols ? slice_cols : len);
    const int64_t nv = (len + VEC - 1) / VEC;
    const uint64_t keep = policy_evict_last();     // first read: stay in L2
    const uint64_t stream = policy_evict_first();  // second read and stores
    // Cluster launches let the next grid start only after the row loop:
    // clusters of the next grid placed early into leftover slots measured
    // slower.  Single-CTA launches let it start at once.
    if (cs == 1)
        pdl_launch_dependents();
    pdl_wait();

    int slot = 0;
    for (int64_t row = cluster_id; row < n_rows; row += n_clusters, slot ^= 1) {
        const T* src = in + row * ld_in + c0;
        // Kept columns of this slice (a causal mask can stop the row early).
        int64_t lim = logits_valid(lg, row, n_cols) - c0;
        lim = lim < 0 ? 0 : (lim > len ? len : lim);
        // ---- pass 1: online (m, l) over this thread's batches
        float m = kNegInf, l = 0.0f;
        pipelined_batches<T, VEC, B, THREADS>(src, nv, lim, keep,
            [&](const float (&x)[B * VEC], int64_t) {
                float bm = kNegInf;
#pragma unroll
                for (int i = 0; i < B * VEC; ++i)
                    bm = fmaxf(bm, x[i]);
                const float mn = fmaxf(m, bm);
                const float ref = (mn == kNegInf) ? 0.0f : mn;
                float s = 0.0f;
#pragma unroll
                for (int i = 0; i < B * VEC; ++i)
                    s += exp_biased(x[i] - ref, lg.k);
                l = l * exp_ftz(m - ref, lg.k) + s;
                m = mn;
            });
        cta_ml_reduce<THREADS>(m, l, red_m, red_l, lg.k);
        if (cs > 1)
            cluster_ml_reduce(m, l, part, slot, cs, lg.k);
        const float inv = 1.0f / l;

        // ---- pass 2: normalise (the re-read mostly hits L2)
        T* dst = out + row * ld_out + c0;
        pipelined_batches<T, VEC, B, THREADS>(src, nv, lim, stream,
            [&](const float (&xin)[B * VEC], int64_t v0) {
#pragma unroll
                for (int k = 0; k < B; ++k) {
                    const int64_t v = v0 + int64_t{k} * THREADS;
                    if (v < nv) {
                        float x[VEC];
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            x[j] = exp_biased(xin[k * VEC + j] - m, lg.k);
                        if (VEC * sizeof(T) == 16 && (v + 1) * VEC <= len)
                            store16_hint<T>(dst + v * VEC, x, inv, stream);
                        else
                            store_vec_masked<T, VEC>(dst, v * VEC, len, x, inv);
                    }
                }
            });
        __syncthreads();                       // red_* reused by the next row
    }
    if (cs > 1)
        pdl_launch_dependents();
    if (cs > 1)
        cooperative_groups::this_cluster().sync();
}

namespace {

template <typename T, int VEC, int THREADS>
cudaError_t launch_tp(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    auto* k = twopass_kernel<T, VEC, THREADS>;
    const int cs = plan.cluster;
    cudaError_t err = cudaSuccess;
    if (cs > 8) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess)
            return err;
    }
    int64_t clusters = plan.grid > 0 ? plan.grid / cs : 0;
    if (clusters <= 0) {
        // Persistent: as many clusters as can be resident at once.
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(cs, 1, 1);
        q.blockDim = dim3(THREADS, 1, 1);
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = cs;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        q.attrs = a;
        q.numAttrs = 1;
        int active = 0;
        if (cs > 1) {
            if (cudaOccupancyMaxActiveClusters(&active, k, &q) != cudaSuccess) {
                cudaGetLastError();
                active = 0;
            }
        } else {
            active = resident_ctas(reinterpret_cast<const void*>(k), THREADS, 0);
        }
        if (active < 1)
            active = 1;
        clusters = balanced_grid(p.n_rows, active, cs == 1 ? sm_count_current() : 0);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, cs));
    err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in), static_cast<T*>(p.out),
                             p.n_rows, p.n_cols, p.ld_in, p.ld_out, plan.slice_cols, cs,
                             logits_of(p));
    note_launch();
    return err;
}

template <typename T, int VEC>
cudaError_t launch_tp_threads(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    switch (plan.threads) {
    case 256: return launch_tp<T, VEC, 256>(p, plan, s);
    case 512: return launch_tp<T, VEC, 512>(p, plan, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_twopass(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (p.dtype == SOFTMAX_F32)
        return plan.vec == 4 ? launch_tp_threads<float, 4>(p, plan, s)
                             : launch_tp_threads<float, 1>(p, plan, s);
    if (p.dtype == SOFTMAX_BF16)
        return plan.vec == 8 ? launch_tp_threads<BF16Bits, 8>(p, plan, s)
                             : launch_tp_threads<BF16Bits, 1>(p, plan, s);
    return plan.vec == 8 ? launch_tp_threads<F16Bits, 8>(p, plan, s)
                         : launch_tp_threads<F16Bits, 1>(p, plan, s);
}

}  // namespace rwsm
