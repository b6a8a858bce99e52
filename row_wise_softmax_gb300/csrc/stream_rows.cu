// TWOPASS path, staged: rows too long to keep on chip, with 16-byte aligned
// input.  A cluster of cs CTAs owns a row; each CTA streams its slice of the
// row twice through a ring of `stages` shared-memory chunks:
//
//   ring    one elected thread keeps `stages` chunk copies in flight
//           (cp.async.bulk, global -> shared, one mbarrier per stage) along
//           the fixed sequence (row, pass, chunk).  Pass-1 copies carry an
//           L2 evict-last policy so the lines stay for the second read;
//           pass-2 copies and the output stores carry evict-first.
//   pass 1  each thread folds its vectors of every chunk into an online
//           (m, l): m_new = max(m, chunk max), l = l * e^(m - m_new) +
//           sum e^(x - m_new) — the running-max rescale of "Triton GPU
//           programming deep dive", section 3.3, over the chunks of the
//           "Level 2: Row Sum (tiling)" loop of the cs336 lecture 6 notes.
//   merge   warp (__shfl_xor), CTA (shared memory), cluster (distributed
//           shared memory after a cluster barrier): every thread gets the
//           row's (M, L).
//   pass 2  the slice streams again (mostly from L2): y = e^(x - M) / L.
//
// In-flight data lives in shared memory, not registers (a thread holds one
// chunk's 16 floats), so each SM keeps several ring stages of HBM reads
// outstanding while its warps reduce.  A stage is refilled after a CTA
// barrier shows every thread has its vectors in registers.  The last chunk of
// a slice may be ragged: its final < 16 bytes are read with plain loads by
// the lane that owns them.
#include "common.cuh"
#include "kernels.h"

#include <atomic>

namespace rwsm {

__device__ unsigned g_error_stream_rows = 0;

constexpr int kStreamMaxStages = 8;
constexpr int kStreamRingAlign = 128;

template <typename T, int THREADS, int NV, bool OUTVEC, bool OPTS>
__global__ void __launch_bounds__(THREADS)
stream_rows_kernel(const T* in, T* out, int64_t n_rows, int64_t n_cols, int64_t ld_in,
                   int64_t ld_out, int64_t slice_cols, int cs, int stages, LogitsArg lg)
{
    constexpr int VEC = Elem<T>::kVec16;
    constexpr int NW = THREADS / 32;
    constexpr int E = NV * VEC;
    constexpr int CHUNK = THREADS * E;                  // elements per chunk
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ float red_m[NW], red_l[NW];
    __shared__ float2 part[2];
    __shared__ __align__(8) unsigned long long full[kStreamMaxStages];
    __shared__ unsigned issued[kStreamMaxStages];

    const int tid = threadIdx.x;
    const float kk = OPTS ? lg.k : kLog2e;       // exponent multiplier, scale * log2 e
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;
    const int64_t c0 = static_cast<int64_t>(rank) * slice_cols;
    int64_t len = n_cols - c0;
    len = len < 0 ? 0 : (len > slice_cols ? slice_cols : len);
    const int64_t K = (len + CHUNK - 1) / CHUNK;        // chunks per pass
    const int64_t my_rows = cluster_id < n_rows ? (n_rows - 1 - cluster_id) / n_clusters + 1 : 0;
    const int64_t total_q = my_rows * 2 * K;            // chunk copies this CTA consumes

    T* ring = reinterpret_cast<T*>((reinterpret_cast<uintptr_t>(smem_raw) + (kStreamRingAlign - 1)) &
                                   ~static_cast<uintptr_t>(kStreamRingAlign - 1));
    auto stage_ptr = [&](int s) { return ring + static_cast<int64_t>(s) * CHUNK; };
    // Chunk q of the sequence: row i = q / 2K, pass = (q / K) & 1, chunk q % K.
    auto chunk_len = [&](int64_t chunk) {
        const int64_t rest = len - chunk * CHUNK;
        return static_cast<int>(rest < CHUNK ? rest : CHUNK);
    };
    // Columns of this slice that take part in `row` (all of them unless a
    // causal mask stops the row inside or before the slice), and of `chunk`
    // given that count (masked columns are never copied).
    auto row_keep = [&](int64_t row) -> int64_t { return kept_cols<OPTS>(lg, row, n_cols) - c0; };
    auto chunk_lim = [&](int64_t keep, int64_t chunk) {
        const int64_t rest = keep - chunk * CHUNK;
        const int clen = chunk_len(chunk);
        return static_cast<int>(rest < 0 ? 0 : (rest > clen ? clen : rest));
    };
    const uint64_t keep = policy_evict_last();
    const uint64_t stream = policy_evict_first();
    auto issue = [&](int64_t q) {                       // thread 0 only
        const int s = static_cast<int>(q % stages);
        const int64_t i = q / (2 * K);
        const bool second = ((q / K) & 1) != 0;
        const int64_t chunk = q % K;
        const int64_t row = cluster_id + i * n_clusters;
        uint32_t bytes;
        if constexpr (OPTS)
            bytes = span_copy_bytes<T>(chunk_lim(row_keep(row), chunk), n_cols - c0 - chunk * CHUNK);
        else
            bytes = static_cast<uint32_t>(chunk_len(chunk) * sizeof(T)) & ~15u;
        const uint32_t bar = smem_addr(&full[s]);
        fence_proxy_async_smem();
        issued[s] += 1;
        if (bytes) {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s_hint(smem_addr(stage_ptr(s)), in + row * ld_in + c0 + chunk * CHUNK, bytes,
                          bar, second ? stream : keep);
        } else {
            mbar_arrive(bar);
        }
    };

    // Cluster launches let the next grid start only after the row loop:
    // clusters of the next grid placed early into leftover slots measured
    // slower.  Single-CTA launches let it start at once.
    if (cs == 1)
        pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            issued[s] = 0;
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();
    if (tid == 0)
        for (int64_t q = 0; q < stages && q < total_q; ++q)
            issue(q);

    bool failed = false;                                 // CTA-uniform
    int64_t q = 0;
    // Wait for chunk q, copy this thread's vectors into registers (ragged
    // tail from HBM), release the stage and start the copy `stages` ahead.
    auto take = [&](int64_t keep, const T* src_row, int64_t chunk, float (&x)[E]) {
        const int s = static_cast<int>(q % stages);
        const uint32_t parity = static_cast<uint32_t>((q / stages) & 1);
        const bool ok = failed ? true : mbar_wait_bounded(smem_addr(&full[s]), parity);
        int clen, bulk;                              // kept columns, copied columns
        if constexpr (OPTS) {
            clen = chunk_lim(keep, chunk);
            bulk = static_cast<int>(span_copy_bytes<T>(clen, n_cols - c0 - chunk * CHUNK) / sizeof(T));
            bulk = bulk < clen ? bulk : clen;
        } else {
            clen = chunk_len(chunk);
            bulk = static_cast<int>((clen * sizeof(T)) & ~size_t{15}) / static_cast<int>(sizeof(T));
        }
        const T* st = stage_ptr(s);
        const T* g = src_row + chunk * CHUNK;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int e0 = (tid + k * THREADS) * VEC;
            if (e0 + VEC <= bulk) {
                lds_vec<T, VEC>(st + e0, &x[k * VEC]);
            } else if (OPTS && e0 >= clen) {
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    x[k * VEC + j] = kNegInf;
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    const int e = e0 + j;
                    x[k * VEC + j] = e < clen ? Elem<T>::load1(g + e) : kNegInf;
                }
            }
        }
        if (__syncthreads_or(!ok))
            failed = true;
        if (tid == 0 && !failed && q + stages < total_q)
            issue(q + stages);
        ++q;
    };

    int slot = 0;
    for (int64_t row = cluster_id; row < n_rows; row += n_clusters, slot ^= 1) {
        const T* src = in + row * ld_in + c0;
        const int64_t keep = row_keep(row);
        // ---- pass 1: online (m, l)
        float m = kNegInf, l = 0.0f;
        for (int64_t chunk = 0; chunk < K; ++chunk) {
            float x[E];
            take(keep, src, chunk, x);
            float bm = kNegInf;
#pragma unroll
            for (int e = 0; e < E; ++e)
                bm = fmaxf(bm, x[e]);
            const float mn = fmaxf(m, bm);
            const float ref = (mn == kNegInf) ? 0.0f : mn;
            float sum = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e)
                sum += exp_biased(x[e] - ref, kk);
            l = l * exp_ftz(m - ref, kk) + sum;
            m = mn;
        }
        cta_ml_reduce<THREADS>(m, l, red_m, red_l, kk);
        if (cs > 1)
            cluster_ml_reduce(m, l, part, slot, cs, kk);
        const float inv = 1.0f / l;
        // ---- pass 2: normalise and store
        T* dst = out + row * ld_out + c0;
        for (int64_t chunk = 0; chunk < K; ++chunk) {
            float x[E];
            take(keep, src, chunk, x);
            const int clen = chunk_len(chunk);
            T* d = dst + chunk * CHUNK;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int e0 = (tid + k * THREADS) * VEC;
                if (e0 < clen) {
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        x[k * VEC + j] = exp_biased(x[k * VEC + j] - m, kk);
                    if constexpr (OUTVEC) {
                        if (e0 + VEC <= clen)
                            store16_hint<T>(d + e0, &x[k * VEC], inv, stream);
                        else
                            store_vec_masked<T, VEC>(d, e0, clen, &x[k * VEC], inv);
                    } else {
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            if (e0 + j < clen)
                                Elem<T>::store1(d + e0 + j, x[k * VEC + j] * inv);
                    }
                }
            }
        }
        __syncthreads();        // red_* are rewritten by the next row's reduction
    }
    if (cs > 1)
        pdl_launch_dependents();
    if (cs > 1)
        cooperative_groups::this_cluster().sync();       // peers may still read `part`
    if (failed && tid == 0) {
        atomicOr(&g_error_stream_rows, kErrMbarrierTimeout);
        for (int s = 0; s < stages; ++s)                  // copies possibly still in flight
            if (issued[s])
                mbar_wait_bounded(smem_addr(&full[s]), (issued[s] - 1) & 1u);
    }
}

// ------------------------------------------------------------------ host side

unsigned read_error_stream_rows(bool clear)
{
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_stream_rows, sizeof v) != cudaSuccess)
        return 0;
    if (clear && v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_error_stream_rows, &zero, sizeof zero);
    }
    return v;
}

namespace {

constexpr int kMaxDevices = 64;

struct StreamAttrs {
    std::atomic<int> smem_set[kMaxDevices];
    std::atomic<bool> flags_set[kMaxDevices];
};

template <typename T, int THREADS, int NV, bool OUTVEC, bool OPTS>
cudaError_t launch_stream_opts(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    auto* k = stream_rows_kernel<T, THREADS, NV, OUTVEC, OPTS>;
    static StreamAttrs attrs;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int smem = plan.smem_bytes + kStreamRingAlign;
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
        int active = 0;
        if (cs > 1) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
            q.blockDim = dim3(THREADS, 1, 1);
            q.dynamicSmemBytes = static_cast<size_t>(smem);
            q.attrs = attr;
            q.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&active, k, &q) != cudaSuccess) {
                cudaGetLastError();
                active = 0;
            }
        } else {
            active = resident_ctas(reinterpret_cast<const void*>(k), THREADS, smem);
        }
        if (active < 1)
            active = 1;
        clusters = balanced_grid(p.n_rows, active, cs == 1 ? sm_count_current() : 0);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n_attr);
    err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in), static_cast<T*>(p.out),
                             p.n_rows, p.n_cols, p.ld_in, p.ld_out, plan.slice_cols, cs,
                             plan.stages, logits_of(p));
    note_launch();
    return err;
}

template <typename T, int THREADS, int NV, bool OUTVEC>
cudaError_t launch_stream(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    return has_options(p) ? launch_stream_opts<T, THREADS, NV, OUTVEC, true>(p, plan, s)
                    : launch_stream_opts<T, THREADS, NV, OUTVEC, false>(p, plan, s);
}

template <typename T, int THREADS>
cudaError_t launch_stream_nv(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    const bool outvec = plan.out_vec > 1;
    switch (plan.chunks) {
    case 2: return outvec ? launch_stream<T, THREADS, 2, true>(p, plan, s)
                          : launch_stream<T, THREADS, 2, false>(p, plan, s);
    case 4: return outvec ? launch_stream<T, THREADS, 4, true>(p, plan, s)
                          : launch_stream<T, THREADS, 4, false>(p, plan, s);
    case 8:
        if constexpr (sizeof(T) == 4)
            return outvec ? launch_stream<T, THREADS, 8, true>(p, plan, s)
                          : launch_stream<T, THREADS, 8, false>(p, plan, s);
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_stream_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (plan.stages < 1 || plan.stages > kStreamMaxStages)
        return cudaErrorInvalidValue;
    if (p.dtype == SOFTMAX_F32) {
        if (plan.threads == 256) return launch_stream_nv<float, 256>(p, plan, s);
        if (plan.threads == 512) return launch_stream_nv<float, 512>(p, plan, s);
    } else if (p.dtype == SOFTMAX_BF16) {
        if (plan.threads == 256) return launch_stream_nv<BF16Bits, 256>(p, plan, s);
        if (plan.threads == 512) return launch_stream_nv<BF16Bits, 512>(p, plan, s);
    } else {
        if (plan.threads == 256) return launch_stream_nv<F16Bits, 256>(p, plan, s);
        if (plan.threads == 512) return launch_stream_nv<F16Bits, 512>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rwsm
