// TWOPASS path, staged: rows too long to keep on chip, with 16-byte aligned
// input.  A cluster of cs CTAs owns a row; each CTA owns a slice of it and
// streams the slice twice through a shared-memory ring: once from HBM, once
// more mostly from L2.
//
//   producer  the last warp of the CTA (one elected lane) keeps `stages`
//             chunk copies in flight (cp.async.bulk, global -> shared, one
//             "full" mbarrier per stage) along the fixed sequence
//             (row, pass, chunk).  First-pass copies carry an L2 evict-last
//             policy so the lines stay for the second read; second-pass
//             copies and the output stores carry evict-first.  It refills a
//             stage as soon as its "empty" mbarrier shows every consumer warp
//             has the chunk in registers: no CTA-wide barrier per chunk.
//   pass 1    the consumer warps fold each chunk into an online (m, l):
//             m_new = max(m, chunk max), l = l * e^(m - m_new) +
//             sum e^(x - m_new) — the running-max rescale of "Triton GPU
//             programming deep dive", section 3.3, over the chunks of the
//             "Level 2: Row Sum (tiling)" loop of the cs336 lecture 6 notes.
//   merge     warp (__shfl_xor), consumer warps (shared memory, a named
//             barrier), cluster: each CTA stores its (m, l) into every peer's
//             shared memory and arrives on the peer's exchange mbarrier
//             (release at cluster scope); each CTA waits on its own.  No
//             cluster-wide barrier per row, so the producer never stops.
//   pass 2    the slice's chunks again: y = e^(x - M) / L.
//
// Exchange slots and mbarriers are double-buffered by row parity: a CTA can
// run at most one row ahead of a peer (it needs the peer's partial of the
// row in between), so a slot is rewritten only after its reader is done.
// In place (in == out) is safe: each element is re-read by the thread that
// then writes it, and every first-pass read of a row precedes the exchange
// that any write of the row waits for.  The last chunk of a slice may be
// ragged: its final < 16 bytes are read with plain loads by the lane that
// owns them.
#include "cluster_ring.cuh"
#include "common.cuh"
#include "kernels.h"

#include <atomic>

namespace rwsm {

__device__ unsigned g_error_stream_rows = 0;

constexpr int kStreamMaxStages = 8;
constexpr int kStreamRingAlign = 128;
constexpr int kStreamMaxCluster = 16;

// CTAs per SM the register budget is set for: a consumer thread holds one
// chunk of E = NV * 16 / sizeof(T) floats plus about 40 registers of
// addresses and state (measured with -Xptxas -v).
template <typename T, int THREADS, int NV>
__host__ __device__ constexpr int stream_min_blocks()
{
    constexpr int b = 65536 / ((THREADS + 32) * (NV * Elem<T>::kVec16 + 40));
    return b < 1 ? 1 : b;
}

template <typename T, int THREADS, int NV, bool OUTVEC, bool OPTS>
__global__ void __launch_bounds__(THREADS + 32, (stream_min_blocks<T, THREADS, NV>()))
stream_rows_kernel(const T* in, T* out, int64_t n_rows, int64_t n_cols, int64_t ld_in,
                   int64_t ld_out, int64_t slice_cols, int cs, int stages, LogitsArg lg)
{
    constexpr int VEC = Elem<T>::kVec16;
    constexpr int NW = THREADS / 32;                    // consumer warps; warp NW produces
    constexpr int E = NV * VEC;
    constexpr int CHUNK = THREADS * E;                  // elements per chunk
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ float red_m[2][NW], red_l[2][NW];
    __shared__ __align__(8) float2 xpart[2][kStreamMaxCluster];
    __shared__ __align__(8) unsigned long long full[kStreamMaxStages];
    __shared__ __align__(8) unsigned long long empty[kStreamMaxStages];
    __shared__ __align__(8) unsigned long long xbar[2];
    __shared__ unsigned issued[kStreamMaxStages];
    __shared__ int s_failed;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float kk = OPTS ? lg.k : kLog2e;       // exponent multiplier, scale * log2 e
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;
    const int64_t c0 = static_cast<int64_t>(rank) * slice_cols;
    int64_t len = n_cols - c0;
    len = len < 0 ? 0 : (len > slice_cols ? slice_cols : len);
    const int64_t K = (len + CHUNK - 1) / CHUNK;        // chunks per pass
    const int64_t my_rows = cluster_id < n_rows ? (n_rows - 1 - cluster_id) / n_clusters + 1 : 0;

    T* ring = reinterpret_cast<T*>((reinterpret_cast<uintptr_t>(smem_raw) + (kStreamRingAlign - 1)) &
                                   ~static_cast<uintptr_t>(kStreamRingAlign - 1));
    auto stage_ptr = [&](int s) { return ring + static_cast<int64_t>(s) * CHUNK; };
    auto chunk_len = [&](int64_t chunk) {
        const int64_t rest = len - chunk * CHUNK;
        return static_cast<int>(rest < CHUNK ? rest : CHUNK);
    };
    // Columns of this slice that take part in `row` (all of them unless a
    // causal mask stops the row inside or before the slice), and of `chunk`
    // given that count (masked columns are never read).
    auto row_keep = [&](int64_t row) -> int64_t { return kept_cols<OPTS>(lg, row, n_cols) - c0; };
    auto chunk_lim = [&](int64_t keep, int64_t chunk) {
        const int64_t rest = keep - chunk * CHUNK;
        const int clen = chunk_len(chunk);
        return static_cast<int>(rest < 0 ? 0 : (rest > clen ? clen : rest));
    };
    // Bytes of `chunk` of `row` the bulk copy moves (whole 16-byte granules).
    auto copy_bytes = [&](int64_t row, int64_t chunk) -> uint32_t {
        if constexpr (OPTS)
            return span_copy_bytes<T>(chunk_lim(row_keep(row), chunk), n_cols - c0 - chunk * CHUNK);
        else
            return static_cast<uint32_t>(chunk_len(chunk) * sizeof(T)) & ~15u;
    };

    // Cluster launches let the next grid start only after the row loop:
    // clusters of the next grid placed early into leftover slots measured
    // slower.  Single-CTA launches let it start at once.
    if (cs == 1)
        pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), NW);
            issued[s] = 0;
        }
        mbar_init(smem_addr(&xbar[0]), static_cast<uint32_t>(cs));
        mbar_init(smem_addr(&xbar[1]), static_cast<uint32_t>(cs));
        s_failed = 0;
        fence_mbar_init();
        // The first row's first chunks into L2 while the preceding grid
        // drains (the grid is one resident wave; the copies after
        // griddepcontrol.wait still see the preceding grid's writes, L2
        // being the point of coherence).
        if (cluster_id < n_rows)
            for (int64_t chunk = 0; chunk < K && chunk < stages; ++chunk) {
                const uint32_t bytes = copy_bytes(cluster_id, chunk);
                if (bytes)
                    bulk_prefetch_l2(in + cluster_id * ld_in + c0 + chunk * CHUNK, bytes);
            }
    }
    // Peers arrive on this CTA's exchange mbarriers: they must be initialised
    // cluster-wide first.
    if (cs > 1)
        cluster_barrier();
    else
        __syncthreads();
    pdl_wait();

    if (warp == NW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t keep_pol = policy_evict_last();
            const uint64_t stream_pol = policy_evict_first();
            const int64_t total_q = my_rows * 2 * K;
            RingPos pos;
            int64_t chunk = 0, row = cluster_id;
            bool second = false;
            // The sequence: for each row, pass 1's K chunks, then pass 2's.
            for (int64_t q = 0; q < total_q; ++q) {
                const int s = pos.slot;
                // The stage's previous use (one trip earlier) must be released.
                if (q >= stages && !mbar_wait_bounded(smem_addr(&empty[s]), pos.phase ^ 1u)) {
                    *reinterpret_cast<volatile int*>(&s_failed) = 1;
                    break;
                }
                if (*reinterpret_cast<volatile int*>(&s_failed))
                    break;
                const uint32_t bytes = copy_bytes(row, chunk);
                const uint32_t bar = smem_addr(&full[s]);
                fence_proxy_async_smem();
                issued[s] += 1;
                if (bytes) {
                    mbar_arrive_expect_tx(bar, bytes);
                    bulk_g2s_hint(smem_addr(stage_ptr(s)), in + row * ld_in + c0 + chunk * CHUNK,
                                  bytes, bar, second ? stream_pol : keep_pol);
                } else {
                    mbar_arrive(bar);
                }
                pos.next(stages);
                if (++chunk == K) {
                    chunk = 0;
                    second = !second;
                    if (!second)
                        row += n_clusters;
                }
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- consumers
        const uint64_t stream_pol = policy_evict_first();
        bool failed = false;                             // warp-uniform
        RingPos cpos;                                    // next chunk's stage and phase
        // Wait for the next chunk of the sequence, copy this thread's vectors
        // into registers (the ragged tail from global memory, masked columns
        // as -inf) and hand the stage back to the producer.
        auto take = [&](int64_t keep, const T* src_row, int64_t chunk, float (&x)[E]) {
            const int s = cpos.slot;
            const bool ok = failed || mbar_wait_bounded(smem_addr(&full[s]), cpos.phase);
            cpos.next(stages);
            if (__any_sync(0xffffffffu, !ok) && !failed) {
                failed = true;
                *reinterpret_cast<volatile int*>(&s_failed) = 1;
            }
            int clen, bulk;                              // kept columns, copied columns
            if constexpr (OPTS) {
                clen = chunk_lim(keep, chunk);
                bulk = static_cast<int>(span_copy_bytes<T>(clen, n_cols - c0 - chunk * CHUNK) /
                                        sizeof(T));
                bulk = bulk < clen ? bulk : clen;
            } else {
                clen = chunk_len(chunk);
                bulk = static_cast<int>((clen * sizeof(T)) & ~size_t{15}) / static_cast<int>(sizeof(T));
            }
            const T* st = stage_ptr(s);
            const T* g = src_row + chunk * CHUNK;
            if (bulk == CHUNK) {                         // CTA-uniform: a whole chunk
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    lds_vec<T, VEC>(st + (tid + k * THREADS) * VEC, &x[k * VEC]);
            } else {
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int e0 = (tid + k * THREADS) * VEC;
                    if (e0 + VEC <= bulk) {
                        lds_vec<T, VEC>(st + e0, &x[k * VEC]);
                    } else if (e0 >= clen) {
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
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&empty[s]));       // stage free for the producer
        };
        int64_t i = 0;                                   // this cluster's row counter
        for (int64_t row = cluster_id; row < n_rows; row += n_clusters, ++i) {
            const T* src = in + row * ld_in + c0;
            T* dst = out + row * ld_out + c0;
            const int64_t keep = row_keep(row);
            // ---- pass 1: online (m, l) over the staged chunks
            float m = kNegInf, l = 0.0f;
            for (int64_t chunk = 0; chunk < K; ++chunk) {
                float x[E];
                take(keep, src, chunk, x);
                // Paired fp32 instructions (two results each, rounded as
                // the scalar ones) and a three-input max.
                const float mn = frag_max<E>(x, m);
                const float ref = (mn == kNegInf) ? 0.0f : mn;
                float s0 = 0.0f, s1 = 0.0f;
                frag_exp_acc<E>(x, ref, kk, s0, s1);
                l = l * exp_ftz(m - ref, kk) + (s0 + s1);
                m = mn;
            }
            // ---- merge over the consumer warps
            const int p = static_cast<int>(i & 1);
            warp_ml_merge(m, l, kk);
            if (lane == 0) {
                red_m[p][warp] = m;
                red_l[p][warp] = l;
            }
            named_barrier(1, THREADS);
            m = lane < NW ? red_m[p][lane] : kNegInf;
            l = lane < NW ? red_l[p][lane] : 0.0f;
            warp_ml_merge(m, l, kk);
            // ---- merge over the cluster (distributed shared memory)
            if (cs > 1) {
                if (tid == 0) {
                    const uint32_t slot = smem_addr(&xpart[p][rank]);
                    const uint32_t bar = smem_addr(&xbar[p]);
                    for (int r = 0; r < cs; ++r) {
                        st_cluster_f2(cluster_map(slot, static_cast<uint32_t>(r)), m, l);
                        mbar_arrive_cluster(cluster_map(bar, static_cast<uint32_t>(r)));
                    }
                }
                const bool ok = failed ||
                                mbar_wait_cluster_bounded(smem_addr(&xbar[p]),
                                                          static_cast<uint32_t>((i >> 1) & 1));
                if (__any_sync(0xffffffffu, !ok) && !failed) {
                    failed = true;
                    *reinterpret_cast<volatile int*>(&s_failed) = 1;
                }
                float pm = kNegInf, pl = 0.0f;
                if (lane < cs) {
                    const float2 v = xpart[p][lane];
                    pm = v.x;
                    pl = v.y;
                }
                warp_ml_merge(pm, pl, kk);
                m = pm;
                l = pl;
            }
            const float inv = 1.0f / l;
            // ---- pass 2: the staged chunks again (mostly L2 hits): normalise, store
            for (int64_t chunk = 0; chunk < K; ++chunk) {
                float x[E];
                take(keep, src, chunk, x);
                const int clen = chunk_len(chunk);
                T* d = dst + chunk * CHUNK;
                const bool whole = OUTVEC && clen == CHUNK;   // CTA-uniform
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int e0 = (tid + k * THREADS) * VEC;
                    if (whole || e0 < clen) {
                        // y = exp_biased(x - M) * (1 / L), two elements per
                        // instruction.
                        float* v = &x[k * VEC];
#pragma unroll
                        for (int j = 0; j < VEC; j += 2) {
                            float d0, d1;
                            add2(d0, d1, v[j], v[j + 1], -m, -m);
                            fma2(d0, d1, d0, d1, kk, kk, kExpBias, kExpBias);
                            mul2(v[j], v[j + 1], ex2_ftz(d0), ex2_ftz(d1), inv, inv);
                        }
                        if constexpr (OUTVEC) {
                            if (whole || e0 + VEC <= clen)
                                store16_hint<T>(d + e0, v, 1.0f, stream_pol);
                            else
                                store_vec_masked<T, VEC>(d, e0, clen, v, 1.0f);
                        } else {
#pragma unroll
                            for (int j = 0; j < VEC; ++j)
                                if (e0 + j < clen)
                                    Elem<T>::store1(d + e0 + j, v[j]);
                        }
                    }
                }
            }
        }
    }
    if (cs > 1)
        pdl_launch_dependents();
    // No CTA may exit while a peer can still write its shared memory.
    if (cs > 1)
        cluster_barrier();
    else
        __syncthreads();
    if (tid == THREADS && *reinterpret_cast<volatile int*>(&s_failed)) {
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
            q.blockDim = dim3(THREADS + 32, 1, 1);
            q.dynamicSmemBytes = static_cast<size_t>(smem);
            q.attrs = attr;
            q.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&active, k, &q) != cudaSuccess) {
                cudaGetLastError();
                active = 0;
            }
        } else {
            active = resident_ctas(reinterpret_cast<const void*>(k), THREADS + 32, smem);
        }
        if (active < 1)
            active = 1;
        const int sms = sm_count_current();
        if (cs == 1 && sms > 0 && active >= 2 * sms) {
            // Two or more CTAs share an SM: two waves, so that SMs whose
            // rows finish first take the remaining ones (a balanced single
            // wave can leave some SMs one CTA short: 4096 x 16384 fp32 on
            // 16 KB chunks 5091 GB/s, 6479 as two waves).
            clusters = p.n_rows < 2 * int64_t{active} ? p.n_rows : 2 * int64_t{active};
        } else {
            clusters = balanced_grid(p.n_rows, active, cs == 1 ? sms : 0);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
    cfg.blockDim = dim3(THREADS + 32, 1, 1);
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
    if (plan.stages < 1 || plan.stages > kStreamMaxStages || plan.cluster < 1 ||
        plan.cluster > kStreamMaxCluster)
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
