// WARP path, staged: short rows (<= 1024 columns) whose input rows are
// 16-byte aligned.  A persistent CTA of four warps walks tiles of R
// consecutive rows through a ring of `stages` shared-memory buffers:
//
//   ring    one elected thread starts one cp.async.bulk copy per row of a tile
//           (global -> shared, all completing on the stage's mbarrier).  A row
//           is copied up to the 16-byte granule holding its last kept column,
//           with its padding when that lies before the next row's start (the
//           padding and any masked columns copied are taken as -inf); only
//           the matrix's last row can leave a < 16-byte tail, read by the
//           lane that owns it with a plain load.
//   rows    each warp owns R/4 rows of the tile and reduces them one after the
//           other straight out of shared memory: lane l reads the vectors at
//           columns (c*32 + l)*VEC, then max (__shfl_xor), e = exp(x - max),
//           sum (__shfl_xor), y = e * (1/sum), coalesced stores.
//   refill  after a CTA barrier (every warp done with the tile) the stage is
//           refilled with the tile `stages` ahead.
//
// Shared memory, not registers, holds the rows in flight, so an SM keeps
// stages x R rows loading while its warps compute.  VEC is the width of the
// output stores: 16 bytes when the output rows are 16-byte aligned, else one
// element (then each store instruction of a warp writes 32 consecutive
// elements).  The softmax itself is the fused kernel of "Triton: write
// CUDA-grade GPU operators in Python", example 2, with -inf padding
// contributing 0 as in the cs336 lecture 6 notes, "Level 1: Softmax".
#include "common.cuh"
#include "kernels.h"

#include <atomic>

namespace rwsm {

__device__ unsigned g_error_tile_rows = 0;

constexpr int kTileWarps = 4;
constexpr int kTileThreads = kTileWarps * 32;
constexpr int kTileMaxStages = 8;
constexpr int kTileMaxRows = 64;             // rows per tile: 4 warps x up to 16 rows
constexpr int kTileRingAlign = 128;
constexpr int64_t kTileGridWaves = 4;       // most waves of resident CTAs launched

template <typename T, int VEC>
__device__ __forceinline__ void lds_any(const T* p, float* v)
{
    if constexpr (VEC == 1) {
        if constexpr (sizeof(T) == 4)
            v[0] = *reinterpret_cast<const float*>(p);
        else
            v[0] = Elem<T>::widen(*reinterpret_cast<const unsigned short*>(p));
    } else {
        lds_vec<T, VEC>(p, v);
    }
}

// At most 64 registers per thread (8 CTAs per SM): the kernel is latency
// bound, so resident warps matter more than registers (no spills at 64).
template <typename T, int VEC, int CHUNKS, bool OPTS>
__global__ void __launch_bounds__(kTileThreads, 8)
tile_rows_kernel(const T* in, T* out, int64_t n_rows, int n_cols, int64_t ld_in,
                 int64_t ld_out, int rows_per_warp, int stages, int row_pad, int64_t prefetch_ctas,
                 LogitsArg lg)
{
    constexpr int E = VEC * CHUNKS;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long full[kTileMaxStages];
    __shared__ unsigned issued[kTileMaxStages];
    // Options build: each row's kept and copied columns, written by the
    // issuing thread with the tile's copies (read after the stage's mbarrier
    // completes).
    __shared__ int2 row_keep[OPTS ? kTileMaxStages : 1][OPTS ? kTileMaxRows : 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float kk = OPTS ? lg.k : kLog2e;       // exponent multiplier, scale * log2 e
    const int R = kTileWarps * rows_per_warp;
    const int64_t n_tiles = (n_rows + R - 1) / R;
    // A row is copied up to the 16-byte granule that holds its last kept
    // column (all of it without a mask).  That granule may reach into the
    // row's padding (up to row_pad elements) when the row stride covers the
    // padding and another row follows.
    const bool pad_ok = ld_in >= row_pad;
    const uint32_t pad_bytes = static_cast<uint32_t>(row_pad * sizeof(T));
    // Plain build, rows packed (stride row_pad): one copy per tile for rows
    // under 2 KB or not a whole number of 128-byte lines (on GB300: 256
    // bf16 columns 4666 -> 5987 GB/s, 1000 columns 5830 -> 6090), one copy
    // per row otherwise (1024 bf16 columns: 6180 per row, 6120 per tile).
    const bool span_copy = !OPTS && ld_in == row_pad && (pad_bytes < 2048 || pad_bytes % 128 != 0);
    const uint32_t row_bytes = static_cast<uint32_t>(n_cols * sizeof(T)) & ~15u;
    auto copy_bytes = [&](int64_t row, int64_t lim) -> uint32_t {
        if constexpr (OPTS)
            return span_copy_bytes<T>(lim, pad_ok && row + 1 < n_rows ? row_pad : n_cols);
        else
            return pad_ok && row + 1 < n_rows ? pad_bytes : row_bytes;
    };

    T* ring = reinterpret_cast<T*>((reinterpret_cast<uintptr_t>(smem_raw) + (kTileRingAlign - 1)) &
                                   ~static_cast<uintptr_t>(kTileRingAlign - 1));
    auto row_ptr = [&](int s, int r) { return ring + (static_cast<int64_t>(s) * R + r) * row_pad; };
    auto issue = [&](int s, int64_t tile) {     // thread 0 only
        const uint32_t bar = smem_addr(&full[s]);
        const int64_t r0 = tile * R;
        const int nr = static_cast<int>(n_rows - r0 < R ? n_rows - r0 : R);
        fence_proxy_async_smem();
        issued[s] += 1;
        if constexpr (OPTS) {
            // One pass: each copy raises the phase's byte count before it
            // starts; the single arrival comes after the last copy.  The
            // tile's rows are consecutive: row r0's position in the mask
            // period (one division), then one step per row.
            uint64_t pos = lg.causal && nr > 0 ? logits_period_pos(lg, r0) : 0;
            for (int r = 0; r < nr; ++r) {
                int64_t lim = n_cols;
                if (lg.causal) {
                    lim = logits_lim(lg, pos, n_cols);
                    if (++pos == static_cast<uint64_t>(lg.period))
                        pos = 0;
                }
                const uint32_t n = copy_bytes(r0 + r, lim);
                row_keep[s][r] = make_int2(static_cast<int>(lim), static_cast<int>(n / sizeof(T)));
                if (n) {
                    mbar_expect_tx(bar, n);
                    bulk_g2s(smem_addr(row_ptr(s, r)), in + (r0 + r) * ld_in, n, bar);
                }
            }
            mbar_arrive(bar);
            return;
        }
        if (span_copy && nr > 0) {
            // Rows packed without padding: the tile is one span in memory and
            // in the stage (every row but the matrix's last copies its whole
            // row_pad), so one copy moves it.
            const uint32_t span = static_cast<uint32_t>(nr - 1) * pad_bytes + copy_bytes(r0 + nr - 1, n_cols);
            if (span) {
                mbar_arrive_expect_tx(bar, span);
                bulk_g2s(smem_addr(row_ptr(s, 0)), in + r0 * ld_in, span, bar);
            } else {
                mbar_arrive(bar);
            }
            return;
        }
        uint32_t total = 0;
        for (int r = 0; r < nr; ++r)
            total += copy_bytes(r0 + r, kept_cols<OPTS>(lg, r0 + r, n_cols));
        if (total) {
            mbar_arrive_expect_tx(bar, total);
            for (int r = 0; r < nr; ++r) {
                const uint32_t n = copy_bytes(r0 + r, kept_cols<OPTS>(lg, r0 + r, n_cols));
                if (n)
                    bulk_g2s(smem_addr(row_ptr(s, r)), in + (r0 + r) * ld_in, n, bar);
            }
        } else {
            mbar_arrive(bar);
        }
    };

    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            issued[s] = 0;
        }
        fence_mbar_init();
        // The first tiles' rows into L2 while the preceding grid drains (a
        // prefetch reads nothing into this CTA: the copies after
        // griddepcontrol.wait see the preceding grid's writes).  Only the
        // CTAs that can be resident before the preceding grid ends (the
        // first wave) do so; later waves copy at once.
        for (int s = 0; s < stages && static_cast<int64_t>(blockIdx.x) < prefetch_ctas; ++s) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (t >= n_tiles)
                break;
            const int64_t r0 = t * R;
            const int nr = static_cast<int>(n_rows - r0 < R ? n_rows - r0 : R);
            if (!OPTS && span_copy) {
                const uint32_t span = static_cast<uint32_t>(nr - 1) * pad_bytes + copy_bytes(r0 + nr - 1, n_cols);
                if (span)
                    bulk_prefetch_l2(in + r0 * ld_in, span);
                continue;
            }
            uint64_t pos = OPTS && lg.causal ? logits_period_pos(lg, r0) : 0;
            for (int r = 0; r < nr; ++r) {
                int64_t lim = n_cols;
                if (OPTS && lg.causal) {
                    lim = logits_lim(lg, pos, n_cols);
                    if (++pos == static_cast<uint64_t>(lg.period))
                        pos = 0;
                }
                const uint32_t n = copy_bytes(r0 + r, lim);
                if (n)
                    bulk_prefetch_l2(in + (r0 + r) * ld_in, n);
            }
        }
    }
    __syncthreads();
    pdl_wait();
    if (tid == 0)
        for (int s = 0; s < stages; ++s) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(s) * gridDim.x;
            if (t < n_tiles)
                issue(s, t);
        }

    bool failed = false;                         // CTA-uniform
    // Ring stage of the current tile and its phase parity, advanced per tile
    // (no 64-bit division).
    int s = 0;
    uint32_t parity = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const bool ok = failed ? true : mbar_wait_bounded(smem_addr(&full[s]), parity);
        for (int rr = 0; rr < rows_per_warp; ++rr) {
            const int r = warp * rows_per_warp + rr;
            const int64_t row = tile * R + r;
            if (row >= n_rows)
                break;                           // warp-uniform
            const T* sp = row_ptr(s, r);
            const T* gp = in + row * ld_in;
            // Columns [0, avail) are in shared memory, [avail, lim) is a
            // < 16-byte tail read from HBM, and from lim on the row is masked
            // or padding (-inf).
            int lim, copied;
            if constexpr (OPTS) {
                const int2 kc = row_keep[s][r];          // kept and copied columns
                lim = kc.x;
                copied = kc.y;
            } else {
                lim = n_cols;
                copied = static_cast<int>(copy_bytes(row, lim) / sizeof(T));
            }
            const int avail = copied < lim ? copied : lim;
            // Whole vectors first: a vector that starts below `avail` is read
            // from shared memory (inside the row's ring slot), any other is
            // -inf.  Only a row whose edges do not fall on vector boundaries
            // needs the per-element fix-up of its edge vectors.
            float x[E];
#pragma unroll
            for (int c = 0; c < CHUNKS; ++c) {
                const int col = (c * 32 + lane) * VEC;
                if (col < avail) {
                    lds_any<T, VEC>(sp + col, &x[c * VEC]);
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        x[c * VEC + j] = kNegInf;
                }
            }
            if (OPTS && avail == lim && lim % VEC != 0) {              // warp-uniform
                // Only the vector holding column lim - 1 straddles the edge
                // (one lane, one chunk): its copied elements past lim are
                // masked; vectors wholly past lim are already -inf.
#pragma unroll
                for (int c = 0; c < CHUNKS; ++c) {
                    const int keep_n = lim - (c * 32 + lane) * VEC;
                    if (keep_n > 0 && keep_n < VEC) {
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            x[c * VEC + j] = j < keep_n ? x[c * VEC + j] : kNegInf;
                    }
                }
            } else if ((avail | lim) % VEC != 0 || avail < lim) {   // warp-uniform
#pragma unroll
                for (int c = 0; c < CHUNKS; ++c) {
                    const int col = (c * 32 + lane) * VEC;
                    if (col + VEC > avail && col < lim) {
#pragma unroll
                        for (int j = 0; j < VEC; ++j) {
                            const int e = col + j;
                            if (e >= avail)
                                x[c * VEC + j] = e < lim ? Elem<T>::load1(gp + e) : kNegInf;
                        }
                    }
                }
            }
            float m = kNegInf;
            if constexpr (OPTS) {
                m = frag_max<E>(x, kNegInf);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    m = fmaxf(m, x[e]);
            }
            m = warp_max_redux(m);
            // exp_biased and the sum.  With options: two elements per
            // instruction, and chunks wholly past `lim` are 0 without
            // computing.  (The plain rows measured faster with scalar math.)
            float s0 = 0.0f, s1 = 0.0f;
            if constexpr (OPTS && E % 2 == 0) {
#pragma unroll
                for (int i = 0; i < E; i += 2) {
                    if (!OPTS || ((i / VEC) * 32 * VEC < lim))          // warp-uniform
                        frag_exp_acc<2>(&x[i], m, kk, s0, s1);
                    else
                        x[i] = x[i + 1] = 0.0f;
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    x[e] = exp_biased(x[e] - m, kk);
                    s0 += x[e];
                }
            }
            const float inv = 1.0f / warp_sum(s0 + s1);
            T* dst = out + row * ld_out;
            if (OPTS && n_cols % VEC == 0) {                        // kernel-uniform
#pragma unroll
                for (int c = 0; c < CHUNKS; ++c) {
                    const int col = (c * 32 + lane) * VEC;
                    if (col < n_cols) {
                        if constexpr (VEC % 2 == 0)
                            store_vec2<T, VEC>(dst + col, &x[c * VEC], inv);
                        else
                            store_vec<T, VEC>(dst + col, &x[c * VEC], inv);
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < CHUNKS; ++c)
                    store_vec_masked<T, VEC>(dst, (c * 32 + lane) * VEC, n_cols, &x[c * VEC], inv);
            }
        }
        if (__syncthreads_or(!ok))
            failed = true;
        if (tid == 0 && !failed) {
            const int64_t next = tile + static_cast<int64_t>(stages) * gridDim.x;
            if (next < n_tiles)
                issue(s, next);
        }
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (failed && tid == 0) {
        atomicOr(&g_error_tile_rows, kErrMbarrierTimeout);
        for (int s = 0; s < stages; ++s)
            if (issued[s])
                mbar_wait_bounded(smem_addr(&full[s]), (issued[s] - 1) & 1u);
    }
}

// ------------------------------------------------------------------ host side

unsigned read_error_tile_rows(bool clear)
{
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_tile_rows, sizeof v) != cudaSuccess)
        return 0;
    if (clear && v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_error_tile_rows, &zero, sizeof zero);
    }
    return v;
}

namespace {

constexpr int kMaxDevices = 64;

template <typename T, int VEC, int CHUNKS, bool OPTS>
cudaError_t launch_tile_opts(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    auto* k = tile_rows_kernel<T, VEC, CHUNKS, OPTS>;
    static std::atomic<int> smem_set[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int smem = plan.smem_bytes + kTileRingAlign;
    if (smem_set[dev].load() < smem) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess)
            return err;
        cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        smem_set[dev].store(smem);
    }
    const int64_t R = int64_t{kTileWarps} * plan.rows_per_warp;
    const int64_t tiles = (p.n_rows + R - 1) / R;
    int64_t grid = plan.grid;
    const int64_t resident = resident_ctas(reinterpret_cast<const void*>(k), kTileThreads, smem);
    if (grid <= 0) {
        // Latency-bound (a warp reduces its rows one after another): every
        // resident CTA is worth more than a fuller last round.  Inputs of at
        // least eight tiles per resident CTA launch four whole waves of CTAs:
        // CTAs that finish early are replaced, so the last tiles spread over
        // every SM.  Measured against one wave on GB300: 65536 x 1024 bf16
        // 5690 -> 6360 GB/s, 131072 x 512 bf16 5485 -> 6030, 262144 x 256
        // bf16 4100 -> 4700.  Smaller inputs keep one wave: 32768 x 1024
        // causal bf16 (6.7 tiles per CTA) measured 5830 at one wave, 5690 at
        // two and 5050 at 1.12 (a partial wave runs its full shares alone).
        const int64_t waves = resident > 0 && tiles >= 8 * resident ? kTileGridWaves : 1;
        grid = tiles < waves * resident ? tiles : waves * resident;
    }
    if (grid < 1)
        grid = 1;
    const int row_pad = static_cast<int>(plan.slice_cols);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kTileThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, 1));
    err = cudaLaunchKernelEx(&cfg, k, static_cast<const T*>(p.in), static_cast<T*>(p.out),
                             p.n_rows, static_cast<int>(p.n_cols), p.ld_in, p.ld_out,
                             plan.rows_per_warp, plan.stages, row_pad, resident, logits_of(p));
    note_launch();
    return err;
}

template <typename T, int VEC, int CHUNKS>
cudaError_t launch_tile(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    return has_options(p) ? launch_tile_opts<T, VEC, CHUNKS, true>(p, plan, s)
                    : launch_tile_opts<T, VEC, CHUNKS, false>(p, plan, s);
}

template <typename T, int VEC>
cudaError_t launch_chunks(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    switch (plan.chunks) {
    case 1: return launch_tile<T, VEC, 1>(p, plan, s);
    case 2: return launch_tile<T, VEC, 2>(p, plan, s);
    case 4: return launch_tile<T, VEC, 4>(p, plan, s);
    case 8:
        if constexpr (VEC * 8 <= 32) return launch_tile<T, VEC, 8>(p, plan, s);
        break;
    case 16:
        if constexpr (VEC * 16 <= 32) return launch_tile<T, VEC, 16>(p, plan, s);
        break;
    case 32:
        if constexpr (VEC * 32 <= 32) return launch_tile<T, VEC, 32>(p, plan, s);
        break;
    default:
        break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_tile_rows(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    if (plan.stages < 1 || plan.stages > kTileMaxStages || plan.rows_per_warp < 1 ||
        plan.rows_per_warp * kTileWarps > kTileMaxRows)
        return cudaErrorInvalidValue;
    if (p.dtype == SOFTMAX_F32) {
        if (plan.vec == 4) return launch_chunks<float, 4>(p, plan, s);
        if (plan.vec == 1) return launch_chunks<float, 1>(p, plan, s);
    } else if (p.dtype == SOFTMAX_BF16) {
        if (plan.vec == 8) return launch_chunks<BF16Bits, 8>(p, plan, s);
        if (plan.vec == 1) return launch_chunks<BF16Bits, 1>(p, plan, s);
    } else {
        if (plan.vec == 8) return launch_chunks<F16Bits, 8>(p, plan, s);
        if (plan.vec == 1) return launch_chunks<F16Bits, 1>(p, plan, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace rwsm
