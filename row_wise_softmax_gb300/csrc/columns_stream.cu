// Column-wise softmax, staged: the softmax runs down the columns of a
// row-major matrix (unit row strides in softmax_strided terms), as in the
// cs336 lecture 6 notes ("Level 1: Softmax": a column-wise softmax changes
// only the strides).  Adjacent softmax rows are adjacent in memory, so a tile
// of W of them is a column of segments of W elements, one per memory row.
//
//   producer  the last warp of the CTA (one elected lane) streams 16 KB boxes
//             (a tile's segments of consecutive memory rows) with the tensor memory
//             accelerator (cp.async.bulk.tensor.2d) into a ring of `stages`
//             shared-memory buffers, along the sequence (tile, pass, box):
//             first-pass boxes with an L2 evict-last policy, second-pass boxes
//             with evict-first.
//   pass 1    lane l of every consumer warp owns softmax rows W/32 * l ..;
//             warp w folds memory rows w, w + 8, ... of each box into an
//             online (m, l) per softmax row (the running-max rescale of
//             "Triton GPU programming deep dive", section 3.3).
//   merge     the consumer warps' partials in shared memory, then the CTAs of
//             the cluster (each splits the memory rows): every lane of warp 0
//             stores its rows' (m, l) into every peer's shared memory and
//             arrives on the peer's exchange mbarrier; each CTA waits on its
//             own (release / acquire at cluster scope).
//   pass 2    the boxes again (mostly L2 hits): y = e^(x - M) / L, written as
//             one segment per memory row per warp instruction.
//
// One HBM read and one write per element when the second read hits L2.
// Memory rows past the CTA's range (a box may overhang it) and softmax rows
// past n_s (zero-filled by the copy engine) never reach a result or memory.
// In place (in == out, same layout) is safe: a tile's elements are all read
// by their CTA's first pass before any CTA of the cluster passes the exchange
// and writes them, and every other tile's columns are disjoint.
#include "cluster_ring.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tensor_map.h"

#include <atomic>

namespace rwsm {

__device__ unsigned g_error_columns_stream = 0;

namespace {

constexpr int kColThreads2 = 256;            // consumer threads (+ one producer warp)
constexpr int kColBoxBytes = 16384;           // one box: 16 KB
constexpr int kColMaxStages = 8;
constexpr int kColMaxCluster = 8;
constexpr int kColRingAlign = 1024;

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

template <typename T, int ROW_BYTES, bool VEC_STORES>
__global__ void __launch_bounds__(kColThreads2 + 32, 2)
columns_stream_kernel(const __grid_constant__ CUtensorMap map, T* out, int64_t n_s, int64_t n_l,
                      int64_t ld_out, int64_t rows_per_cta, int cs, int stages)
{
    constexpr int ESZ = static_cast<int>(sizeof(T));
    constexpr int W = ROW_BYTES / ESZ;          // softmax rows per tile
    constexpr int CPT = W / 32;                 // softmax rows per lane (adjacent)
    constexpr int LB = CPT * ESZ;               // bytes a lane reads per memory row
    constexpr int NW = kColThreads2 / 32;       // consumer warps; warp NW produces
    constexpr int B = kColBoxBytes / ROW_BYTES; // memory rows per box
    constexpr int RPW = B / NW;                 // memory rows of a box per warp
    static_assert(LB == 4 || LB == 8 || LB == 16, "lane vector");
    static_assert(RPW % 2 == 0, "paired arithmetic over a box's rows");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ float red_m[NW][W], red_l[NW][W];
    __shared__ __align__(8) unsigned long long full[kColMaxStages];
    __shared__ __align__(8) unsigned long long empty[kColMaxStages];
    __shared__ __align__(8) unsigned long long xbar[2];
    __shared__ unsigned issued[kColMaxStages];
    __shared__ int s_failed;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = static_cast<int>(blockIdx.x % cs);
    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;
    const int64_t r0 = static_cast<int64_t>(rank) * rows_per_cta;
    int64_t len = n_l - r0;                             // memory rows of this CTA
    len = len < 0 ? 0 : (len > rows_per_cta ? rows_per_cta : len);
    const int64_t K = (len + B - 1) / B;                // boxes per pass
    const int64_t n_tiles = (n_s + W - 1) / W;
    const int64_t my_tiles = cluster_id < n_tiles ? (n_tiles - 1 - cluster_id) / n_clusters + 1 : 0;

    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + (kColRingAlign - 1)) &
        ~static_cast<uintptr_t>(kColRingAlign - 1));
    // Exchange slots after the ring: [2][cs][W] (m, l) pairs, by tile parity.
    float2* xpart = reinterpret_cast<float2*>(ring + static_cast<size_t>(stages) * kColBoxBytes);
    auto slot = [&](int par, int r, int col) { return xpart + (par * cs + r) * W + col; };

    if (cs == 1)
        pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), NW);
            issued[s] = 0;
        }
        mbar_init(smem_addr(&xbar[0]), static_cast<uint32_t>(32 * cs));
        mbar_init(smem_addr(&xbar[1]), static_cast<uint32_t>(32 * cs));
        s_failed = 0;
        fence_mbar_init();
    }
    // Peers arrive on this CTA's exchange mbarriers: initialised cluster-wide
    // first.  (The launch always carries a cluster dimension, 1 included.)
    cluster_barrier();
    pdl_wait();

    if (warp == NW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&map)) : "memory");
            const uint64_t keep_pol = policy_evict_last();
            const uint64_t stream_pol = policy_evict_first();
            const int64_t total_q = my_tiles * 2 * K;
            RingPos pos;
            int64_t box = 0, tile = cluster_id;
            bool second = false;
            for (int64_t q = 0; q < total_q; ++q) {
                const int s = pos.slot;
                if (q >= stages && !mbar_wait_bounded(smem_addr(&empty[s]), pos.phase ^ 1u)) {
                    *reinterpret_cast<volatile int*>(&s_failed) = 1;
                    break;
                }
                if (*reinterpret_cast<volatile int*>(&s_failed))
                    break;
                const uint32_t bar = smem_addr(&full[s]);
                fence_proxy_async_smem();
                issued[s] += 1;
                mbar_arrive_expect_tx(bar, kColBoxBytes);
                tma_load_2d(smem_addr(ring + static_cast<size_t>(s) * kColBoxBytes), &map,
                            static_cast<int>(tile * W), static_cast<int>(r0 + box * B), bar,
                            second ? stream_pol : keep_pol);
                pos.next(stages);
                if (++box == K) {
                    box = 0;
                    second = !second;
                    if (!second)
                        tile += n_clusters;
                }
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- consumers
        const uint64_t stream_pol = policy_evict_first();
        bool failed = false;                             // warp-uniform
        RingPos cpos;
        auto wait_full = [&]() {
            const int s = cpos.slot;
            const bool ok = failed || mbar_wait_bounded(smem_addr(&full[s]), cpos.phase);
            if (__any_sync(0xffffffffu, !ok) && !failed) {
                failed = true;
                *reinterpret_cast<volatile int*>(&s_failed) = 1;
            }
            cpos.next(stages);
            return s;
        };
        auto release = [&](int s) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&empty[s]));
        };
        // This lane's CPT values of memory row `row` of the box in stage s
        // (bytes [lane * LB, lane * LB + LB) of the row).
        auto read_row = [&](int s, int row, float (&v)[CPT]) {
            const unsigned char* a = ring + static_cast<size_t>(s) * kColBoxBytes +
                                     row * ROW_BYTES + lane * LB;
            uint32_t w[LB / 4];
            if constexpr (LB == 16) {
                const uint4 q = *reinterpret_cast<const uint4*>(a);
                w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
            } else if constexpr (LB == 8) {
                const uint2 q = *reinterpret_cast<const uint2*>(a);
                w[0] = q.x; w[1] = q.y;
            } else {
                w[0] = *reinterpret_cast<const uint32_t*>(a);
            }
            if constexpr (ESZ == 4) {
#pragma unroll
                for (int c = 0; c < CPT; ++c)
                    v[c] = __uint_as_float(w[c]);
            } else {
#pragma unroll
                for (int c = 0; c < CPT / 2; ++c)
                    Elem<T>::unpack2(w[c], v[2 * c], v[2 * c + 1]);
            }
        };
        int64_t i = 0;                                   // this cluster's tile counter
        for (int64_t tile = cluster_id; tile < n_tiles; tile += n_clusters, ++i) {
            // ---- pass 1: online (m, l) per softmax row of this lane
            float m[CPT], l[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                m[c] = kNegInf;
                l[c] = 0.0f;
            }
            for (int64_t b = 0; b < K; ++b) {
                const int s = wait_full();
                const int64_t valid = len - b * B;       // rows of this box in the slice
                float x[RPW][CPT];
#pragma unroll
                for (int k = 0; k < RPW; ++k)
                    read_row(s, warp + k * NW, x[k]);
                if (valid < B) {                         // CTA-uniform: only a slice's last box
#pragma unroll
                    for (int k = 0; k < RPW; ++k)
                        if (warp + k * NW >= valid) {
#pragma unroll
                            for (int c = 0; c < CPT; ++c)
                                x[k][c] = kNegInf;
                        }
                }
                release(s);
                // Per softmax row: the box's RPW values, two per paired fp32
                // instruction (rounded as the scalar ones), three-input max.
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    float v[RPW];
#pragma unroll
                    for (int k = 0; k < RPW; ++k)
                        v[k] = x[k][c];
                    const float bm = frag_max<RPW>(v, m[c]);
                    const float ref = (bm == kNegInf) ? 0.0f : bm;
                    float s0 = 0.0f, s1 = 0.0f;
                    frag_exp_acc<RPW>(v, ref, kLog2e, s0, s1);
                    l[c] = l[c] * exp_ftz(m[c] - ref, kLog2e) + (s0 + s1);
                    m[c] = bm;
                }
            }
            // ---- merge over the consumer warps (shared memory)
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                red_m[warp][lane * CPT + c] = m[c];
                red_l[warp][lane * CPT + c] = l[c];
            }
            named_barrier(1, kColThreads2);
            const int p = static_cast<int>(i & 1);
            if (warp == 0) {
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    float mm = red_m[0][lane * CPT + c], ll = red_l[0][lane * CPT + c];
#pragma unroll
                    for (int w = 1; w < NW; ++w)
                        ml_merge(mm, ll, red_m[w][lane * CPT + c], red_l[w][lane * CPT + c], kLog2e);
                    m[c] = mm;
                    l[c] = ll;
                }
                // ---- to every CTA of the cluster (itself included)
                for (int r = 0; r < cs; ++r) {
#pragma unroll
                    for (int c = 0; c < CPT; ++c)
                        st_cluster_f2(cluster_map(smem_addr(slot(p, rank, lane * CPT + c)),
                                                  static_cast<uint32_t>(r)), m[c], l[c]);
                    mbar_arrive_cluster(cluster_map(smem_addr(&xbar[p]), static_cast<uint32_t>(r)));
                }
            }
            const bool ok = failed ||
                            mbar_wait_cluster_bounded(smem_addr(&xbar[p]), static_cast<uint32_t>((i >> 1) & 1));
            if (__any_sync(0xffffffffu, !ok) && !failed) {
                failed = true;
                *reinterpret_cast<volatile int*>(&s_failed) = 1;
            }
            float inv[CPT];
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                float mm = kNegInf, ll = 0.0f;
                for (int r = 0; r < cs; ++r) {
                    const float2 v = *slot(p, r, lane * CPT + c);
                    ml_merge(mm, ll, v.x, v.y, kLog2e);
                }
                m[c] = mm;
                inv[c] = 1.0f / ll;
            }
            // ---- pass 2: normalise and write the 128-byte segments
            const int64_t col0 = tile * W + lane * CPT;      // this lane's first softmax row
            for (int64_t b = 0; b < K; ++b) {
                const int s = wait_full();
                const int64_t valid = len - b * B;
                float x[RPW][CPT];
#pragma unroll
                for (int k = 0; k < RPW; ++k)
                    read_row(s, warp + k * NW, x[k]);
                release(s);
                // Memory row warp + k * NW of the box: advance by NW rows.
                T* dst = out + (r0 + b * B + warp) * ld_out + col0;
                const int64_t step = static_cast<int64_t>(NW) * ld_out;
#pragma unroll
                for (int k = 0; k < RPW; ++k, dst += step) {
                    if (valid < B && warp + k * NW >= valid)
                        continue;
                    float y[CPT];
                    if constexpr (CPT % 2 == 0) {
#pragma unroll
                        for (int c = 0; c < CPT; c += 2) {
                            float d0, d1;
                            add2(d0, d1, x[k][c], x[k][c + 1], -m[c], -m[c + 1]);
                            fma2(d0, d1, d0, d1, kLog2e, kLog2e, kExpBias, kExpBias);
                            mul2(y[c], y[c + 1], ex2_ftz(d0), ex2_ftz(d1), inv[c], inv[c + 1]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < CPT; ++c)
                            y[c] = exp_biased(x[k][c] - m[c], kLog2e) * inv[c];
                    }
                    if (VEC_STORES && col0 + CPT <= n_s) {
                        // LB bytes in one store, evict-first.
                        uint32_t w[LB / 4];
                        if constexpr (ESZ == 4) {
#pragma unroll
                            for (int c = 0; c < CPT; ++c)
                                w[c] = __float_as_uint(y[c]);
                        } else {
#pragma unroll
                            for (int c = 0; c < CPT / 2; ++c)
                                w[c] = Elem<T>::pack2(y[2 * c], y[2 * c + 1]);
                        }
                        if constexpr (LB == 16)
                            asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                                         :: "l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]),
                                            "l"(stream_pol) : "memory");
                        else if constexpr (LB == 8)
                            asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;"
                                         :: "l"(dst), "r"(w[0]), "r"(w[1]), "l"(stream_pol) : "memory");
                        else
                            asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;"
                                         :: "l"(dst), "r"(w[0]), "l"(stream_pol) : "memory");
                    } else {
#pragma unroll
                        for (int c = 0; c < CPT; ++c)
                            if (col0 + c < n_s)
                                Elem<T>::store1(dst + c, y[c]);
                    }
                }
            }
        }
    }
    if (cs > 1)
        pdl_launch_dependents();
    // No CTA may exit while a peer can still write its shared memory.
    cluster_barrier();
    if (tid == kColThreads2 && *reinterpret_cast<volatile int*>(&s_failed)) {
        atomicOr(&g_error_columns_stream, kErrMbarrierTimeout);
        for (int s = 0; s < stages; ++s)                  // copies possibly still in flight
            if (issued[s])
                mbar_wait_bounded(smem_addr(&full[s]), (issued[s] - 1) & 1u);
    }
}

constexpr int kMaxDevices = 64;

template <typename T, int ROW_BYTES, bool VEC>
cudaError_t launch_cs(const StridedProblem& p, const ColumnsShape& sh, const CUtensorMap& map,
                      cudaStream_t s)
{
    auto* k = columns_stream_kernel<T, ROW_BYTES, VEC>;
    static std::atomic<int> smem_set[kMaxDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int smem = sh.smem_bytes + kColRingAlign;     // ring + exchange slots + alignment
    if (smem_set[dev].load() < smem) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess)
            return err;
        cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        smem_set[dev].store(smem);
    }
    constexpr int BLOCK = kColThreads2 + 32;
    const int cs = sh.cluster;
    // An explicit cluster dimension even for one CTA: the kernel's exchange
    // addresses the CTAs of its cluster.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    const int n_attr = 2;
    int64_t clusters = 0;
    {
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
        q.blockDim = dim3(BLOCK, 1, 1);
        q.dynamicSmemBytes = static_cast<size_t>(smem);
        q.attrs = attr;
        q.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, k, &q) != cudaSuccess) {
            cudaGetLastError();
            active = 0;
        }
        clusters = active;
    }
    if (clusters < 1)
        clusters = 1;
    clusters = balanced_grid(sh.tiles, clusters, cs == 1 ? sm_count_current() : 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
    cfg.blockDim = dim3(BLOCK, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(n_attr);
    err = cudaLaunchKernelEx(&cfg, k, map, static_cast<T*>(p.out), p.n_rows, p.n_cols,
                             p.out_col_stride, static_cast<int64_t>(sh.rows_per_cta), cs,
                             sh.stages);
    note_launch();
    return err;
}

template <int RB>
cudaError_t launch_rb(const StridedProblem& p, const ColumnsShape& sh, const CUtensorMap& map,
                      cudaStream_t s)
{
    if (p.dtype == SOFTMAX_F32)
        return sh.vec_out ? launch_cs<float, RB, true>(p, sh, map, s)
                          : launch_cs<float, RB, false>(p, sh, map, s);
    if (p.dtype == SOFTMAX_BF16)
        return sh.vec_out ? launch_cs<BF16Bits, RB, true>(p, sh, map, s)
                          : launch_cs<BF16Bits, RB, false>(p, sh, map, s);
    return sh.vec_out ? launch_cs<F16Bits, RB, true>(p, sh, map, s)
                      : launch_cs<F16Bits, RB, false>(p, sh, map, s);
}

}  // namespace

// Shape of the staged columns kernel, or ok = false when the input cannot be
// described to the tensor memory accelerator (16-byte aligned base and memory
// row pitch, at most 2^31 - 1 rows and columns, rows not overlapping).
ColumnsShape columns_stream_shape(const StridedProblem& p, int sm_count, int max_smem_per_sm)
{
    ColumnsShape sh{};
    const int64_t esz = p.dtype == SOFTMAX_F32 ? 4 : 2;
    if (p.in_row_stride != 1 || p.out_row_stride != 1 || p.n_rows < 1 || p.n_cols < 1)
        return sh;
    if (reinterpret_cast<uintptr_t>(p.in) % 16 || (p.in_col_stride * esz) % 16 ||
        p.in_col_stride < p.n_rows || p.in_col_stride * esz >= (int64_t{1} << 40) ||
        p.n_rows >= (int64_t{1} << 31) || p.n_cols >= (int64_t{1} << 31))
        return sh;
    if (p.n_cols > 1 && p.out_col_stride < p.n_rows)
        return sh;
    if (!tensor_map_encoder())
        return sh;
    // Tiles 256 bytes wide, or 128 when wider tiles would leave fewer CTAs
    // than SMs even on clusters of 8 (measured on GB300: 32768 x 1024 fp32
    // 2656 -> 3174 GB/s; 8192 x 4096 bf16 keeps 256).
    const int rb = (p.n_rows * esz + 255) / 256 * kColMaxCluster < sm_count ? 128 : 256;
    const int64_t w = rb / esz;
    const int64_t box_rows = kColBoxBytes / rb;
    const int64_t tiles = (p.n_rows + w - 1) / w;
    const int64_t col_bytes = p.n_cols * rb;             // one tile's memory rows
    // Slices of about 256 KB on clusters of up to 4 CTAs, and larger
    // clusters (slices of at least 64 KB) while there are too few CTAs.
    int64_t cs = 1;
    while (cs < kColMaxCluster && (col_bytes > cs * 256 * 1024 ||
                                   (tiles * cs < sm_count && col_bytes / (2 * cs) >= 64 * 1024)))
        cs *= 2;
    int64_t rows = (p.n_cols + cs - 1) / cs;
    rows = (rows + box_rows - 1) / box_rows * box_rows;
    // Two CTAs per SM: ring, exchange slots, alignment slack, the static
    // shared memory and the 1 KB the runtime reserves per CTA.
    const int64_t xpart_bytes = 2 * cs * w * 8;
    const int64_t static_bytes = w * 2 * 8 * 4 + 512;
    int stages = 6;                                      // 96 KB ring
    while (stages > 2 && 2 * (stages * kColBoxBytes + xpart_bytes + kColRingAlign + static_bytes +
                              1024) > max_smem_per_sm)
        --stages;
    sh.ok = true;
    sh.stream = true;
    sh.row_bytes = rb;
    sh.cluster = static_cast<int>(cs);
    sh.rows_per_cta = static_cast<int>(rows);
    sh.stages = stages;
    sh.smem_bytes = static_cast<int>(stages * kColBoxBytes + xpart_bytes);
    sh.tiles = tiles;
    sh.vec_in = true;
    const int64_t lane_bytes = rb / 32;
    sh.vec_out = reinterpret_cast<uintptr_t>(p.out) % lane_bytes == 0 &&
                 (p.out_col_stride * esz) % lane_bytes == 0;
    return sh;
}

cudaError_t launch_columns_stream(const StridedProblem& p, const ColumnsShape& sh, cudaStream_t s)
{
    auto encode = tensor_map_encoder();
    const int64_t esz = p.dtype == SOFTMAX_F32 ? 4 : 2;
    if (!encode || (sh.row_bytes != 128 && sh.row_bytes != 256 && sh.row_bytes != 512) ||
        sh.stages < 1 || sh.stages > kColMaxStages || sh.cluster < 1 ||
        sh.cluster > kColMaxCluster || sh.rows_per_cta % (kColBoxBytes / sh.row_bytes) ||
        sh.smem_bytes < sh.stages * kColBoxBytes + 2 * sh.cluster * (sh.row_bytes / esz) * 8 ||
        static_cast<int64_t>(sh.rows_per_cta) * sh.cluster < p.n_cols)
        return cudaErrorInvalidValue;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.n_rows), static_cast<cuuint64_t>(p.n_cols)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.in_col_stride * esz)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(sh.row_bytes / esz),
                               static_cast<cuuint32_t>(kColBoxBytes / sh.row_bytes)};
    const cuuint32_t estride[2] = {1, 1};
    const CUtensorMapDataType dt = p.dtype == SOFTMAX_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : p.dtype == SOFTMAX_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (encode(&map, dt, 2, const_cast<void*>(p.in), dims, strides, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    switch (sh.row_bytes) {
    case 128: return launch_rb<128>(p, sh, map, s);
    case 256: return launch_rb<256>(p, sh, map, s);
    case 512: return launch_rb<512>(p, sh, map, s);
    default: return cudaErrorInvalidValue;
    }
}

unsigned read_error_columns_stream(bool clear)
{
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_columns_stream, sizeof v) != cudaSuccess)
        return 0;
    if (clear && v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_error_columns_stream, &zero, sizeof zero);
    }
    return v;
}

}  // namespace rwsm
