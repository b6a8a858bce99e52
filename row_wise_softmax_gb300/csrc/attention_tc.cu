// Attention forward on the fifth-generation tensor cores (tcgen05, sm_100
// family): the same online softmax as attention_mma.cu ("Triton GPU
// programming deep dive", section 3.3), with both products issued by one
// thread as tcgen05.mma and accumulated in tensor memory (TMEM).  Two
// kernels:
//
// attention_pp_kernel (the library's choice): a CTA owns two 128-query tiles
// A and B and ping-pongs them, so that one tile's softmax runs while the
// tensor cores compute the other's products.  One warp's lane 0 issues every
// tensor-map copy (Q once; K and V tiles of 128 keys through a ring of 2
// slots at head_dim 128, of 64 keys through 4 slots at 64, all with the
// 128-byte swizzle), another's
// every product; two warpgroups run the softmax, one per tile, and keep P in
// tensor memory.  The protocol is described beside the kernel.
//
// attention_tc_kernel, one tile per CTA:
//
//   CTA      128 queries of one (batch, head), 4 warps; thread t of warp w
//            owns query row 32w + t, which is TMEM lane 32w + t of every
//            accumulator.
//   TMEM     256 columns: S (one tile of keys) at column 0, O (head_dim) at
//            128.
//   staging  Q once, K and V tiles of 64 keys by cp.async, double-buffered
//            (the next tile loads while this one is computed), written in the
//            tensor cores' canonical layout without swizzle: 8 x 8 "core
//            matrices" of 128 contiguous bytes.  Q, K and P are K-major (rows
//            of 8 elements along the reduced dimension in a core matrix);
//            V is the B operand of P V with its rows along N = head_dim, i.e.
//            MN-major.
//   per tile S = Q K^T (head_dim / 16 MMAs of 128 x 64 x 16), committed to
//            an mbarrier; each thread loads its S row from TMEM, masks it,
//            updates its running max m and sum l (base-2 domain), writes its
//            row of P (16-bit) to shared memory in the canonical layout and
//            rescales its O row in TMEM by 2^(m_old - m_new) (a warp whose
//            rows all kept their maximum skips it); then O += P V (64 / 16
//            MMAs of 128 x head_dim x 16), committed to a second mbarrier.
//   SM       112 KB of shared memory and 256 TMEM columns per CTA at
//            head_dim 128: two CTAs share an SM, so one's softmax overlaps
//            the other's tensor-core work.
//   output   O / l from TMEM, and the natural-log logsumexp per query.
//
// Every mbarrier wait is bounded; on a timeout the kernel records the error
// word, stops issuing, waits (bounded) for what it issued and frees TMEM.
#include "attention_pp.h"
#include "cluster_ring.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tensor_map.h"

#include <atomic>

namespace rwsm {

__device__ unsigned g_error_attention_tc = 0;

namespace {

constexpr int kTcBM = 128;          // queries per CTA (MMA M)
constexpr int kTcThreads = 128;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemO = 128;    // column of the O accumulator
constexpr float kLazyRescaleLog2 = 8.0f;    // p <= 2^8 between rescales

// ---- tcgen05 wrappers -----------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit operands, fp32 accumulators.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x 16) read from tensor memory, lane
// = row, each 32-bit column two consecutive 16-bit K elements (the lower
// index in the low half).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread has
// issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive TMEM columns of this thread's lane (warp w reads lanes
// 32w..32w+31; `taddr` carries the lane in bits 31..16, the column below).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),
          "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
          "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),
          "=f"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        :: "r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
           "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]),
           "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]),
           "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]),
           "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
           "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
           "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- operand layouts and descriptors ---------------------------------------
//
// Canonical layout without swizzle: the matrix is cut into 8 x 8 core
// matrices of 16-bit elements, each 128 contiguous bytes (8 rows of 16
// bytes).  For a K-major operand a core-matrix row holds 8 consecutive K
// elements of one M (or N) row; the core matrix of rows 8i.. and K elements
// 8j.. starts at i * SBO + j * LBO.  For an MN-major operand a core-matrix
// row holds 8 consecutive MN elements of one K row; the core matrix of MN
// elements 8i.. and K rows 8j.. starts at i * SBO + j * LBO.  Here LBO is
// always 128 bytes (core matrices adjacent along K) and SBO the size of one
// 8-row band.

// Byte offset of the 16-byte chunk holding elements [8c, 8c + 8) of row r of
// a K-major operand with `kdim` elements per row.
__device__ __forceinline__ uint32_t kmajor_off(int r, int c, int kdim)
{
    return static_cast<uint32_t>((r >> 3) * (kdim / 8) * 128 + c * 128 + (r & 7) * 16);
}

// Byte offset of the 16-byte chunk holding MN elements [8c, 8c + 8) of K row
// `kr` of an MN-major operand with `kdim` K rows.
__device__ __forceinline__ uint32_t mnmajor_off(int kr, int c, int kdim)
{
    return static_cast<uint32_t>(c * (kdim / 8) * 128 + (kr >> 3) * 128 + (kr & 7) * 16);
}

// Shared-memory matrix descriptor: start address, leading (K direction) and
// stride (8-row band) byte offsets, each in units of 16 bytes; descriptor
// version 1 at bits 46..47; no swizzle (layout type 0 at bits 61..63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
           (static_cast<uint64_t>(1) << 46);
}

// Same, for operands stored with the 128-byte swizzle (layout type 2 in
// bits 61..63): 8-row atoms of 128-byte rows whose 16-byte chunks are
// permuted by row % 8, atoms 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return smem_desc(addr, lbo, sbo) | (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4..5 = 1), A
// and B formats (bits 7..9, 10..12: 0 fp16, 1 bf16), B MN-major flag (bit 16),
// N / 8 (bits 17..22), M / 16 (bits 24..28); A is K-major.
__host__ __device__ constexpr uint32_t umma_idesc(int m, int n, bool bf16, bool b_mn_major)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// 16-byte global -> shared copy; src_bytes 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Wait until at most n (0, 1 or 2) of this thread's cp.async groups are
// still pending (the most recent ones).
__device__ __forceinline__ void cp_async_wait_pending(int n)
{
    if (n <= 0)
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    else if (n == 1)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
        asm volatile("cp.async.wait_group 2;" ::: "memory");
}

// Rows [row0, row0 + ROWS) of a [n][D] matrix into shared memory, K-major
// (MN_MAJOR = false: rows are M/N, elements along K) or as the MN-major B
// operand with the rows as K (MN_MAJOR = true).  Rows past n are zero.
template <int D, int ROWS, bool MN_MAJOR>
__device__ __forceinline__ void stage(uint32_t base, const unsigned short* g, int64_t row0,
                                      int64_t n, int tid)
{
    constexpr int CH = D / 8;
    for (int i = tid; i < ROWS * CH; i += kTcThreads) {
        const int r = i / CH, c = i % CH;
        const int64_t gr = row0 + r;
        const bool ok = gr < n;
        const uint32_t off = MN_MAJOR ? mnmajor_off(r, c, ROWS) : kmajor_off(r, c, D);
        cp16(base + off, g + (ok ? gr : 0) * D + c * 8, ok ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <typename T, int D, int BN, bool CAUSAL>
__global__ void __launch_bounds__(kTcThreads, BN == 64 ? 2 : 1)
attention_tc_kernel(const T* q, const T* k, const T* v, T* o, float* lse, int64_t bh,
                    int64_t n_q, int64_t n_k, float scale_log2, int64_t offset)
{
    constexpr bool kBF16 = sizeof(T) == 2 && Elem<T>::kNegInfBits == 0xff80u;
    constexpr uint32_t Q_BYTES = kTcBM * D * 2, KV_BYTES = BN * D * 2;
    constexpr uint32_t SBO_QK = (D / 8) * 128;              // 8-row band of Q, K
    constexpr uint32_t SBO_P = (BN / 8) * 128;              // 8-row band of P
    constexpr uint32_t SBO_V = (BN / 8) * 128;              // 8-column band of V
    constexpr uint32_t IDESC_S = umma_idesc(kTcBM, BN, kBF16, false);
    constexpr uint32_t IDESC_PV = umma_idesc(kTcBM, D, kBF16, true);
    constexpr int NCH = BN / 32;                             // 32-column S chunks
    extern __shared__ __align__(128) unsigned char tc_smem[];
    __shared__ __align__(8) unsigned long long bar_s, bar_o;
    __shared__ uint32_t tmem_slot;

    const uint32_t base = (smem_addr(tc_smem) + 127u) & ~127u;
    const uint32_t sQ = base, sK = sQ + Q_BYTES, sV = sK + 2 * KV_BYTES, sP = sV + 2 * KV_BYTES;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t n_qt = (n_q + kTcBM - 1) / kTcBM;
    const int64_t b = blockIdx.x / n_qt;
    int64_t qt = blockIdx.x % n_qt;
    if (CAUSAL)
        qt = n_qt - 1 - qt;
    const int64_t q0 = qt * kTcBM, qi = q0 + tid;            // this thread's query
    const unsigned short* gq = reinterpret_cast<const unsigned short*>(q) + b * n_q * D;
    const unsigned short* gk = reinterpret_cast<const unsigned short*>(k) + b * n_k * D;
    const unsigned short* gv = reinterpret_cast<const unsigned short*>(v) + b * n_k * D;
    int64_t n_kt = (n_k + BN - 1) / BN;
    if (CAUSAL) {
        const int64_t last = q0 + kTcBM - 1 + offset;
        const int64_t lim = last < 0 ? 0 : last / BN + 1;
        n_kt = lim < n_kt ? lim : n_kt;
    }

    if (warp == 0) {
        tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_addr(&bar_s), 1);
        mbar_init(smem_addr(&bar_o), 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(warp * 32) << 16);   // this warp's lanes

    pdl_launch_dependents();
    pdl_wait();
    stage<D, kTcBM, false>(sQ, gq, q0, n_q, tid);
    if (n_kt > 0) {
        stage<D, BN, false>(sK, gk, 0, n_k, tid);
        stage<D, BN, true>(sV, gv, 0, n_k, tid);
    }

    float m = kNegInf, l = 0.0f;
    bool failed = false;
    uint32_t issued_s = 0, issued_o = 0;                      // commits to bar_s, bar_o
    // One tensor-core wait per tile: P V(t - 1) is issued at the end of tile
    // t - 1 and S(t) right after it, so S(t) completing (bar_s) also means
    // P V(t - 1) has completed (a commit covers every earlier tcgen05 op of
    // the issuing thread).  K(t + 1) is prefetched as soon as S(t) is issued
    // (its buffer held K(t - 1)), V(t + 1) once S(t) has completed (its
    // buffer held V(t - 1)).
    for (int64_t t = 0; t < n_kt; ++t) {
        // (a) K(t) has landed; V(t), issued after it, may still be in flight
        cp_async_wait_pending(t == 0 ? 0 : 1);
        fence_proxy_async_smem();                            // copies -> tensor cores
        __syncthreads();
        const uint32_t cK = sK + static_cast<uint32_t>(t & 1) * KV_BYTES;
        const uint32_t cV = sV + static_cast<uint32_t>(t & 1) * KV_BYTES;

        // (b) S = Q K^T into TMEM columns [0, BN), queued behind P V(t - 1)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_f16(tmem, smem_desc(sQ + ks * 256, 128, SBO_QK),
                         smem_desc(cK + ks * 256, 128, SBO_QK), IDESC_S, ks > 0 ? 1u : 0u);
            umma_commit(smem_addr(&bar_s));
        }
        ++issued_s;
        // (c) K(t + 1) into the buffer S(t - 1) finished with
        if (t + 1 < n_kt)
            stage<D, BN, false>(sK + static_cast<uint32_t>((t + 1) & 1) * KV_BYTES, gk,
                                (t + 1) * BN, n_k, tid);
        // (d) S(t), and with it P V(t - 1), has completed
        const bool ok_s = mbar_wait_bounded(smem_addr(&bar_s), static_cast<uint32_t>(t & 1));
        failed = __syncthreads_or(!ok_s) != 0;
        if (failed)
            break;
        tc_fence_after();
        // (e) V(t + 1) into the buffer P V(t - 1) finished with
        if (t + 1 < n_kt)
            stage<D, BN, true>(sV + static_cast<uint32_t>((t + 1) & 1) * KV_BYTES, gv,
                               (t + 1) * BN, n_k, tid);

        // (f) this thread's S row: mask, running max, p, P row to shared memory.
        // The max is taken on the raw scores (the scale is positive) and the
        // scale folds into p = 2^(S * scale * log2 e - m).  Only a tile that
        // reaches past the last key or (causal) past the diagonal of the
        // CTA's first query is masked, with one integer compare per score.
        const int64_t k0 = t * BN;
        float mx = kNegInf;
        float sv[NCH][32];
#pragma unroll
        for (int c = 0; c < NCH; ++c)
            tmem_ld32(t_row + c * 32, sv[c]);
        tmem_wait_ld();
        const bool edge = k0 + BN > n_k || (CAUSAL && k0 + BN - 1 > q0 + offset);
        if (edge) {
            int64_t lim = n_k - k0;                          // keys of the tile kept
            if (CAUSAL && qi + offset + 1 - k0 < lim)
                lim = qi + offset + 1 - k0;
            const int keep = static_cast<int>(lim < 0 ? 0 : (lim > BN ? BN : lim));
#pragma unroll
            for (int c = 0; c < NCH; ++c)
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c * 32 + j >= keep)
                        sv[c][j] = kNegInf;
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int j = 0; j < 32; j += 2)
                mx = max3(mx, sv[c][j], sv[c][j + 1]);
        // Lazy rescaling: the reference m (base 2) moves only when the tile's
        // max exceeds it by more than 2^8, so p stays below 2^8 and most
        // tiles leave O alone; O / l and the logsumexp only need m and l to
        // agree.
        const float mx_s = mx * scale_log2;
        float alpha = 1.0f;
        if (mx_s > m + kLazyRescaleLog2) {
            alpha = ex2_ftz(m - mx_s);                      // 0 while m is -inf
            m = mx_s;
        }
        const float ref = m == kNegInf ? 0.0f : m;
        float sum = 0.0f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {                    // 8 keys per 16-byte chunk
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    p[e] = ex2_ftz(fmaf(sv[c][g * 8 + e], scale_log2, -ref));
                    sum += p[e];
                }
                const uint32_t w0 = Elem<T>::pack2(p[0], p[1]), w1 = Elem<T>::pack2(p[2], p[3]);
                const uint32_t w2 = Elem<T>::pack2(p[4], p[5]), w3 = Elem<T>::pack2(p[6], p[7]);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                             :: "r"(sP + kmajor_off(tid, c * 4 + g, BN)), "r"(w0), "r"(w1),
                                "r"(w2), "r"(w3) : "memory");
            }
        }
        l = l * alpha + sum;
        // rescale this thread's O row; skipped by a warp whose rows all kept
        // their maximum (alpha = 1)
        if (t > 0 && !__all_sync(0xffffffffu, alpha == 1.0f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float ov[32];
                tmem_ld32(t_row + kTmemO + c * 32, ov);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    ov[j] *= alpha;
                tmem_st32(t_row + kTmemO + c * 32, ov);
            }
            tmem_wait_st();
        }
        // (g) V(t) has landed: only the two copies of this tile may be pending
        cp_async_wait_pending(t + 1 < n_kt ? 2 : 0);
        fence_proxy_async_smem();                            // P, V -> tensor cores
        tc_fence_before();
        __syncthreads();

        // (h) O += P V(t) into TMEM columns [128, 128 + D); waited for through
        // the next S (or after the loop)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
                umma_f16(tmem + kTmemO, smem_desc(sP + ks * 256, 128, SBO_P),
                         smem_desc(cV + ks * 256, 128, SBO_V), IDESC_PV,
                         (t > 0 || ks > 0) ? 1u : 0u);
            umma_commit(smem_addr(&bar_o));
        }
        ++issued_o;
    }
    if (!failed && n_kt > 0) {
        const bool ok_o = mbar_wait_bounded(smem_addr(&bar_o),
                                            static_cast<uint32_t>((n_kt - 1) & 1));
        failed = __syncthreads_or(!ok_o) != 0;
        tc_fence_after();
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    if (!failed) {
        // ---- O / l to global (this thread's row), logsumexp
        const float inv = 1.0f / l;
        unsigned short* go = reinterpret_cast<unsigned short*>(o) + b * n_q * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tmem_ld32(t_row + kTmemO + c * 32, ov);
            tmem_wait_ld();
            if (qi < n_q) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint4 w;
                    w.x = Elem<T>::pack2(ov[g * 8 + 0] * inv, ov[g * 8 + 1] * inv);
                    w.y = Elem<T>::pack2(ov[g * 8 + 2] * inv, ov[g * 8 + 3] * inv);
                    w.z = Elem<T>::pack2(ov[g * 8 + 4] * inv, ov[g * 8 + 5] * inv);
                    w.w = Elem<T>::pack2(ov[g * 8 + 6] * inv, ov[g * 8 + 7] * inv);
                    *reinterpret_cast<uint4*>(go + qi * D + c * 32 + g * 8) = w;
                }
            }
        }
        if (n_kt == 0 && qi < n_q) {                         // no key at all: NaN rows
            const float nan = __int_as_float(0x7fc00000);
            for (int d0 = 0; d0 < D; d0 += 2)
                *reinterpret_cast<uint32_t*>(go + qi * D + d0) = Elem<T>::pack2(nan, nan);
        }
        if (lse && qi < n_q)
            lse[b * n_q + qi] = l > 0.0f ? (m + __log2f(l)) * 0.69314718055994531f : kNegInf;
    } else {
        if (tid == 0) {
            atomicOr(&g_error_attention_tc, kErrMbarrierTimeout);
            // Wait (bounded) for what was issued before freeing TMEM.
            if (issued_s)
                mbar_wait_bounded(smem_addr(&bar_s), (issued_s - 1) & 1u);
            if (issued_o)
                mbar_wait_bounded(smem_addr(&bar_o), (issued_o - 1) & 1u);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, kTmemCols);
}

// ---- two query tiles per CTA in ping-pong ---------------------------------
//
//   CTA      256 queries of one (batch, head): tile A (queries 0..127) and
//            tile B (128..255).  Warps 0-3 run tile A's softmax, warps 4-7
//            tile B's (thread t of a warpgroup owns query row t = TMEM lane
//            t); lane 0 of warp 8 issues every tcgen05.mma, lane 0 of warp 9
//            every tensor-map copy.
//   operands Q, K and V land by cp.async.bulk.tensor (3-D maps: element,
//            row, head; rows past a head's end read as zero) in boxes of 64
//            elements with the 128-byte swizzle, read by the tensor cores
//            through swizzled descriptors.  Key tiles hold BN keys (128 at
//            d = 128, 64 at d = 64).
//   TMEM     S_A at column 0, S_B at BN, O_A at 2 BN, O_B at 2 BN + D (512
//            columns at d = 128, 256 at d = 64).  A softmax thread reads its S row twice (the max,
//            then the exponentials) and writes its P row, rounded to the
//            operand type, over the first BN / 2 columns of S: P V takes its
//            A operand from tensor memory, so P never passes through shared
//            memory.
//   order    per key tile t the MMA lane waits for P_A(t) (bar_p[A]),
//            issues O_A += P_A V(t) and S_A(t+1) = Q_A K(t+1)^T, commits
//            (bar_s[A]); then the same for B.  So the tensor cores compute
//            one tile's products while the other tile's warpgroup runs its
//            softmax, and every K/V tile copied serves 256 queries.  A
//            warpgroup's wait on S_X(t+1) also covers O_X += P_X V(t) (one
//            commit covers every earlier operation of the issuing thread), so
//            O_X is free for it when S_X(t+1) has landed; S_X(t+1) overwrites
//            P_X(t) only after P_X V(t) has read it (the tensor cores perform
//            one thread's products in the order issued).
//   ring     K and V in KVS slots (tile t in slot t % KVS): the copy lane
//            refills K(t)'s slot with K(t+KVS) once a commit issued right
//            after S_B(t) has arrived (k_free), V(t)'s with V(t+KVS) once one
//            issued after P_B V(t) has (v_free).  Its waits never hold up the
//            MMA lane, which only waits for operands and for P: with one lane
//            doing both, a time-stamped build showed it reacting to a written
//            P about 1700 cycles late (blocked on the P V wait and the
//            copies), in a 3600-cycle period per key tile.
//
// Every wait is bounded; a timed-out wait records the error word and the
// kernel stops issuing, waits (bounded) for what it issued and frees TMEM.
constexpr int kPpWarpgroups = 2;                          // query tiles per CTA

// Warps that share a row of S (each takes BN / split of its keys): two at
// d = 128, so a query tile's softmax runs on eight warps; one at d = 64
// (two CTAs share an SM there and their registers would not fit twice).
template <int D>
__host__ __device__ constexpr int pp_split()
{
    return D == 128 ? 2 : 1;
}

// Softmax warps, plus the MMA warp and the copy warp.
template <int D>
__host__ __device__ constexpr int pp_threads()
{
    return kPpWarpgroups * 4 * pp_split<D>() * 32 + 64;
}

// Keys per tile of the ping-pong kernel.  d = 128: 128, so that S = Q K^T
// is a 128 x 128 product (a 128 x 64 x 16 product reads 6 KB of operands
// from shared memory for 32 cycles of arithmetic; a time-stamped build saw
// about 90 cycles per such product issued), one CTA per SM (S_A, S_B, O_A,
// O_B fill the 512 TMEM columns).  d = 64: 64 keys and two CTAs per SM (256
// columns each): the exponentials, not the products, bound it there (one
// exponential per 2 x 64 multiply-adds), and two CTAs keep four softmax
// warpgroups on each SM.
template <int D>
__host__ __device__ constexpr int pp_bn()
{
    return D == 128 ? 128 : 64;
}

// Key/value ring depth: two slots at d = 128 (Q, K and V fill 192 KB), four
// at d = 64 (96 KB a CTA).
template <int D>
__host__ __device__ constexpr int pp_kv_stages()
{
    return D == 128 ? 2 : 4;
}

template <typename T, int D, int BN, bool CAUSAL>
__global__ void __launch_bounds__(pp_threads<D>(), D == 64 ? 2 : 1)
attention_pp_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, T* o, float* lse, int64_t bh,
                    int64_t n_q, int64_t n_k, float scale_log2, int64_t offset)
{
    constexpr bool kBF16 = sizeof(T) == 2 && Elem<T>::kNegInfBits == 0xff80u;
    constexpr uint32_t QT_BYTES = kTcBM * D * 2, KV_BYTES = BN * D * 2;
    constexpr int KVS = pp_kv_stages<D>();
    constexpr uint32_t IDESC_S = umma_idesc(kTcBM, BN, kBF16, false);
    constexpr uint32_t IDESC_PV = umma_idesc(kTcBM, D, kBF16, true);
    constexpr uint32_t TMEM_COLS = 2 * BN + 2 * D <= 256 ? 256u : 512u;
    static_assert(2 * BN + 2 * D <= 512, "S_A, S_B, O_A and O_B fill at most 512 columns");
    constexpr int NCH = BN / 32;
    constexpr int HS = pp_split<D>();                        // warps per row group
    constexpr int CW = BN / HS;                              // keys of S per softmax warp
    constexpr int CTRL = kPpWarpgroups * 4 * HS;             // the MMA warp
    constexpr int LOADW = CTRL + 1;                          // the copy warp
    extern __shared__ __align__(128) unsigned char tc_smem[];
    __shared__ __align__(8) unsigned long long bar_s[2], bar_p[2], bar_fin[2], bar_drain;
    __shared__ __align__(8) unsigned long long q_full, k_full[KVS], v_full[KVS];
    __shared__ __align__(8) unsigned long long k_free[KVS], v_free[KVS];
    __shared__ uint32_t tmem_slot;
    __shared__ int s_failed;
    // Row maxima (by tile parity) and final sums of the warps sharing a row.
    __shared__ float xmax[HS > 1 ? 2 : 1][kPpWarpgroups][HS][kTcBM];
    __shared__ float xsum[kPpWarpgroups][HS][kTcBM];

    const uint32_t base = (smem_addr(tc_smem) + 1023u) & ~1023u;   // swizzle atoms
    const uint32_t sQ = base, sK = sQ + 2 * QT_BYTES, sV = sK + KVS * KV_BYTES;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n_qt = (n_q + 2 * kTcBM - 1) / (2 * kTcBM);
    // Causal: query tiles of every head, longest (last) first, so that the
    // CTAs dispatched last are the short ones and the tail is short.
    const int64_t b = CAUSAL ? static_cast<int64_t>(blockIdx.x) % bh : blockIdx.x / n_qt;
    const int64_t qt = CAUSAL ? n_qt - 1 - static_cast<int64_t>(blockIdx.x) / bh
                              : static_cast<int64_t>(blockIdx.x) % n_qt;
    const int64_t q0 = qt * 2 * kTcBM;
    // Key tiles the CTA visits (n_kt, all of them for tile B) and tile A's
    // share: under the causal mask tile A stops where its own last query
    // does (at 128-key tiles one tile before B when the mask is the pages').
    int64_t n_kt = (n_k + BN - 1) / BN, n_kt_a = n_kt;
    if (CAUSAL) {
        auto tiles_to = [&](int64_t last) {                  // through query `last`
            const int64_t lim = last < 0 ? 0 : last / BN + 1;
            return lim < n_kt ? lim : n_kt;
        };
        n_kt_a = tiles_to(q0 + kTcBM - 1 + offset);
        n_kt = tiles_to(q0 + 2 * kTcBM - 1 + offset);
    }

    if (warp == 0) {
        tmem_alloc(smem_addr(&tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_addr(&bar_s[x]), 1);
            mbar_init(smem_addr(&bar_p[x]), 128 * HS);
            mbar_init(smem_addr(&bar_fin[x]), 1);
        }
        mbar_init(smem_addr(&bar_drain), 1);
        mbar_init(smem_addr(&q_full), 1);
        for (int x = 0; x < KVS; ++x) {
            mbar_init(smem_addr(&k_full[x]), 1);
            mbar_init(smem_addr(&v_full[x]), 1);
            mbar_init(smem_addr(&k_free[x]), 1);
            mbar_init(smem_addr(&v_free[x]), 1);
        }
        s_failed = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    pdl_launch_dependents();
    pdl_wait();

    // Key tile t lives in ring slot t % KVS; its barriers' phase is t / KVS.
    auto slot = [](int64_t t) { return static_cast<uint32_t>(t) % KVS; };
    auto phase = [](int64_t t) { return (static_cast<uint32_t>(t) / KVS) & 1u; };
    if (warp == LOADW) {
        // --------------------------------------------------------- copy warp
        // Lane 0 issues every copy (the tensor memory accelerator).  An
        // operand tile lands as D/64 boxes of 64 elements x ROWS rows, each
        // row 128 bytes with the copy engine's 128-byte swizzle, so box c is
        // ROWS/8 swizzle atoms of 1024 bytes.  Rows past a head's end are
        // zero-filled by the copy engine (the tensor maps are 3-D: element,
        // row, head).  K(t + KVS) goes into K(t)'s slot once both S(t) have
        // completed (k_free), V(t + KVS) into V(t)'s once both P V(t) have
        // (v_free): the MMA warp commits those barriers, so neither of its
        // waits holds up the products.
        if (lane == 0) {
            bool failed = false;
            auto wait1 = [&](uint32_t bar, uint32_t parity) {
                if (!failed && !mbar_wait_bounded(bar, parity)) {
                    failed = true;
                    *reinterpret_cast<volatile int*>(&s_failed) = 1;
                }
            };
            auto tma3 = [&](uint32_t dst, const CUtensorMap* map, int xe, int64_t row, uint32_t bar) {
                asm volatile(
                    "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%2, %3, %4}], [%5];"
                    :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(xe),
                       "r"(static_cast<int>(row)), "r"(static_cast<int>(b)), "r"(bar)
                    : "memory");
            };
            auto load_rows = [&](uint32_t dst, const CUtensorMap* map, int rows, int64_t row0,
                                 uint32_t bar, uint32_t bytes) {
                mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma3(dst + static_cast<uint32_t>(c * rows * 128), map, c * 64, row0, bar);
            };
            int64_t k_issued = 0, v_issued = 0;
            auto load_k = [&](int64_t t) {
                load_rows(sK + slot(t) * KV_BYTES, &map_k, BN, t * BN, smem_addr(&k_full[slot(t)]),
                          KV_BYTES);
                k_issued = t + 1;
            };
            auto load_v = [&](int64_t t) {
                load_rows(sV + slot(t) * KV_BYTES, &map_v, BN, t * BN, smem_addr(&v_full[slot(t)]),
                          KV_BYTES);
                v_issued = t + 1;
            };
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&map_q)) : "memory");
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&map_k)) : "memory");
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&map_v)) : "memory");
            if (n_kt > 0) {
                load_rows(sQ, &map_q, kTcBM, q0, smem_addr(&q_full), 2 * QT_BYTES);
                // (the second Q tile completes on the same barrier)
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma3(sQ + QT_BYTES + static_cast<uint32_t>(c * kTcBM * 128), &map_q, c * 64,
                         q0 + kTcBM, smem_addr(&q_full));
                for (int64_t t = 0; t < KVS && t < n_kt; ++t) {
                    load_k(t);
                    load_v(t);
                }
                for (int64_t t = 0; t + KVS < n_kt && !failed; ++t) {
                    wait1(smem_addr(&k_free[slot(t)]), phase(t));      // both S(t) done
                    if (failed || *reinterpret_cast<volatile int*>(&s_failed))
                        break;
                    load_k(t + KVS);
                    wait1(smem_addr(&v_free[slot(t)]), phase(t));      // both P V(t) done
                    if (failed || *reinterpret_cast<volatile int*>(&s_failed))
                        break;
                    load_v(t + KVS);
                }
                if (failed || *reinterpret_cast<volatile int*>(&s_failed)) {
                    // Let the copies still in flight land (each wait bounded):
                    // Q, and the last KVS tiles issued into each ring (an
                    // earlier tile of a slot was consumed before its slot
                    // was refilled).
                    mbar_wait_bounded(smem_addr(&q_full), 0u);
                    for (int64_t t = k_issued > KVS ? k_issued - KVS : 0; t < k_issued; ++t)
                        mbar_wait_bounded(smem_addr(&k_full[slot(t)]), phase(t));
                    for (int64_t t = v_issued > KVS ? v_issued - KVS : 0; t < v_issued; ++t)
                        mbar_wait_bounded(smem_addr(&v_full[slot(t)]), phase(t));
                }
            }
        }
        __syncwarp();
    } else if (warp == CTRL) {
        // ---------------------------------------------------------- MMA warp
        // Lane 0 issues every product.  Q and K are K-major: a 16-element
        // step of the contraction is 32 bytes into the swizzle atom row (the
        // tensor cores apply the same swizzle to the address), SBO = 1024
        // between 8-row bands.  V is MN-major (rows = keys, the output
        // dimension contiguous): SBO = 1024 between 8-key bands, LBO = one
        // box between the 64-element halves of D.
        if (lane == 0) {
            bool failed = false;
            auto wait1 = [&](uint32_t bar, uint32_t parity) {
                if (!failed && !mbar_wait_bounded(bar, parity)) {
                    failed = true;
                    *reinterpret_cast<volatile int*>(&s_failed) = 1;
                }
            };
            auto issue_s = [&](int x, int64_t t) {
                const uint32_t cK = sK + slot(t) * KV_BYTES;
                const uint32_t qx = sQ + static_cast<uint32_t>(x) * QT_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma_f16(tmem + static_cast<uint32_t>(x * BN),
                             smem_desc_sw128(qx + (ks >> 2) * (kTcBM * 128) + (ks & 3) * 32, 16, 1024),
                             smem_desc_sw128(cK + (ks >> 2) * (BN * 128) + (ks & 3) * 32, 16, 1024),
                             IDESC_S,
                             ks > 0 ? 1u : 0u);
            };
            // P_X (16-bit) sits over S_X: each softmax warp's CW keys in the
            // first CW / 2 columns of its own CW-column part of S_X, so a
            // 16-key step of the product reads 8 columns, CW / 2 further on
            // in the second part.
            auto issue_pv = [&](int x, int64_t t) {
                const uint32_t cV = sV + slot(t) * KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks)
                    umma_f16_ta(tmem + static_cast<uint32_t>(2 * BN + x * D),
                                tmem + static_cast<uint32_t>(x * BN + ks * 8 +
                                                             (ks * 16 / CW) * (CW / 2)),
                                smem_desc_sw128(cV + ks * 2048, BN * 128, 1024), IDESC_PV,
                                (t > 0 || ks > 0) ? 1u : 0u);
            };
            if (n_kt > 0) {
                wait1(smem_addr(&q_full), 0u);
                wait1(smem_addr(&k_full[0]), 0u);
                if (!failed) {
                    tc_fence_after();
                    if (n_kt_a > 0) {
                        issue_s(0, 0);
                        umma_commit(smem_addr(&bar_s[0]));
                    }
                    issue_s(1, 0);
                    umma_commit(smem_addr(&bar_s[1]));
                    umma_commit(smem_addr(&k_free[0]));           // S(0) done
                }
            }
            // Per key tile t: P_A V(t) and S_A(t+1) once the softmax of A
            // has written P_A(t) (while A has tiles left), then the same for
            // B.  After P_B V(t) a commit frees V(t)'s slot, after S_B(t+1)
            // one frees K(t+1)'s (B visits every tile the CTA loads).
            for (int64_t t = 0; t < n_kt && !failed; ++t) {
                wait1(smem_addr(&v_full[slot(t)]), phase(t));
                for (int x = 0; x < 2 && !failed; ++x) {
                    const int64_t tiles = x == 0 ? n_kt_a : n_kt;
                    if (t >= tiles)
                        continue;
                    const bool more = t + 1 < tiles;
                    wait1(smem_addr(&bar_p[x]), static_cast<uint32_t>(t & 1));   // P_X(t) written
                    if (failed)
                        break;
                    tc_fence_after();
                    issue_pv(x, t);
                    if (x == 1)
                        umma_commit(smem_addr(&v_free[slot(t)]));   // P V(t) done
                    if (more) {
                        wait1(smem_addr(&k_full[slot(t + 1)]), phase(t + 1));
                        if (failed)
                            break;
                        issue_s(x, t + 1);
                        if (x == 1)
                            umma_commit(smem_addr(&k_free[slot(t + 1)]));   // S(t+1) done
                    }
                    umma_commit(smem_addr(more ? &bar_s[x] : &bar_fin[x]));
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax warps
        // Warp w: query tile x, TMEM lane group w % 4 (rows 32 (w % 4) ..),
        // and part h of the tile's keys and of O's columns when HS warps
        // share a row (h = 0 at d = 64).
        const int x = warp / (4 * HS);                       // 0: tile A, 1: tile B
        const int h = (warp / 4) % HS;
        const int r = (warp & 3) * 32 + lane;                // row of the tile = TMEM lane
        const int64_t qx0 = q0 + static_cast<int64_t>(x) * kTcBM;
        const int64_t qi = qx0 + r;                          // this thread's query
        const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = static_cast<uint32_t>(x * BN + h * CW);   // this warp's keys
        constexpr int OW = D / HS;                           // O columns per warp
        const uint32_t o_col = static_cast<uint32_t>(2 * BN + x * D + h * OW);
        const int64_t my_kt = x == 0 ? n_kt_a : n_kt;         // key tiles of this query tile
        constexpr int NCH = CW / 32;                         // 32-column chunks per warp
        float m = kNegInf, l = 0.0f;                         // l: this warp's part of the sum
        bool failed = false;                                 // warp-uniform
        for (int64_t t = 0; t < my_kt; ++t) {
            const bool ok = failed || mbar_wait_bounded(smem_addr(&bar_s[x]), static_cast<uint32_t>(t & 1));
            if (__any_sync(0xffffffffu, !ok) && !failed) {
                failed = true;
                *reinterpret_cast<volatile int*>(&s_failed) = 1;
            }
            tc_fence_after();
            const int64_t k0 = t * BN;
            const bool edge = k0 + BN > n_k || (CAUSAL && k0 + BN - 1 > qx0 + offset);
            int keep = CW;                                   // this warp's keys kept
            if (edge) {
                int64_t lim = n_k - k0;
                if (CAUSAL && qi + offset + 1 - k0 < lim)
                    lim = qi + offset + 1 - k0;
                lim -= h * CW;
                keep = static_cast<int>(lim < 0 ? 0 : (lim > CW ? CW : lim));
            }
            // This warp's CW scores stay in registers: loaded together,
            // waited for once.
            float sv[NCH][32];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                tmem_ld32(t_row + s_col + c * 32, sv[c]);
            tmem_wait_ld();
            if (edge) {
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c * 32 + j >= keep)
                            sv[c][j] = kNegInf;
            }
            float mx = kNegInf;
#pragma unroll
            for (int c = 0; c < NCH; ++c)
#pragma unroll
                for (int j = 0; j < 32; j += 2)
                    mx = max3(mx, sv[c][j], sv[c][j + 1]);
            if constexpr (HS > 1) {
                // The row's maximum over the warps that share it (named
                // barrier of the tile's warps; slots by tile parity, so a
                // slot is rewritten only after the next barrier).
                const int par = static_cast<int>(t & 1);
                xmax[par][x][h][r] = mx;
                named_barrier(1 + x, 128 * HS);
#pragma unroll
                for (int o = 0; o < HS; ++o)
                    mx = fmaxf(mx, xmax[par][x][o][r]);
            }
            // Lazy rescaling as in attention_tc_kernel: the reference m moves
            // only when a tile's max exceeds it by more than 2^8.
            const float mx_s = mx * scale_log2;
            float alpha = 1.0f;
            if (mx_s > m + kLazyRescaleLog2) {
                alpha = ex2_ftz(m - mx_s);
                m = mx_s;
            }
            const float ref = m == kNegInf ? 0.0f : m;
            // p = 2^(S scale log2 e - m), summed, rounded to the operand type
            // in pairs and stored over the first CW / 2 columns of this
            // warp's part of S (its own scores, already in registers).  The
            // loop is written out twice, for tiles with and without masked
            // keys: the same arithmetic, but compiled apart it keeps fewer
            // registers live and measured faster.
            float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const float (&v)[32] = sv[c];
                uint32_t w[16];
                if (edge) {                                  // masked scores are -inf: p = 0
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float p0 = ex2_ftz(fmaf(v[2 * j], scale_log2, -ref));
                        const float p1 = ex2_ftz(fmaf(v[2 * j + 1], scale_log2, -ref));
                        sum0 += p0;
                        sum1 += p1;
                        w[j] = Elem<T>::pack2(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float p0 = ex2_ftz(fmaf(v[2 * j], scale_log2, -ref));
                        const float p1 = ex2_ftz(fmaf(v[2 * j + 1], scale_log2, -ref));
                        sum0 += p0;
                        sum1 += p1;
                        w[j] = Elem<T>::pack2(p0, p1);
                    }
                }
                tmem_st16(t_row + s_col + c * 16, w);
            }
            tmem_wait_st();
            l = l * alpha + (sum0 + sum1);
            if (t > 0 && !__all_sync(0xffffffffu, alpha == 1.0f)) {
#pragma unroll
                for (int c = 0; c < OW / 32; ++c) {
                    float ov[32];
                    tmem_ld32(t_row + o_col + c * 32, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        ov[j] *= alpha;
                    tmem_st32(t_row + o_col + c * 32, ov);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&bar_p[x]));               // release: P_X(t), O_X rescaled
        }
        if (my_kt > 0) {
            const bool ok = failed || mbar_wait_bounded(smem_addr(&bar_fin[x]), 0u);
            if (__any_sync(0xffffffffu, !ok) && !failed) {
                failed = true;
                *reinterpret_cast<volatile int*>(&s_failed) = 1;
            }
            tc_fence_after();
        }
        if constexpr (HS > 1) {
            // The row's sum over the warps that share it.
            xsum[x][h][r] = l;
            named_barrier(1 + x, 128 * HS);
            l = 0.0f;
#pragma unroll
            for (int o = 0; o < HS; ++o)
                l += xsum[x][o][r];
        }
        if (!failed) {
            const float inv = 1.0f / l;
            unsigned short* go = reinterpret_cast<unsigned short*>(o) + b * n_q * D + h * OW;
#pragma unroll
            for (int c = 0; c < OW / 32; ++c) {
                float ov[32];
                tmem_ld32(t_row + o_col + c * 32, ov);
                tmem_wait_ld();
                if (qi < n_q && my_kt > 0) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint4 w;
                        w.x = Elem<T>::pack2(ov[g * 8 + 0] * inv, ov[g * 8 + 1] * inv);
                        w.y = Elem<T>::pack2(ov[g * 8 + 2] * inv, ov[g * 8 + 3] * inv);
                        w.z = Elem<T>::pack2(ov[g * 8 + 4] * inv, ov[g * 8 + 5] * inv);
                        w.w = Elem<T>::pack2(ov[g * 8 + 6] * inv, ov[g * 8 + 7] * inv);
                        *reinterpret_cast<uint4*>(go + qi * D + c * 32 + g * 8) = w;
                    }
                }
            }
            if (my_kt == 0 && qi < n_q) {                    // no key at all: NaN rows
                const float nan = __int_as_float(0x7fc00000);
                for (int d0 = 0; d0 < OW; d0 += 2)
                    *reinterpret_cast<uint32_t*>(go + qi * D + d0) = Elem<T>::pack2(nan, nan);
            }
            if (lse && qi < n_q && h == 0)
                lse[b * n_q + qi] = l > 0.0f ? (m + __log2f(l)) * 0.69314718055994531f : kNegInf;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == CTRL * 32 && *reinterpret_cast<volatile int*>(&s_failed)) {
        // One more commit: it arrives once every tensor-core operation this
        // thread issued has completed; wait for it (bounded) before TMEM is
        // freed.
        atomicOr(&g_error_attention_tc, kErrMbarrierTimeout);
        tc_fence_after();
        umma_commit(smem_addr(&bar_drain));
        mbar_wait_bounded(smem_addr(&bar_drain), 0u);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// 3-D tensor map of a [bh][n][D] operand (element, row, head) with boxes of
// 64 elements (128 bytes, 128-byte swizzle) x `rows` rows of one head: rows
// past a head's end read as zero.
inline bool pp_tensor_map(CUtensorMap* map, const void* ptr, int64_t bh, int64_t n, int d,
                          int rows, int dtype)
{
    auto encode = tensor_map_encoder();
    if (!encode || bh >= (int64_t{1} << 31) || n >= (int64_t{1} << 31))
        return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n),
                                static_cast<cuuint64_t>(bh)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(n) * d * 2};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(rows), 1u};
    const cuuint32_t estride[3] = {1u, 1u, 1u};
    return encode(map, dtype == SOFTMAX_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(ptr), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <typename T, int D, bool CAUSAL>
cudaError_t launch_pp(const AttentionProblem& p, cudaStream_t s)
{
    constexpr int BN = pp_bn<D>();
    auto* kern = attention_pp_kernel<T, D, BN, CAUSAL>;
    const int smem = (2 * kTcBM * D + 2 * pp_kv_stages<D>() * BN * D) * 2 + 1024;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_set[dev].store(true);
    }
    CUtensorMap mq, mk, mv;
    if (!pp_tensor_map(&mq, p.q, p.bh, p.n_q, D, kTcBM, p.dtype) ||
        !pp_tensor_map(&mk, p.k, p.bh, p.n_k, D, BN, p.dtype) ||
        !pp_tensor_map(&mv, p.v, p.bh, p.n_k, D, BN, p.dtype))
        return cudaErrorNotSupported;                    // nothing launched
    const int64_t n_qt = (p.n_q + 2 * kTcBM - 1) / (2 * kTcBM);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_qt * p.bh), 1, 1);
    cfg.blockDim = dim3(pp_threads<D>(), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, 1));
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, static_cast<T*>(p.o),
                                               p.lse, p.bh, p.n_q, p.n_k, scale_log2, p.offset);
    note_launch();
    return err;
}

template <typename T>
cudaError_t launch_pp_t(const AttentionProblem& p, cudaStream_t s)
{
    if (p.head_dim == 64)
        return p.causal ? launch_pp<T, 64, true>(p, s) : launch_pp<T, 64, false>(p, s);
    if (p.head_dim == 128)
        return p.causal ? launch_pp<T, 128, true>(p, s) : launch_pp<T, 128, false>(p, s);
    return cudaErrorInvalidValue;
}

template <typename T, int D, int BN, bool CAUSAL>
cudaError_t launch_tc(const AttentionProblem& p, cudaStream_t s)
{
    auto* kern = attention_tc_kernel<T, D, BN, CAUSAL>;
    // At most two CTAs per SM (each holds 256 TMEM columns of 512): the
    // request is at least a third of an SM's shared memory.
    int smem = (kTcBM * D + 4 * BN * D + kTcBM * BN) * 2 + 128;
    smem = smem < 80 * 1024 ? 80 * 1024 : smem;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (!attr_set[dev].load()) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_set[dev].store(true);
    }
    const int64_t n_qt = (p.n_q + kTcBM - 1) / kTcBM;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_qt * p.bh), 1, 1);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, 1));
    const float scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(p.q),
                                               static_cast<const T*>(p.k),
                                               static_cast<const T*>(p.v), static_cast<T*>(p.o),
                                               p.lse, p.bh, p.n_q, p.n_k, scale_log2, p.offset);
    note_launch();
    return err;
}

template <typename T, int D>
cudaError_t launch_tc_d(const AttentionProblem& p, cudaStream_t s)
{
    // 64-key tiles: 112 KB of shared memory at d = 128, so two CTAs share an
    // SM and one's softmax overlaps the other's tensor-core work.
    return p.causal ? launch_tc<T, D, 64, true>(p, s) : launch_tc<T, D, 64, false>(p, s);
}

template <typename T>
cudaError_t launch_tc_t(const AttentionProblem& p, cudaStream_t s)
{
    if (p.head_dim == 64) return launch_tc_d<T, 64>(p, s);
    if (p.head_dim == 128) return launch_tc_d<T, 128>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attention_tc(const AttentionProblem& p, cudaStream_t s)
{
    if (p.bh * ((p.n_q + kTcBM - 1) / kTcBM) > 0x7fffffff)
        return cudaErrorInvalidValue;
    return p.dtype == SOFTMAX_BF16 ? launch_tc_t<BF16Bits>(p, s) : launch_tc_t<F16Bits>(p, s);
}

cudaError_t launch_attention_pp(const AttentionProblem& p, cudaStream_t s)
{
    if (p.bh * ((p.n_q + 2 * kTcBM - 1) / (2 * kTcBM)) > 0x7fffffff)
        return cudaErrorInvalidValue;                    // grid too large: nothing launched
    return p.dtype == SOFTMAX_BF16 ? launch_pp_t<BF16Bits>(p, s) : launch_pp_t<F16Bits>(p, s);
}

unsigned read_error_attention_tc(bool clear)
{
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_attention_tc, sizeof v) != cudaSuccess)
        return 0;
    if (clear && v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_error_attention_tc, &zero, sizeof zero);
    }
    return v;
}

}  // namespace rwsm
