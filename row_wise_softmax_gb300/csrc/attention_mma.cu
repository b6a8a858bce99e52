// Attention forward with the online softmax inside it, on the warp-level
// tensor-core path (mma.sync m16n8k16, 16-bit operands, fp32 accumulators).
//
// "Triton GPU programming deep dive", section 3.3: for a tile of queries,
// walk the keys a tile at a time; per tile compute the scores S = Q K^T,
// mask keys past the query (causal), update the running max m and sum l,
// rescale the output accumulator by exp(m_old - m_new), add P V; at the end
// divide by l.  Here:
//
//   CTA      64 queries of one (batch, head), 4 warps of 16 queries each.
//   staging  Q once, then K and V tiles of 64 keys double-buffered in shared
//            memory with cp.async (16-byte chunks, XOR-swizzled by row so
//            that ldmatrix reads are free of bank conflicts).
//   S        per warp 16 x 64 scores: ldmatrix fragments of Q (kept in
//            registers for the whole walk) and K, mma.sync m16n8k16.
//   softmax  in the base-2 domain: x = S * scale * log2(e); the row max over
//            a quad of lanes (__shfl_xor), p = 2^(x - m), alpha = 2^(m_old -
//            m_new); each lane keeps its part of l, summed over the quad at
//            the end.
//   P V      the score accumulators, rounded to the operand type, are the A
//            fragments of the second product directly (the m16n8 accumulator
//            layout is the m16k16 operand layout); V fragments come from
//            ldmatrix.trans.
//   output   O = acc / l, and optionally the natural-log logsumexp per query.
//
// A query with no visible key ends with l = 0: its output is 0/0 = NaN, the
// softmax of only -inf (its logsumexp is -inf).
#include "common.cuh"
#include "kernels.h"

#include <atomic>

namespace rwsm {

namespace {

constexpr int kAttBM = 64;          // queries per CTA
constexpr int kAttBN = 64;          // keys per tile
constexpr int kAttThreads = 128;    // 4 warps x 16 queries

template <typename T> struct MmaType;
template <> struct MmaType<BF16Bits> {
    __device__ static __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                     "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};
template <> struct MmaType<F16Bits> {
    __device__ static __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
    {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                     "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// 16-byte global -> shared copy; src_bytes 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all_groups()
{
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Byte offset of 16-byte chunk `c` of row `r` in a tile of D-element rows,
// chunks XOR-swizzled by the row's low 3 bits.
template <int D>
__device__ __forceinline__ uint32_t tile_off(int r, int c)
{
    return static_cast<uint32_t>(r * D * 2 + ((c ^ (r & 7)) << 4));
}

// Copy rows [row0, row0 + ROWS) of a [n][D] matrix into a swizzled tile;
// rows past n are zero.
template <int D, int ROWS>
__device__ __forceinline__ void load_tile(uint32_t smem, const unsigned short* g, int64_t row0,
                                          int64_t n, int tid)
{
    constexpr int CH = D / 8;                     // 16-byte chunks per row
    for (int i = tid; i < ROWS * CH; i += kAttThreads) {
        const int r = i / CH, c = i % CH;
        const int64_t gr = row0 + r;
        const bool ok = gr < n;
        const unsigned short* src = g + (ok ? gr : 0) * D + c * 8;
        cp_async16_zfill(smem + tile_off<D>(r, c), src, ok ? 16 : 0);
    }
}

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(kAttThreads)
attention_mma_kernel(const T* q, const T* k, const T* v, T* o, float* lse, int64_t bh,
                     int64_t n_q, int64_t n_k, float scale_log2, int64_t offset)
{
    constexpr int KS = D / 16;                    // k-steps over the head dimension
    constexpr int DB = D / 8;                     // 8-wide output column blocks
    extern __shared__ __align__(128) unsigned char att_smem[];
    const uint32_t s_base = smem_addr(att_smem);
    const uint32_t sQ = s_base;
    const uint32_t sK = sQ + kAttBM * D * 2;                  // 2 buffers
    const uint32_t sV = sK + 2 * kAttBN * D * 2;              // 2 buffers

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n_qt = (n_q + kAttBM - 1) / kAttBM;
    const int64_t b = blockIdx.x / n_qt;
    int64_t qt = blockIdx.x % n_qt;
    if (CAUSAL)
        qt = n_qt - 1 - qt;                       // longest tiles first
    if (b >= bh)
        return;
    const int64_t q0 = qt * kAttBM;
    const unsigned short* gq = reinterpret_cast<const unsigned short*>(q) + b * n_q * D;
    const unsigned short* gk = reinterpret_cast<const unsigned short*>(k) + b * n_k * D;
    const unsigned short* gv = reinterpret_cast<const unsigned short*>(v) + b * n_k * D;

    // Key tiles this query tile sees (causal: up to its last query's diagonal).
    int64_t n_kt = (n_k + kAttBN - 1) / kAttBN;
    if (CAUSAL) {
        const int64_t last = q0 + kAttBM - 1 + offset;        // last visible key
        const int64_t lim = last < 0 ? 0 : last / kAttBN + 1;
        n_kt = lim < n_kt ? lim : n_kt;
    }

    pdl_launch_dependents();
    pdl_wait();
    load_tile<D, kAttBM>(sQ, gq, q0, n_q, tid);
    if (n_kt > 0) {
        load_tile<D, kAttBN>(sK, gk, 0, n_k, tid);
        load_tile<D, kAttBN>(sV, gv, 0, n_k, tid);
    }
    cp_async_commit();

    const int r_a = lane >> 2, c_q = (lane & 3) * 2;          // fragment row / column
    const int64_t qi_a = q0 + warp * 16 + r_a, qi_b = qi_a + 8;
    float m_a = kNegInf, m_b = kNegInf, l_a = 0.0f, l_b = 0.0f;
    float acc[DB][4];
#pragma unroll
    for (int i = 0; i < DB; ++i)
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    uint32_t qa[KS][4];

    for (int64_t t = 0; t < n_kt; ++t) {
        cp_async_wait_all_groups();
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                const int mi = lane >> 3;
                const int row = warp * 16 + (lane & 7) + (mi & 1) * 8;
                ldsm_x4(qa[kk], sQ + tile_off<D>(row, kk * 2 + (mi >> 1)));
            }
        }
        if (t + 1 < n_kt) {
            const int nb = static_cast<int>((t + 1) & 1);
            load_tile<D, kAttBN>(sK + nb * kAttBN * D * 2, gk, (t + 1) * kAttBN, n_k, tid);
            load_tile<D, kAttBN>(sV + nb * kAttBN * D * 2, gv, (t + 1) * kAttBN, n_k, tid);
        }
        cp_async_commit();
        const uint32_t cK = sK + static_cast<uint32_t>(t & 1) * kAttBN * D * 2;
        const uint32_t cV = sV + static_cast<uint32_t>(t & 1) * kAttBN * D * 2;

        // ---- S = Q K^T for this warp's 16 queries and the tile's 64 keys
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int mi = lane >> 3;
                const int n = p * 16 + (lane & 7) + (mi >> 1) * 8;
                uint32_t bk[4];
                ldsm_x4(bk, cK + tile_off<D>(n, kk * 2 + (mi & 1)));
                MmaType<T>::mma(s[2 * p], qa[kk], bk[0], bk[1]);
                MmaType<T>::mma(s[2 * p + 1], qa[kk], bk[2], bk[3]);
            }
        }

        // ---- mask, running max, p = 2^(x - m)
        const int64_t k0 = t * kAttBN;
        const bool edge = k0 + kAttBN > n_k || (CAUSAL && k0 + kAttBN - 1 > q0 + warp * 16 + offset);
        float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float xa = s[nb][e] * scale_log2, xb = s[nb][2 + e] * scale_log2;
                if (edge) {
                    const int64_t j = k0 + nb * 8 + c_q + e;
                    if (j >= n_k || (CAUSAL && j > qi_a + offset)) xa = kNegInf;
                    if (j >= n_k || (CAUSAL && j > qi_b + offset)) xb = kNegInf;
                }
                s[nb][e] = xa;
                s[nb][2 + e] = xb;
                mx_a = fmaxf(mx_a, xa);
                mx_b = fmaxf(mx_b, xb);
            }
        }
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
        const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
        const float ref_a = mn_a == kNegInf ? 0.0f : mn_a;
        const float ref_b = mn_b == kNegInf ? 0.0f : mn_b;
        const float al_a = ex2_ftz(m_a - ref_a), al_b = ex2_ftz(m_b - ref_b);
        m_a = mn_a;
        m_b = mn_b;
        l_a *= al_a;
        l_b *= al_b;
#pragma unroll
        for (int i = 0; i < DB; ++i) {
            acc[i][0] *= al_a; acc[i][1] *= al_a;
            acc[i][2] *= al_b; acc[i][3] *= al_b;
        }
        // p, its partial row sums, and the A fragments of P (16-bit)
        uint32_t pa[4][4];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            const float p0 = ex2_ftz(s[nb][0] - ref_a), p1 = ex2_ftz(s[nb][1] - ref_a);
            const float p2 = ex2_ftz(s[nb][2] - ref_b), p3 = ex2_ftz(s[nb][3] - ref_b);
            l_a += p0 + p1;
            l_b += p2 + p3;
            const int ks = nb >> 1, hi = nb & 1;
            pa[ks][hi * 2 + 0] = Elem<T>::pack2(p0, p1);
            pa[ks][hi * 2 + 1] = Elem<T>::pack2(p2, p3);
        }

        // ---- acc += P V
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int mi = lane >> 3;
                const int kr = ks * 16 + (lane & 7) + (mi & 1) * 8;
                uint32_t bv[4];
                ldsm_x4_trans(bv, cV + tile_off<D>(kr, dp * 2 + (mi >> 1)));
                MmaType<T>::mma(acc[2 * dp], pa[ks], bv[0], bv[1]);
                MmaType<T>::mma(acc[2 * dp + 1], pa[ks], bv[2], bv[3]);
            }
        }
    }
    cp_async_wait_all_groups();

    // ---- O = acc / l; logsumexp = (m + log2 l) * ln 2
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    const float inv_a = 1.0f / l_a, inv_b = 1.0f / l_b;
    unsigned short* go = reinterpret_cast<unsigned short*>(o) + b * n_q * D;
#pragma unroll
    for (int db = 0; db < DB; ++db) {
        const int col = db * 8 + c_q;
        if (qi_a < n_q)
            *reinterpret_cast<uint32_t*>(go + qi_a * D + col) =
                Elem<T>::pack2(acc[db][0] * inv_a, acc[db][1] * inv_a);
        if (qi_b < n_q)
            *reinterpret_cast<uint32_t*>(go + qi_b * D + col) =
                Elem<T>::pack2(acc[db][2] * inv_b, acc[db][3] * inv_b);
    }
    if (lse && (lane & 3) == 0) {
        const float ln2 = 0.69314718055994531f;
        if (qi_a < n_q)
            lse[b * n_q + qi_a] = l_a > 0.0f ? (m_a + __log2f(l_a)) * ln2 : kNegInf;
        if (qi_b < n_q)
            lse[b * n_q + qi_b] = l_b > 0.0f ? (m_b + __log2f(l_b)) * ln2 : kNegInf;
    }
}

template <typename T, int D, bool CAUSAL>
cudaError_t launch_att(const AttentionProblem& p, cudaStream_t s)
{
    auto* kern = attention_mma_kernel<T, D, CAUSAL>;
    const int smem = (kAttBM + 4 * kAttBN) * D * 2;
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
    const int64_t n_qt = (p.n_q + kAttBM - 1) / kAttBM;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(n_qt * p.bh), 1, 1);
    cfg.blockDim = dim3(kAttThreads, 1, 1);
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
cudaError_t launch_att_d(const AttentionProblem& p, cudaStream_t s)
{
    return p.causal ? launch_att<T, D, true>(p, s) : launch_att<T, D, false>(p, s);
}

template <typename T>
cudaError_t launch_att_t(const AttentionProblem& p, cudaStream_t s)
{
    if (p.head_dim == 64) return launch_att_d<T, 64>(p, s);
    if (p.head_dim == 128) return launch_att_d<T, 128>(p, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_attention_mma(const AttentionProblem& p, cudaStream_t s)
{
    if (p.n_q * ((p.n_q + kAttBM - 1) / kAttBM) < 0 || p.bh * ((p.n_q + kAttBM - 1) / kAttBM) > 0x7fffffff)
        return cudaErrorInvalidValue;
    return p.dtype == SOFTMAX_BF16 ? launch_att_t<BF16Bits>(p, s) : launch_att_t<F16Bits>(p, s);
}

}  // namespace rwsm
