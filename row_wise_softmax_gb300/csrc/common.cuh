// Device helpers shared by the softmax kernels: element I/O, the base-2
// exponential, warp reductions, the (m, l) merge, and the cp.async.bulk /
// mbarrier primitives (inline PTX, sm_90+ forms, compiled for sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rwsm {

constexpr float kNegInf = -__builtin_inff();
// log2(e), rounded to binary32: e^d = 2^(d * log2 e).
constexpr float kLog2e = 1.4426950408889634f;
// Give up a bounded wait after this long (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// Longest suspension a bounded wait asks for in one try (the waiting thread
// resumes as soon as the phase completes).
constexpr uint32_t kWaitSuspendNs = 100000u;

// Error word written by a kernel that gave up a bounded wait.  Each kernel
// translation unit holds its own copy; the host reads and clears them all.
enum : unsigned { kErrMbarrierTimeout = 1u };

// ---------------------------------------------------------------- exp
// e^d = 2^(d * log2 e), with the hardware base-2 exponential (ex2.approx,
// flush-to-zero form: one instruction).
//
// exp_biased(d) = 2^64 * e^d for d <= 0.  The bias of 2^64 keeps the result a
// normal float down to d = -131 instead of -87, so a softmax output
// y = exp_biased(x - m) * (1 / (2^64 * l)) is formed by one correctly rounded
// multiply, which produces subnormal outputs where the exact value is
// subnormal.  Sums of biased terms stay below 2^95 for rows of up to 2^31
// elements.  d = 0 gives exactly 2^64 (a row's maximum maps to exactly 1 before
// the final scale); d = -inf gives +0; NaN stays NaN.
constexpr float kExpBias = 64.0f;

__device__ __forceinline__ float ex2_ftz(float t)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
    return y;
}

__device__ __forceinline__ float exp_biased(float d, float k)
{
    return ex2_ftz(fmaf(d, k, kExpBias));
}

// Unbiased e^(d * k / log2 e) for d <= 0, flushed to zero below 2^-126
// (rescale factors).
__device__ __forceinline__ float exp_ftz(float d, float k)
{
    return ex2_ftz(d * k);
}

// ------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Warp-wide maximum in one instruction (redux.sync on fp32, sm_100 family);
// like fmaxf, a NaN operand is ignored unless every lane holds NaN.  Faster
// than the shuffle tree in the kernels where a warp reduces whole rows on its
// own (measured); the CTA kernels keep the tree.
__device__ __forceinline__ float warp_max_redux(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- paired fp32 arithmetic (sm_100 family): one instruction computes two
// fp32 results, each rounded exactly as the scalar instruction would.
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1)
{
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// max(a, b, c) in one instruction; NaN operands are ignored as by fmaxf.
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Maximum of n floats (three-input max tree).
template <int N>
__device__ __forceinline__ float frag_max(const float* x, float m)
{
    int i = 0;
#pragma unroll
    for (; i + 1 < N; i += 2)
        m = max3(m, x[i], x[i + 1]);
    if constexpr (N % 2 == 1)
        m = fmaxf(m, x[N - 1]);
    return m;
}

// x[i] = exp_biased(x[i] - m, k) for n (even) elements, two per instruction,
// summed into s0 (even positions) and s1 (odd positions).
template <int N>
__device__ __forceinline__ void frag_exp_acc(float* x, float m, float k, float& s0, float& s1)
{
    static_assert(N % 2 == 0, "pairs");
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        float d0, d1;
        add2(d0, d1, x[i], x[i + 1], -m, -m);
        fma2(d0, d1, d0, d1, k, k, kExpBias, kExpBias);
        x[i] = ex2_ftz(d0);
        x[i + 1] = ex2_ftz(d1);
        add2(s0, s1, s0, s1, x[i], x[i + 1]);
    }
}

// Merge two online-softmax partials (m, l) and (m2, l2), where l is a sum of
// exp_biased(x - m) over the partial's elements:
//   M = max(m, m2),  l = l * e^(m - M) + l2 * e^(m2 - M).
// A partial whose m is -inf holds no finite element: its factor is e^-inf = 0.
// When both are -inf the reference point is 0 instead of M so that no
// -inf - (-inf) appears; a NaN carried in either l still propagates.  A
// factor below 2^-126 flushes to zero: that partial is then below 2^-62 of
// the merged sum, which is at least 2^64.
__device__ __forceinline__ void ml_merge(float& m, float& l, float m2, float l2, float k)
{
    const float M = fmaxf(m, m2);
    const float ref = (M == kNegInf) ? 0.0f : M;
    l = l * exp_ftz(m - ref, k) + l2 * exp_ftz(m2 - ref, k);
    m = M;
}

__device__ __forceinline__ void warp_ml_merge(float& m, float& l, float k)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        ml_merge(m, l, m2, l2, k);
    }
}

// ------------------------------------------------------------ element I/O
// Elements travel as fp32 in registers.  bf16 is the upper half of a binary32,
// so widening is a shift; fp16 (binary16) widens exactly with cvt.f32.f16.
// Narrowing rounds to nearest even.  A 16-bit Elem also provides the pair
// conversions of one 32-bit word (element 2i in the low half).
struct BF16Bits { unsigned short b; };
struct F16Bits { unsigned short b; };

template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kVec16 = 4;                 // elements per 16 bytes
    __device__ static __forceinline__ float load1(const float* p) { return __ldg(p); }
    __device__ static __forceinline__ void store1(float* p, float v) { *p = v; }
};

template <> struct Elem<BF16Bits> {
    static constexpr int kVec16 = 8;
    static constexpr unsigned short kNegInfBits = 0xff80u;
    __device__ static __forceinline__ float widen(unsigned short b)
    {
        return __uint_as_float(static_cast<unsigned>(b) << 16);
    }
    __device__ static __forceinline__ float load1(const BF16Bits* p)
    {
        return widen(__ldg(reinterpret_cast<const unsigned short*>(p)));
    }
    __device__ static __forceinline__ void store1(BF16Bits* p, float v)
    {
        unsigned short h;
        asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
        *reinterpret_cast<unsigned short*>(p) = h;
    }
    __device__ static __forceinline__ void unpack2(unsigned w, float& lo, float& hi)
    {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
    __device__ static __forceinline__ unsigned pack2(float lo, float hi)
    {
        unsigned w;   // cvt packs its first source operand into the upper half
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
        return w;
    }
};

template <> struct Elem<F16Bits> {
    static constexpr int kVec16 = 8;
    static constexpr unsigned short kNegInfBits = 0xfc00u;
    __device__ static __forceinline__ float widen(unsigned short b)
    {
        float f;
        asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(b));
        return f;
    }
    __device__ static __forceinline__ float load1(const F16Bits* p)
    {
        return widen(__ldg(reinterpret_cast<const unsigned short*>(p)));
    }
    __device__ static __forceinline__ void store1(F16Bits* p, float v)
    {
        unsigned short h;
        asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
        *reinterpret_cast<unsigned short*>(p) = h;
    }
    __device__ static __forceinline__ void unpack2(unsigned w, float& lo, float& hi)
    {
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
            : "=f"(lo), "=f"(hi) : "r"(w));
    }
    __device__ static __forceinline__ unsigned pack2(float lo, float hi)
    {
        unsigned w;   // cvt packs its first source operand into the upper half
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
        return w;
    }
};

// Load VEC consecutive elements starting at p (p aligned to VEC elements).
template <typename T, int VEC>
__device__ __forceinline__ void load_vec(const T* p, float* v)
{
    if constexpr (VEC == 1) {
        v[0] = Elem<T>::load1(p);
    } else if constexpr (sizeof(T) == 4) {
        if constexpr (VEC == 4) {
            const float4 q = __ldg(reinterpret_cast<const float4*>(p));
            v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else {
            static_assert(VEC == 2, "fp32 vector width");
            const float2 q = __ldg(reinterpret_cast<const float2*>(p));
            v[0] = q.x; v[1] = q.y;
        }
    } else {
        if constexpr (VEC == 8) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
            Elem<T>::unpack2(q.x, v[0], v[1]); Elem<T>::unpack2(q.y, v[2], v[3]);
            Elem<T>::unpack2(q.z, v[4], v[5]); Elem<T>::unpack2(q.w, v[6], v[7]);
        } else if constexpr (VEC == 4) {
            const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
            Elem<T>::unpack2(q.x, v[0], v[1]); Elem<T>::unpack2(q.y, v[2], v[3]);
        } else {
            static_assert(VEC == 2, "16-bit vector width");
            const unsigned q = __ldg(reinterpret_cast<const unsigned*>(p));
            Elem<T>::unpack2(q, v[0], v[1]);
        }
    }
}

// Store VEC consecutive elements v[j] * scale at p (p aligned to VEC elements).
template <typename T, int VEC>
__device__ __forceinline__ void store_vec(T* p, const float* v, float scale)
{
    if constexpr (VEC == 1) {
        Elem<T>::store1(p, v[0] * scale);
    } else if constexpr (sizeof(T) == 4) {
        if constexpr (VEC == 4) {
            *reinterpret_cast<float4*>(p) =
                make_float4(v[0] * scale, v[1] * scale, v[2] * scale, v[3] * scale);
        } else {
            *reinterpret_cast<float2*>(p) = make_float2(v[0] * scale, v[1] * scale);
        }
    } else {
        if constexpr (VEC == 8) {
            uint4 q;
            q.x = Elem<T>::pack2(v[0] * scale, v[1] * scale);
            q.y = Elem<T>::pack2(v[2] * scale, v[3] * scale);
            q.z = Elem<T>::pack2(v[4] * scale, v[5] * scale);
            q.w = Elem<T>::pack2(v[6] * scale, v[7] * scale);
            *reinterpret_cast<uint4*>(p) = q;
        } else if constexpr (VEC == 4) {
            uint2 q;
            q.x = Elem<T>::pack2(v[0] * scale, v[1] * scale);
            q.y = Elem<T>::pack2(v[2] * scale, v[3] * scale);
            *reinterpret_cast<uint2*>(p) = q;
        } else {
            *reinterpret_cast<unsigned*>(p) = Elem<T>::pack2(v[0] * scale, v[1] * scale);
        }
    }
}

// store_vec with the scaling done two elements per instruction (VEC even).
template <typename T, int VEC>
__device__ __forceinline__ void store_vec2(T* p, const float* v, float scale)
{
    static_assert(VEC % 2 == 0, "pairs");
    float y[VEC];
#pragma unroll
    for (int j = 0; j < VEC; j += 2)
        mul2(y[j], y[j + 1], v[j], v[j + 1], scale, scale);
    store_vec<T, VEC>(p, y, 1.0f);
}

// Masked forms: positions at or past `limit` read -inf and are not written.
template <typename T, int VEC, bool SKIP = false>
__device__ __forceinline__ void load_vec_masked(const T* row, int64_t col, int64_t limit, float* v)
{
    if (col + VEC <= limit) {
        load_vec<T, VEC>(row + col, v);
    } else if (SKIP && col >= limit) {           // wholly masked: no per-element tests
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            v[j] = kNegInf;
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            v[j] = (col + j < limit) ? Elem<T>::load1(row + col + j) : kNegInf;
    }
}

template <typename T, int VEC>
__device__ __forceinline__ void store_vec_masked(T* row, int64_t col, int64_t limit,
                                                 const float* v, float scale)
{
    if (col + VEC <= limit) {
        store_vec<T, VEC>(row + col, v, scale);
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (col + j < limit)
                Elem<T>::store1(row + col + j, v[j] * scale);
    }
}

// Shared-memory vector load of VEC elements (16 bytes when VEC == kVec16).
template <typename T, int VEC>
__device__ __forceinline__ void lds_vec(const T* p, float* v)
{
    if constexpr (sizeof(T) == 4) {
        static_assert(VEC == 4, "smem fp32 vector is 16 bytes");
        const float4 q = *reinterpret_cast<const float4*>(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
        static_assert(VEC == 8, "smem 16-bit vector is 16 bytes");
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        Elem<T>::unpack2(q.x, v[0], v[1]); Elem<T>::unpack2(q.y, v[2], v[3]);
        Elem<T>::unpack2(q.z, v[4], v[5]); Elem<T>::unpack2(q.w, v[6], v[7]);
    }
}

// ------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialisation: the next
// kernel in the stream may start its CTAs once every CTA of this grid has
// called pdl_launch_dependents() (done first thing: the grids are persistent
// and already resident), and every kernel calls pdl_wait() before its first
// global-memory access, which returns once the preceding grid has completed
// and its writes are visible.  Launched without the attribute (or after a
// kernel that does not trigger) both are no-ops in effect.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------- L2 eviction priorities
// Cache policies for loads and stores that should stay in L2 (evict_last:
// data read again soon) or leave it first (evict_first: streamed once).
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16-byte load / store with an L2 cache policy (p 16-byte aligned).
template <typename T>
__device__ __forceinline__ void load16_hint(const T* p, float* v, uint64_t pol)
{
    unsigned a, b, c, d;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "l"(p), "l"(pol));
    if constexpr (sizeof(T) == 4) {
        v[0] = __uint_as_float(a); v[1] = __uint_as_float(b);
        v[2] = __uint_as_float(c); v[3] = __uint_as_float(d);
    } else {
        Elem<T>::unpack2(a, v[0], v[1]); Elem<T>::unpack2(b, v[2], v[3]);
        Elem<T>::unpack2(c, v[4], v[5]); Elem<T>::unpack2(d, v[6], v[7]);
    }
}

template <typename T>
__device__ __forceinline__ void store16_hint(T* p, const float* v, float scale, uint64_t pol)
{
    unsigned a, b, c, d;
    if constexpr (sizeof(T) == 4) {
        a = __float_as_uint(v[0] * scale); b = __float_as_uint(v[1] * scale);
        c = __float_as_uint(v[2] * scale); d = __float_as_uint(v[3] * scale);
    } else {
        a = Elem<T>::pack2(v[0] * scale, v[1] * scale); b = Elem<T>::pack2(v[2] * scale, v[3] * scale);
        c = Elem<T>::pack2(v[4] * scale, v[5] * scale); d = Elem<T>::pack2(v[6] * scale, v[7] * scale);
    }
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
                 :: "l"(p), "r"(a), "r"(b), "r"(c), "r"(d), "l"(pol) : "memory");
}

// ------------------------------------------------- mbarrier + bulk copies
__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

// Raise the transaction count the current phase waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Bytes to bulk-copy of a span (16-byte aligned start) whose first `keep`
// elements take part in the softmax and whose first `inb` elements lie inside
// the row (or its padding before the next row): whole 16-byte granules up to
// the one that holds the last kept element when that granule is in bounds,
// else only the whole granules below it (the rest is read with plain loads).
// Elements copied past `keep` are never used.
template <typename T>
__device__ __forceinline__ uint32_t span_copy_bytes(int64_t keep, int64_t inb)
{
    const uint64_t b = static_cast<uint64_t>(keep) * sizeof(T);
    const uint64_t up = (b + 15u) & ~uint64_t{15};
    return static_cast<uint32_t>(up <= static_cast<uint64_t>(inb) * sizeof(T) ? up : (b & ~uint64_t{15}));
}

// Global -> shared bulk copy completing on an mbarrier.  dst, src 16-byte
// aligned; bytes a nonzero multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Bulk prefetch of global memory into L2 (no destination, no completion):
// src 16-byte aligned, bytes a nonzero multiple of 16.  L2 is the point of
// coherence for device memory, so lines prefetched before a preceding grid
// has finished writing them are updated by those writes: a kernel may warm
// L2 with its first inputs before griddepcontrol.wait.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// The same copy with an L2 cache policy (createpolicy) for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended for up to `hint_ns`
// nanoseconds while the phase is incomplete (it resumes as soon as the phase
// completes), so a waiting warp issues few instructions.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

// Wait for the mbarrier phase with the given parity to complete, for at most
// kWaitLimitNs (checked every iteration; each iteration suspends at most
// kWaitSuspendNs).  Returns false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait_suspend(bar, parity, kWaitSuspendNs))
            return true;
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return false;
}

}  // namespace rwsm

// ------------------------------------------- CTA and cluster (m, l) reductions
#include <cooperative_groups.h>

namespace rwsm {

// Reduce every thread's (m, l) partial over the CTA; all threads return the
// CTA's (m, l).  red_m / red_l hold THREADS/32 floats; the caller separates
// consecutive uses with a __syncthreads().
template <int THREADS>
__device__ __forceinline__ void cta_ml_reduce(float& m, float& l, float* red_m, float* red_l,
                                              float k)
{
    constexpr int NW = THREADS / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_ml_merge(m, l, k);
    if (lane == 0) {
        red_m[warp] = m;
        red_l[warp] = l;
    }
    __syncthreads();
    m = lane < NW ? red_m[lane] : kNegInf;
    l = lane < NW ? red_l[lane] : 0.0f;
    warp_ml_merge(m, l, k);
}

// Exchange the CTA partials of a cluster through distributed shared memory:
// thread 0 publishes (m, l) in part[slot], the cluster barrier (release /
// acquire) makes all of them visible, then each warp reads the cs partials
// (lane k from CTA rank k) and merges them.  Every thread of every CTA ends
// with the row's (m, l).  part has two slots, used alternately by consecutive
// rows, so a slot is rewritten only after the next barrier has shown that
// every peer finished reading it.
__device__ __forceinline__ void cluster_ml_reduce(float& m, float& l, float2* part,
                                                  int slot, int cs, float k)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    if (threadIdx.x == 0)
        part[slot] = make_float2(m, l);
    cluster.sync();
    const int lane = threadIdx.x & 31;
    float pm = kNegInf, pl = 0.0f;
    if (lane < cs) {
        const float2 q = *cluster.map_shared_rank(part + slot, lane);
        pm = q.x;
        pl = q.y;
    }
    warp_ml_merge(pm, pl, k);
    m = pm;
    l = pl;
}

}  // namespace rwsm
