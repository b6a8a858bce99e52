// C ABI of libsoftmax (declared in include/softmax.h): argument validation,
// device description cache, dispatch to the path launchers, host-buffer
// staging, status strings.  No C++ exception crosses this boundary and the
// library allocates no memory.
#include "attention_pp.h"
#include "kernels.h"

#include <cmath>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace rwsm {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceCache {
    std::once_flag once[kMaxDevices];
    softmax_device_desc_t desc[kMaxDevices];
    int status[kMaxDevices];
};

DeviceCache& device_cache()
{
    static DeviceCache c;
    return c;
}

std::atomic<uint64_t> g_launches{0};

int query_device(int dev, softmax_device_desc_t* d)
{
    auto attr = [dev](cudaDeviceAttr a, int* v) { return cudaDeviceGetAttribute(v, a, dev); };
    if (attr(cudaDevAttrMultiProcessorCount, &d->sm_count) != cudaSuccess ||
        attr(cudaDevAttrMaxThreadsPerMultiProcessor, &d->max_threads_per_sm) != cudaSuccess ||
        attr(cudaDevAttrMaxSharedMemoryPerMultiprocessor, &d->max_smem_per_sm) != cudaSuccess ||
        attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, &d->max_smem_per_block_optin) != cudaSuccess ||
        attr(cudaDevAttrMaxRegistersPerMultiprocessor, &d->regs_per_sm) != cudaSuccess ||
        attr(cudaDevAttrComputeCapabilityMajor, &d->cc_major) != cudaSuccess ||
        attr(cudaDevAttrComputeCapabilityMinor, &d->cc_minor) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    d->max_cluster = 1;
    if (d->cc_major == 10 && d->cc_minor == 3) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur == dev)
            d->max_cluster = max_cluster_size_row_slices();
    }
    return SOFTMAX_OK;
}

// Description of the current device, queried once per device.
int current_device(softmax_device_desc_t* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_UNSUPPORTED;
    }
    if (dev < 0 || dev >= kMaxDevices)
        return SOFTMAX_ERR_UNSUPPORTED;
    DeviceCache& c = device_cache();
    std::call_once(c.once[dev], [&] { c.status[dev] = query_device(dev, &c.desc[dev]); });
    if (c.status[dev] != SOFTMAX_OK)
        return SOFTMAX_ERR_UNSUPPORTED;
    *out = c.desc[dev];
    return SOFTMAX_OK;
}

// Occupancy cache: resident CTAs of one kernel on the current device.
struct OccEntry {
    const void* kernel;
    int dev, threads, smem, ctas;
};
std::mutex g_occ_mu;
OccEntry g_occ[256];
int g_occ_n = 0;

}  // namespace

// Validate softmax_options_t and copy it into the problem (NULL: defaults).
int apply_options(const softmax_options_t* o, Problem* p)
{
    if (!o)
        return SOFTMAX_OK;
    // scale * log2(e) must stay finite in float: 0 < scale <= 2^127 (rejects NaN).
    if (!(o->scale > 0.0f) || !(o->scale <= 0x1p127f))
        return SOFTMAX_ERR_INVALID_ARG;
    if (o->causal != 0 && o->causal != 1)
        return SOFTMAX_ERR_INVALID_ARG;
    const int64_t lim = int64_t{1} << 62;
    if (o->causal_offset >= lim || o->causal_offset <= -lim)
        return SOFTMAX_ERR_INVALID_ARG;
    p->scale = o->scale;
    p->causal = o->causal;
    // Rows are < n_rows, so a period of n_rows or more is the same as n_rows;
    // clamped, (row mod period) + offset + 1 stays far inside int64.
    const int64_t whole = p->n_rows > 0 ? p->n_rows : 1;
    p->causal_period = o->causal_period > 0 && o->causal_period < whole ? o->causal_period : whole;
    p->causal_offset = o->causal_offset;
    return SOFTMAX_OK;
}

namespace {

int launch_path(const Problem& p, const softmax_plan_t& plan, cudaStream_t s)
{
    cudaError_t err = cudaErrorInvalidValue;
    switch (plan.path) {
    case SOFTMAX_PATH_WARP:
        err = plan.bulk_copy ? launch_tile_rows(p, plan, s) : launch_warp_rows(p, plan, s);
        break;
    case SOFTMAX_PATH_CTA:
    case SOFTMAX_PATH_CLUSTER: err = launch_row_slices(p, plan, s); break;
    case SOFTMAX_PATH_TWOPASS:
        err = plan.bulk_copy ? launch_stream_rows(p, plan, s) : launch_twopass(p, plan, s);
        break;
    default: break;
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    return SOFTMAX_OK;
}

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count_current()
{
    softmax_device_desc_t d;
    return current_device(&d) == SOFTMAX_OK ? d.sm_count : 1;
}

int resident_ctas(const void* kernel, int threads, int smem_bytes)
{
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> g(g_occ_mu);
        for (int i = 0; i < g_occ_n; ++i)
            if (g_occ[i].kernel == kernel && g_occ[i].dev == dev && g_occ[i].threads == threads &&
                g_occ[i].smem == smem_bytes)
                return g_occ[i].ctas;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem_bytes) !=
            cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int ctas = per_sm * sm_count_current();
    std::lock_guard<std::mutex> g(g_occ_mu);
    if (g_occ_n < 256)
        g_occ[g_occ_n++] = OccEntry{kernel, dev, threads, smem_bytes, ctas};
    return ctas;
}

}  // namespace rwsm

using rwsm::Problem;

extern "C" {

int softmax_abi_version(void) { return SOFTMAX_ABI_VERSION; }

uint64_t softmax_launch_count(void) { return rwsm::g_launches.load(); }

const char* softmax_status_string(int status)
{
    switch (status) {
    case SOFTMAX_OK: return "ok";
    case SOFTMAX_ERR_INVALID_ARG: return "invalid argument";
    case SOFTMAX_ERR_UNSUPPORTED: return "unsupported device or shape";
    case SOFTMAX_ERR_CUDA: return "CUDA error";
    case SOFTMAX_ERR_DEVICE_TIMEOUT: return "kernel gave up a bounded wait";
    default: return "unknown status";
    }
}

int softmax_plan(const softmax_device_desc_t* dev, const void* in, const void* out,
                 int64_t n_rows, int64_t n_cols, int64_t in_row_stride, int64_t out_row_stride,
                 int dtype, int path, softmax_plan_t* plan)
{
    if (!plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const Problem p{in, const_cast<void*>(out), n_rows, n_cols, in_row_stride, out_row_stride,
                    dtype};
    softmax_device_desc_t d;
    if (dev) {
        d = *dev;
    } else {
        const int st = rwsm::validate(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype);
        if (st != SOFTMAX_OK)
            return st;
        const int ds = rwsm::current_device(&d);
        if (ds != SOFTMAX_OK)
            return ds;
    }
    return rwsm::make_plan(d, p, path, plan);
}

int softmax_plan_format(const softmax_plan_t* plan, char* buf, size_t len)
{
    static const char* names[] = {"warp", "cta", "cluster", "twopass"};
    if (!plan)
        return 0;
    const char* name = (plan->path >= 0 && plan->path <= 3) ? names[plan->path] : "?";
    return std::snprintf(buf, len,
                         "path=%s dtype=%s vec=%d out_vec=%d bulk=%d threads=%d cluster=%d "
                         "rows_per_warp=%d chunks=%d slice_cols=%lld stages=%d smem=%d grid=%lld "
                         "lanes_per_row=%d",
                         name, plan->dtype == SOFTMAX_F32 ? "f32" : plan->dtype == SOFTMAX_BF16 ? "bf16" : "f16",
                         plan->vec,
                         plan->out_vec, plan->bulk_copy, plan->threads, plan->cluster,
                         plan->rows_per_warp, plan->chunks,
                         static_cast<long long>(plan->slice_cols), plan->stages, plan->smem_bytes,
                         static_cast<long long>(plan->grid),
                         plan->lanes_per_row > 0 ? plan->lanes_per_row : 32);
}

int softmax_plan_describe(int64_t n_rows, int64_t n_cols, int dtype, char* buf, size_t len)
{
    if (len > 0 && !buf)
        return SOFTMAX_ERR_INVALID_ARG;
    if (len > 0)
        buf[0] = '\0';
    // Contiguous rows at a 256-byte aligned address, as a device allocator
    // returns them; the same buffer for input and output (in place), which
    // the scheduler treats like separate buffers.
    const void* at = reinterpret_cast<const void*>(uintptr_t{256});
    softmax_plan_t plan;
    const int st = softmax_plan(nullptr, at, at, n_rows, n_cols, n_cols, n_cols, dtype,
                                SOFTMAX_PATH_AUTO, &plan);
    if (st != SOFTMAX_OK)
        return st;
    softmax_plan_format(&plan, buf, len);
    return SOFTMAX_OK;
}

int softmax_rows_path(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                      int64_t in_row_stride, int64_t out_row_stride, int dtype,
                      void* stream, int path)
{
    return softmax_rows_ex(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype,
                           nullptr, path, stream);
}

int softmax_plan_check(const softmax_device_desc_t* dev, const void* in, const void* out,
                       int64_t n_rows, int64_t n_cols, int64_t in_row_stride,
                       int64_t out_row_stride, int dtype, const softmax_plan_t* plan)
{
    if (!plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const int st = rwsm::validate(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    softmax_device_desc_t d;
    if (dev) {
        d = *dev;
    } else {
        const int ds = rwsm::current_device(&d);
        if (ds != SOFTMAX_OK)
            return ds;
    }
    const Problem p{in, const_cast<void*>(out), n_rows, n_cols, in_row_stride, out_row_stride,
                    dtype};
    return rwsm::check_plan(d, p, *plan);
}

int softmax_rows_planned(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                         int64_t in_row_stride, int64_t out_row_stride, int dtype,
                         const softmax_plan_t* plan, void* stream)
{
    if (!plan)
        return SOFTMAX_ERR_INVALID_ARG;
    const int st = rwsm::validate(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    softmax_device_desc_t d;
    const int ds = rwsm::current_device(&d);
    if (ds != SOFTMAX_OK)
        return ds;
    const Problem p{in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype};
    const int cs = rwsm::check_plan(d, p, *plan);
    if (cs != SOFTMAX_OK)
        return cs;
    return rwsm::launch_path(p, *plan, static_cast<cudaStream_t>(stream));
}

int softmax_rows_ex(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                    int64_t in_row_stride, int64_t out_row_stride, int dtype,
                    const softmax_options_t* options, int path, void* stream)
{
    const int st = rwsm::validate(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (path < SOFTMAX_PATH_AUTO || path > SOFTMAX_PATH_TWOPASS)
        return SOFTMAX_ERR_INVALID_ARG;
    Problem p{in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype};
    const int os = rwsm::apply_options(options, &p);
    if (os != SOFTMAX_OK)
        return os;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    softmax_device_desc_t d;
    const int ds = rwsm::current_device(&d);
    if (ds != SOFTMAX_OK)
        return ds;
    softmax_plan_t plan;
    const int ps = rwsm::make_plan(d, p, path, &plan);
    if (ps != SOFTMAX_OK)
        return ps;
    return rwsm::launch_path(p, plan, static_cast<cudaStream_t>(stream));
}

int64_t softmax_visible_cols(const softmax_options_t* options, int64_t n_rows, int64_t n_cols,
                             int64_t row)
{
    if (n_rows < 0 || n_cols < 0 || row < 0 || row >= n_rows || n_rows > (int64_t{1} << 62))
        return -1;
    Problem p{nullptr, nullptr, n_rows, n_cols, n_cols, n_cols, SOFTMAX_F32};
    if (rwsm::apply_options(options, &p) != SOFTMAX_OK)
        return -1;
    return rwsm::logits_valid(rwsm::logits_of(p), row, n_cols);
}

int softmax_attention_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                              int64_t batch_heads, int64_t n_q, int64_t n_k, int64_t head_dim,
                              int dtype, const softmax_attention_options_t* options, void* stream)
{
    if (batch_heads < 0 || n_q < 0 || n_k < 0 || head_dim < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16 && dtype != SOFTMAX_F16)
        return SOFTMAX_ERR_INVALID_ARG;
    float scale = head_dim > 0 ? static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim)))
                               : 1.0f;
    int causal = 0, impl = 0;
    int64_t offset = 0;
    if (options) {
        if (!(options->scale > 0.0f) || !(options->scale <= 0x1p127f))
            return SOFTMAX_ERR_INVALID_ARG;
        if (options->causal != 0 && options->causal != 1)
            return SOFTMAX_ERR_INVALID_ARG;
        const int64_t big = int64_t{1} << 62;
        if (options->causal_offset >= big || options->causal_offset <= -big)
            return SOFTMAX_ERR_INVALID_ARG;
        if (options->impl < 0 || options->impl > 3)
            return SOFTMAX_ERR_INVALID_ARG;
        scale = options->scale;
        causal = options->causal;
        offset = options->causal_offset;
        impl = options->impl;
    }
    if (batch_heads == 0 || n_q == 0)
        return SOFTMAX_OK;
    if (dtype == SOFTMAX_F32 || (head_dim != 64 && head_dim != 128))
        return SOFTMAX_ERR_UNSUPPORTED;
    if (!q || !o || (n_k > 0 && (!k || !v)))           // no key: k and v may be NULL
        return SOFTMAX_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    if (!a16(q) || !a16(k) || !a16(v) || !a16(o) || (lse && reinterpret_cast<uintptr_t>(lse) % 4))
        return SOFTMAX_ERR_INVALID_ARG;
    // Sizes: every extent in bytes must fit comfortably in int64.
    const int64_t lim = INT64_MAX / 4;
    if (n_q > lim / head_dim / batch_heads || (n_k > 0 && n_k > lim / head_dim / batch_heads))
        return SOFTMAX_ERR_INVALID_ARG;
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(o);
    const uintptr_t o1 = o0 + static_cast<uintptr_t>(batch_heads * n_q * head_dim * 2);
    auto hits = [&](const void* p, int64_t n) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        const uintptr_t e = a + static_cast<uintptr_t>(batch_heads * n * head_dim * 2);
        return a < o1 && o0 < e;
    };
    if ((q != o && hits(q, n_q)) || hits(k, n_k) || hits(v, n_k))
        return SOFTMAX_ERR_INVALID_ARG;            // o may be q itself, nothing else
    if (lse) {
        // The logsumexp rows are written while other CTAs still read q, k
        // and v and write o: lse may overlap none of them.
        const uintptr_t l0 = reinterpret_cast<uintptr_t>(lse);
        const uintptr_t l1 = l0 + static_cast<uintptr_t>(batch_heads * n_q) * sizeof(float);
        auto meets = [&](const void* a, int64_t n) {
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
            const uintptr_t a1 = a0 + static_cast<uintptr_t>(batch_heads * n * head_dim * 2);
            return a0 < l1 && l0 < a1;
        };
        if (meets(q, n_q) || meets(k, n_k) || meets(v, n_k) || meets(o, n_q))
            return SOFTMAX_ERR_INVALID_ARG;
    }
    // Grid sizes: one CTA per 64 queries of a head (mma.sync kernel), per 128
    // (single-tile tcgen05) or per 256 (ping-pong); a grid past 2^31 - 1 CTAs
    // cannot be launched.  With no key at all every kernel choice takes the
    // single-tile kernel (the ping-pong kernel's copy descriptors cannot
    // describe an empty K and V): rows of NaN, logsumexp -inf.
    auto grid_fits = [&](int64_t rows_per_cta) {
        return batch_heads <= 0x7fffffff / ((n_q + rows_per_cta - 1) / rows_per_cta);
    };
    if (n_k == 0 && (impl == 0 || impl == 3))
        impl = 2;
    if (!grid_fits(impl == 1 ? 64 : impl == 2 ? 128 : 256))
        return SOFTMAX_ERR_UNSUPPORTED;
    softmax_device_desc_t d;
    const int ds = rwsm::current_device(&d);
    if (ds != SOFTMAX_OK)
        return ds;
    const rwsm::AttentionProblem p{q, k, v, o, lse, batch_heads, n_q, n_k, head_dim, dtype,
                                   scale, causal, offset};
    // The library's choice: the ping-pong kernel (the fastest of the three
    // on GB300 at both head dimensions, causal or not); the single-tile
    // tcgen05 kernel where the ping-pong one's copy descriptors cannot be
    // made (no tensor-map encoder, sizes past their 32-bit coordinates).
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (impl == 1) {
        err = rwsm::launch_attention_mma(p, st);
    } else if (impl == 0 || impl == 3) {
        err = rwsm::launch_attention_pp(p, st);
        if (err == cudaErrorNotSupported) {
            if (impl == 3 || !grid_fits(128))
                return SOFTMAX_ERR_UNSUPPORTED;
            err = rwsm::launch_attention_tc(p, st);
        }
    } else {
        err = rwsm::launch_attention_tc(p, st);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    return SOFTMAX_OK;
}

int softmax_strided(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                    int64_t in_row_stride, int64_t in_col_stride, int64_t out_row_stride,
                    int64_t out_col_stride, int dtype, void* stream)
{
    if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16 && dtype != SOFTMAX_F16)
        return SOFTMAX_ERR_INVALID_ARG;
    if (n_rows < 0 || n_cols < 0 || in_row_stride < 0 || in_col_stride < 0 ||
        out_row_stride < 0 || out_col_stride < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    if (in_col_stride == 1 && out_col_stride == 1)          // contiguous rows
        return softmax_rows(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype, stream);
    if (!in || !out)
        return SOFTMAX_ERR_INVALID_ARG;
    const int64_t esz = dtype == SOFTMAX_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(in) % esz || reinterpret_cast<uintptr_t>(out) % esz)
        return SOFTMAX_ERR_INVALID_ARG;
    // Every output element distinct: rows nested in columns or columns in rows.
    const int64_t lim = INT64_MAX / 8;
    auto span = [&](int64_t rs, int64_t cs_) -> int64_t {   // last element index + 1
        if ((n_rows > 1 && rs > (lim - 1) / (n_rows - 1)) || (n_cols > 1 && cs_ > (lim - 1) / (n_cols - 1)))
            return -1;
        const int64_t a = (n_rows - 1) * rs, b = (n_cols - 1) * cs_;
        return a > lim - b - 1 ? -1 : a + b + 1;
    };
    const int64_t in_span = span(in_row_stride, in_col_stride);
    const int64_t out_span = span(out_row_stride, out_col_stride);
    if (in_span < 0 || out_span < 0)
        return SOFTMAX_ERR_INVALID_ARG;
    const bool distinct = n_rows == 1 || n_cols == 1 ||
                          (out_col_stride >= 1 && out_row_stride >= n_cols * out_col_stride) ||
                          (out_row_stride >= 1 && out_col_stride >= n_rows * out_row_stride);
    if (!distinct)
        return SOFTMAX_ERR_INVALID_ARG;
    // In place with the same layout, or no shared bytes at all.
    const uintptr_t i0 = reinterpret_cast<uintptr_t>(in), o0 = reinterpret_cast<uintptr_t>(out);
    const uintptr_t i1 = i0 + static_cast<uintptr_t>(in_span * esz);
    const uintptr_t o1 = o0 + static_cast<uintptr_t>(out_span * esz);
    const bool same = in == out && in_row_stride == out_row_stride && in_col_stride == out_col_stride;
    if (!same && i0 < o1 && o0 < i1)
        return SOFTMAX_ERR_INVALID_ARG;
    softmax_device_desc_t d;
    const int ds = rwsm::current_device(&d);
    if (ds != SOFTMAX_OK)
        return ds;
    const rwsm::StridedProblem p{in, out, n_rows, n_cols, in_row_stride, in_col_stride,
                                 out_row_stride, out_col_stride, dtype};
    rwsm::ColumnsShape sh{};
    if (in_row_stride == 1 && out_row_stride == 1)
        sh = rwsm::columns_stream_shape(p, d.sm_count, d.max_smem_per_sm);
    if (!sh.ok && ((in_row_stride == 1 && out_row_stride == 1) || n_rows == 1))
        sh = rwsm::columns_shape(p, d.max_smem_per_block_optin);
    if (rwsm::launch_strided(p, sh, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    return SOFTMAX_OK;
}

int softmax_backward_rows(const void* y, const void* dy, void* dx, int64_t n_rows,
                          int64_t n_cols, int64_t y_row_stride, int64_t dy_row_stride,
                          int64_t dx_row_stride, int dtype, void* stream)
{
    // dx against each input: the forward pass's rules (in place allowed,
    // partial overlap rejected); y and dy are both only read.
    int st = rwsm::validate(y, dx, n_rows, n_cols, y_row_stride, dx_row_stride, dtype);
    if (st != SOFTMAX_OK)
        return st;
    st = rwsm::validate(dy, dx, n_rows, n_cols, dy_row_stride, dx_row_stride, dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    softmax_device_desc_t d;
    const int ds = rwsm::current_device(&d);
    if (ds != SOFTMAX_OK)
        return ds;
    const int64_t esz = dtype == SOFTMAX_F32 ? 4 : 2;
    auto aligned = [&](const void* p, int64_t ld) {
        return reinterpret_cast<uintptr_t>(p) % 16 == 0 && (n_rows == 1 || (ld * esz) % 16 == 0);
    };
    const bool vec = aligned(y, y_row_stride) && aligned(dy, dy_row_stride) &&
                     aligned(dx, dx_row_stride);
    const rwsm::BackwardProblem p{y, dy, dx, n_rows, n_cols, y_row_stride, dy_row_stride,
                                  dx_row_stride, dtype};
    if (rwsm::launch_backward_rows(p, vec, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    return SOFTMAX_OK;
}

int softmax_rows(const void* in, void* out, int64_t n_rows, int64_t n_cols,
                 int64_t in_row_stride, int64_t out_row_stride, int dtype, void* stream)
{
    return softmax_rows_path(in, out, n_rows, n_cols, in_row_stride, out_row_stride, dtype,
                             stream, SOFTMAX_PATH_AUTO);
}

namespace {

// Device address of host memory the current device can access (pinned or
// registered host memory, or managed memory); NULL otherwise.
void* device_view(const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged)
        return nullptr;
    return a.devicePointer;
}

}  // namespace

int softmax_rows_host(const void* h_in, void* h_out, int64_t n_rows, int64_t n_cols,
                      int64_t in_row_stride, int64_t out_row_stride, int dtype,
                      void* d_in, void* d_out, void* stream)
{
    int st = rwsm::validate(h_in, h_out, n_rows, n_cols, in_row_stride, out_row_stride, dtype);
    if (st != SOFTMAX_OK)
        return st;
    if (n_rows == 0 || n_cols == 0)
        return SOFTMAX_OK;
    if (!d_in && !d_out) {
        // Direct: the kernel reads and writes the host rows over the host link.
        softmax_device_desc_t d;
        const int ds = rwsm::current_device(&d);
        if (ds != SOFTMAX_OK)
            return ds;
        const void* vin = device_view(h_in);
        void* vout = device_view(h_out);
        if (!vin || !vout)
            return SOFTMAX_ERR_INVALID_ARG;
        Problem p{vin, vout, n_rows, n_cols, in_row_stride, out_row_stride, dtype};
        p.no_bulk = true;
        softmax_plan_t plan;
        const int ps = rwsm::make_plan(d, p, SOFTMAX_PATH_AUTO, &plan);
        if (ps != SOFTMAX_OK)
            return ps;
        return rwsm::launch_path(p, plan, static_cast<cudaStream_t>(stream));
    }
    if (!d_in || !d_out)
        return SOFTMAX_ERR_INVALID_ARG;
    // Device side: dense rows; in place allowed.
    st = rwsm::validate(d_in, d_out, n_rows, n_cols, n_cols, n_cols, dtype);
    if (st != SOFTMAX_OK)
        return st;
    const size_t esz = dtype == SOFTMAX_F32 ? 4 : 2;
    const size_t width = static_cast<size_t>(n_cols) * esz;
    const size_t hp_in = n_rows > 1 ? static_cast<size_t>(in_row_stride) * esz : width;
    const size_t hp_out = n_rows > 1 ? static_cast<size_t>(out_row_stride) * esz : width;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpy2DAsync(d_in, width, h_in, hp_in, width, static_cast<size_t>(n_rows),
                          cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    st = softmax_rows(d_in, d_out, n_rows, n_cols, n_cols, n_cols, dtype, stream);
    if (st != SOFTMAX_OK)
        return st;
    if (cudaMemcpy2DAsync(h_out, hp_out, d_out, width, width, static_cast<size_t>(n_rows),
                          cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    return SOFTMAX_OK;
}

int softmax_selftest_wait_timeout(void* stream)
{
    softmax_device_desc_t d;
    const int ds = rwsm::current_device(&d);
    if (ds != SOFTMAX_OK)
        return ds;
    if (d.cc_major != 10 || d.cc_minor != 3)
        return SOFTMAX_ERR_UNSUPPORTED;
    if (rwsm::launch_selftest_wait(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    return SOFTMAX_OK;
}

int softmax_device_status(int clear)
{
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return SOFTMAX_ERR_CUDA;
    }
    const unsigned e = rwsm::read_error_row_slices(clear != 0) |
                       rwsm::read_error_tile_rows(clear != 0) |
                       rwsm::read_error_stream_rows(clear != 0) |
                       rwsm::read_error_columns_stream(clear != 0) |
                       rwsm::read_error_attention_tc(clear != 0);
    return e ? SOFTMAX_ERR_DEVICE_TIMEOUT : SOFTMAX_OK;
}

}  // extern "C"
