// The C ABI of librope_chain.so (declared in include/rope_chain.h): argument
// checks on the host, then launches on the caller's stream.  Nothing here
// allocates device memory or synchronises, except rc_read_device_faults.
#include "rope_chain.h"
#include "rc_internal.cuh"

#include <algorithm>
#include <numeric>
#include <cstdarg>
#include <cstdio>

namespace {

thread_local char g_err[512] = "";

rc_status fail(rc_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

rc_status ok() {
    g_err[0] = '\0';
    return RC_OK;
}

rc_status cuda_fail(cudaError_t e, const char *what) {
    return fail(RC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int num_sms_current() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (dev < 64 && cache[dev])
        return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < 64)
        cache[dev] = n;
    return n;
}

constexpr int64_t kMaxProjectRows = 65535LL * 128;

rc_status check_project_sizes(int32_t L, int64_t T, int32_t D, int32_t N) {
    if (L < 1 || L > 4096)
        return fail(RC_ERR_INVALID_ARG, "rc_kv_project: L=%d outside [1, 4096]", L);
    if (T < 0 || T > kMaxProjectRows)
        return fail(RC_ERR_INVALID_ARG, "rc_kv_project: T=%lld outside [0, %lld]", (long long)T,
                    (long long)kMaxProjectRows);
    if (D < 64 || D % 64 != 0)
        return fail(RC_ERR_UNSUPPORTED, "rc_kv_project: D=%d is not a positive multiple of 64", D);
    if (N < 128 || N % 128 != 0)
        return fail(RC_ERR_UNSUPPORTED, "rc_kv_project: N=%d is not a positive multiple of 128", N);
    return RC_OK;
}

}  // namespace

namespace {

// rc_kv_store and rc_kv_store_rows: layer l inserts layer_rows[l] rows
// (`rows` for every layer when layer_rows is NULL).
rc_status kv_store_impl(const char *fn, const uint16_t *k, const uint16_t *v,
                        int64_t k_layer_stride, int64_t k_row_stride, int64_t v_layer_stride,
                        int64_t v_row_stride, const int64_t *positions,
                        const int64_t *const *slots, const uint16_t *cos_sin,
                        int64_t max_position, uint16_t *const *caches, int32_t num_blocks,
                        int32_t block_size, int32_t H, int32_t L, float eps,
                        const int64_t *layer_rows, int64_t rows, int32_t *err,
                        cudaStream_t stream)
{
    if (H != 1 && H != 2 && H != 4 && H != 8 && H != 16 && H != 32)
        return fail(RC_ERR_UNSUPPORTED, "%s: H=%d is not a power of two <= 32", fn, H);
    if (L < 1 || L > 4096)
        return fail(RC_ERR_INVALID_ARG, "%s: L=%d outside [1, 4096]", fn, L);
    int64_t max_rows = 0;
    for (int32_t l = 0; l < L; ++l) {
        const int64_t r = layer_rows ? layer_rows[l] : rows;
        if (r < 0 || r > 0x7FFFFFFFLL)
            return fail(RC_ERR_INVALID_ARG, "%s: rows of layer %d = %lld outside [0, 2^31)", fn, l,
                        (long long)r);
        max_rows = std::max(max_rows, r);
    }
    if (num_blocks < 1 || block_size < 1 || (int64_t)num_blocks * block_size >= (1LL << 31))
        return fail(RC_ERR_INVALID_ARG,
                    "%s: need num_blocks, block_size >= 1 and num_blocks*block_size < 2^31", fn);
    if (!k || !v || !slots || !caches)
        return fail(RC_ERR_INVALID_ARG, "%s: k, v, slots and caches must not be NULL", fn);
    if (!aligned(k, 4) || !aligned(v, 4))
        return fail(RC_ERR_INVALID_ARG, "%s: k and v must be 4-byte aligned", fn);
    if (k_layer_stride < 0 || k_row_stride < 0 || v_layer_stride < 0 || v_row_stride < 0 ||
        (k_layer_stride | k_row_stride | v_layer_stride | v_row_stride) & 1)
        return fail(RC_ERR_INVALID_ARG, "%s: strides must be even and non-negative", fn);
    if (cos_sin) {
        if (!positions || !aligned(positions, 8))
            return fail(RC_ERR_INVALID_ARG, "%s: RoPE needs 8-byte aligned positions", fn);
        if (max_position < 1)
            return fail(RC_ERR_INVALID_ARG, "%s: max_position must be >= 1 with a table", fn);
        if (!aligned(cos_sin, 2))
            return fail(RC_ERR_INVALID_ARG, "%s: cos_sin must be 2-byte aligned", fn);
    }
    for (int32_t l = 0; l < L; ++l) {
        if (!slots[l])
            continue;
        if (!aligned(slots[l], 8))
            return fail(RC_ERR_INVALID_ARG, "%s: slots[%d] must be 8-byte aligned", fn, l);
        if (!caches[l] || !aligned(caches[l], 4))
            return fail(RC_ERR_INVALID_ARG, "%s: caches[%d] must be a 4-byte aligned pointer", fn, l);
    }
    if (max_rows == 0)
        return ok();

    // Layers go to the GPU in chunks of at most 8 (the pointer tables are
    // kernel parameters); a chunk whose layers all lack slots is skipped.
    for (int32_t first = 0; first < L; first += rc::kMaxLayersPerLaunch) {
        const int32_t n = std::min(rc::kMaxLayersPerLaunch, L - first);
        rc::StoreLaunch p{};
        bool any = false;
        int64_t chunk_rows = 0;
        for (int32_t i = 0; i < n; ++i) {
            const int64_t r = layer_rows ? layer_rows[first + i] : rows;
            p.slots[i] = r > 0 ? slots[first + i] : nullptr;
            p.caches[i] = caches[first + i];
            p.rows[i] = (int32_t)r;
            any = any || p.slots[i] != nullptr;
            if (p.slots[i])
                chunk_rows = std::max(chunk_rows, r);
        }
        if (!any)
            continue;
        p.k = k + first * k_layer_stride;
        p.v = v + first * v_layer_stride;
        p.k_layer_stride = k_layer_stride;
        p.k_row_stride = k_row_stride;
        p.v_layer_stride = v_layer_stride;
        p.v_row_stride = v_row_stride;
        p.positions = positions;
        p.cos_sin = cos_sin;
        p.max_position = max_position;
        p.capacity = (int64_t)num_blocks * block_size;
        p.block_size = block_size;
        p.grid_rows = (int32_t)chunk_rows;
        p.eps = eps;
        p.err = err;
        const cudaError_t e = rc::launch_kv_store(p, H, n, stream);
        if (e != cudaSuccess)
            return cuda_fail(e, fn);
    }
    return ok();
}

}  // namespace

namespace {

// The two norms' parameters of the option calls, checked and turned into
// the kernels' descriptors.
rc_status norm_descs(const char *fn, const rc_norm_params *hidden, const rc_norm_params *pre,
                     rc::NormDesc d[2])
{
    const rc_norm_params *np[2] = {hidden, pre};
    for (int i = 0; i < 2; ++i) {
        const rc_norm_params &n = *np[i];
        const char *which = i ? "pre" : "hidden";
        if (n.weight_dtype != RC_NORM_NONE && n.weight_dtype != RC_NORM_BF16 &&
            n.weight_dtype != RC_NORM_F32)
            return fail(RC_ERR_INVALID_ARG, "%s: %s weight_dtype=%d unknown", fn, which, n.weight_dtype);
        if ((n.weight_dtype == RC_NORM_NONE) != (n.weight == nullptr))
            return fail(RC_ERR_INVALID_ARG, "%s: %s weight must be NULL exactly when weight_dtype is "
                        "RC_NORM_NONE", fn, which);
        if (n.weight && !aligned(n.weight, 16))
            return fail(RC_ERR_INVALID_ARG, "%s: %s weight must be 16-byte aligned", fn, which);
        d[i].w = n.weight;
        d[i].fp32 = n.weight_dtype == RC_NORM_F32;
        d[i].input_scale = n.weight != nullptr && n.input_scale != 0;   // weightless: ignored
        d[i].center = n.gain_center;
        d[i].eps = n.eps;
    }
    return RC_OK;
}

// Whether a norm runs in the default kernel: no weight, or a bf16
// output-scale weight without a centre.
bool plain_norm(const rc::NormDesc &n) {
    return n.w == nullptr || (!n.fp32 && !n.input_scale && n.center == 0.0f);
}

// The norms kernel for two descriptors: the default kernel where both norms
// are plain, the option kernel otherwise.
cudaError_t launch_norms(const uint16_t *x, int64_t T, const rc::NormDesc d[2], int32_t L,
                         uint16_t *out, cudaStream_t stream, bool early = false)
{
    if (plain_norm(d[0]) && plain_norm(d[1]))
        return rc::launch_context_norms(x, T, static_cast<const uint16_t *>(d[0].w),
                                        static_cast<const uint16_t *>(d[1].w), L, d[0].eps,
                                        d[1].eps, out, stream, early);
    return rc::launch_context_norms_ex(x, T, d[0], d[1], L, out, stream, early);
}

}  // namespace

namespace rc {
void set_last_error(const char *msg) { snprintf(g_err, sizeof g_err, "%s", msg); }

rc_status check_project_call(const char *fn, const uint16_t *normed, const uint16_t *W,
                             int32_t w_layout, const uint16_t *out, int32_t L, int64_t T,
                             int32_t D, int32_t N)
{
    const rc_status s = check_project_sizes(L, T, D, N);
    if (s != RC_OK)
        return s;
    if (w_layout != RC_W_KN && w_layout != RC_W_NK)
        return fail(RC_ERR_INVALID_ARG, "%s: unknown weight layout %d", fn, w_layout);
    if (!normed || !W || !out)
        return fail(RC_ERR_INVALID_ARG, "%s: normed, W and out must not be NULL", fn);
    if (!aligned(normed, 16) || !aligned(W, 16) || !aligned(out, 16))
        return fail(RC_ERR_INVALID_ARG, "%s: operands must be 16-byte aligned", fn);
    if (T == 0)
        return RC_OK;
    const size_t obytes = (size_t)L * T * N * 2;
    if (overlap(out, obytes, normed, (size_t)L * T * D * 2) ||
        overlap(out, obytes, W, (size_t)L * D * N * 2))
        return fail(RC_ERR_INVALID_ARG, "%s: out overlaps an input", fn);
    return RC_OK;
}
}  // namespace rc

extern "C" {

const char *rc_last_error(void) { return g_err; }

int32_t rc_version(void) { return 100; }

rc_status rc_context_norms(const uint16_t *x, int64_t T, int32_t D, const uint16_t *hidden_w,
                           const uint16_t *pre_w, int32_t L, float eps, uint16_t *out,
                           cudaStream_t stream)
{
    if (D != rc::kHidden)
        return fail(RC_ERR_UNSUPPORTED, "rc_context_norms: D=%d, the row norm takes D=8192", D);
    if (T < 0 || T > 0x7FFFFFFFLL)
        return fail(RC_ERR_INVALID_ARG, "rc_context_norms: T=%lld outside [0, 2^31)", (long long)T);
    if (L < 1 || L > 64)
        return fail(RC_ERR_INVALID_ARG, "rc_context_norms: L=%d outside [1, 64]", L);
    if (!x || !out)
        return fail(RC_ERR_INVALID_ARG, "rc_context_norms: x and out must not be NULL");
    if (!aligned(x, 16) || !aligned(out, 16) || (hidden_w && !aligned(hidden_w, 16)) ||
        (pre_w && !aligned(pre_w, 16)))
        return fail(RC_ERR_INVALID_ARG, "rc_context_norms: x, out and weights must be 16-byte aligned");
    const size_t xbytes = (size_t)T * D * 2, obytes = (size_t)L * T * D * 2;
    if (T > 0 && overlap(x, xbytes, out, obytes))
        return fail(RC_ERR_INVALID_ARG, "rc_context_norms: out overlaps x");
    if (T == 0)
        return ok();
    const cudaError_t e = rc::launch_context_norms(x, T, hidden_w, pre_w, L, eps, eps, out, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "rc_context_norms launch");
    return ok();
}

rc_status rc_context_norms_ex(const uint16_t *x, int64_t T, int32_t D,
                              const rc_norm_params *hidden, const rc_norm_params *pre, int32_t L,
                              uint16_t *out, cudaStream_t stream)
{
    const char *fn = "rc_context_norms_ex";
    if (D != rc::kHidden)
        return fail(RC_ERR_UNSUPPORTED, "%s: D=%d, the row norm takes D=8192", fn, D);
    if (T < 0 || T > 0x7FFFFFFFLL)
        return fail(RC_ERR_INVALID_ARG, "%s: T=%lld outside [0, 2^31)", fn, (long long)T);
    if (L < 1 || L > 64)
        return fail(RC_ERR_INVALID_ARG, "%s: L=%d outside [1, 64]", fn, L);
    if (!x || !out || !hidden || !pre)
        return fail(RC_ERR_INVALID_ARG, "%s: x, out, hidden and pre must not be NULL", fn);
    if (!aligned(x, 16) || !aligned(out, 16))
        return fail(RC_ERR_INVALID_ARG, "%s: x and out must be 16-byte aligned", fn);
    rc::NormDesc d[2];
    const rc_status st = norm_descs(fn, hidden, pre, d);
    if (st != RC_OK)
        return st;
    const size_t xbytes = (size_t)T * D * 2, obytes = (size_t)L * T * D * 2;
    if (T > 0 && overlap(x, xbytes, out, obytes))
        return fail(RC_ERR_INVALID_ARG, "%s: out overlaps x", fn);
    if (T == 0)
        return ok();
    const cudaError_t e = launch_norms(x, T, d, L, out, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "rc_context_norms_ex launch");
    return ok();
}

size_t rc_kv_project_workspace_size(int32_t L, int64_t T, int32_t D, int32_t N)
{
    if (check_project_sizes(L, T, D, N) != RC_OK || T == 0)
        return 0;
    const int sms = num_sms_current();
    if (sms <= 0)
        return 0;
    return rc::plan_kv_project(L, T, D, N, sms, SIZE_MAX).workspace;
}

size_t rc_kv_project_workspace_size_sms(int32_t L, int64_t T, int32_t D, int32_t N,
                                        int32_t num_sms)
{
    if (check_project_sizes(L, T, D, N) != RC_OK || T == 0 || num_sms < 1)
        return 0;
    return rc::plan_kv_project(L, T, D, N, num_sms, SIZE_MAX).workspace;
}

rc_status rc_kv_project_plan(int32_t L, int64_t T, int32_t D, int32_t N, int32_t num_sms,
                             size_t workspace_bytes, rc_project_plan *plan)
{
    const rc_status s = check_project_sizes(L, T, D, N);
    if (s != RC_OK)
        return s;
    if (num_sms < 1 || plan == nullptr)
        return fail(RC_ERR_INVALID_ARG, "rc_kv_project_plan: need num_sms >= 1 and a plan to fill");
    const rc::ProjectPlan p = rc::plan_kv_project(L, T, D, N, num_sms, workspace_bytes);
    plan->kernel = !p.pair ? 0 : (p.splits == 1 ? 2 : 1);
    plan->splits = p.splits;
    plan->tail_splits = p.tail_tiles > 0 ? p.tail_splits : 0;
    plan->dynamic_tiles = p.tile_ctr_offset >= 0 ? 1 : 0;
    plan->tail_row0 = p.tail_tiles > 0 ? p.tail_row0 : T;
    plan->workspace_bytes = p.workspace;
    return ok();
}

rc_status rc_kv_project(const uint16_t *normed, const uint16_t *W, int32_t w_layout, uint16_t *out,
                        int32_t L, int64_t T, int32_t D, int32_t N, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream)
{
    const rc_status s = rc::check_project_call("rc_kv_project", normed, W, w_layout, out, L, T, D, N);
    if (s != RC_OK)
        return s;
    if (workspace && !aligned(workspace, 16))
        return fail(RC_ERR_INVALID_ARG, "rc_kv_project: operands must be 16-byte aligned");
    if (T == 0)
        return ok();
    const size_t obytes = (size_t)L * T * N * 2;
    const int sms = num_sms_current();
    if (sms <= 0)
        return fail(RC_ERR_CUDA, "rc_kv_project: no current CUDA device");
    const rc::ProjectPlan plan =
        rc::plan_kv_project(L, T, D, N, sms, workspace ? workspace_bytes : 0);
    if (plan.workspace > 0 && overlap(workspace, plan.workspace, out, obytes))
        return fail(RC_ERR_INVALID_ARG, "rc_kv_project: workspace overlaps out");
    const char *why = "launch";
    const cudaError_t e = rc::launch_kv_project(normed, W, w_layout == RC_W_NK, out, L, T, D, N,
                                                plan, static_cast<float *>(workspace), stream, &why);
    if (e != cudaSuccess)
        return cuda_fail(e, why);
    return ok();
}

rc_status rc_kv_store(const uint16_t *k, const uint16_t *v, int64_t k_layer_stride,
                      int64_t k_row_stride, int64_t v_layer_stride, int64_t v_row_stride,
                      const int64_t *positions, const int64_t *const *slots,
                      const uint16_t *cos_sin, int64_t max_position, uint16_t *const *caches,
                      int32_t num_blocks, int32_t block_size, int32_t H, int32_t L, float eps,
                      int64_t rows, int32_t *err, cudaStream_t stream)
{
    return kv_store_impl("rc_kv_store", k, v, k_layer_stride, k_row_stride, v_layer_stride,
                         v_row_stride, positions, slots, cos_sin, max_position, caches, num_blocks,
                         block_size, H, L, eps, nullptr, rows, err, stream);
}

rc_status rc_kv_store_rows(const uint16_t *k, const uint16_t *v, int64_t k_layer_stride,
                           int64_t k_row_stride, int64_t v_layer_stride, int64_t v_row_stride,
                           const int64_t *positions, const int64_t *const *slots,
                           const uint16_t *cos_sin, int64_t max_position, uint16_t *const *caches,
                           int32_t num_blocks, int32_t block_size, int32_t H, int32_t L, float eps,
                           const int64_t *layer_rows, int32_t *err, cudaStream_t stream)
{
    if (!layer_rows)
        return fail(RC_ERR_INVALID_ARG, "rc_kv_store_rows: layer_rows must not be NULL");
    return kv_store_impl("rc_kv_store_rows", k, v, k_layer_stride, k_row_stride, v_layer_stride,
                         v_row_stride, positions, slots, cos_sin, max_position, caches, num_blocks,
                         block_size, H, L, eps, layer_rows, 0, err, stream);
}

}  // extern "C"

namespace {

// Checks the store operands of the fused calls and fills a FusedStore.
rc_status fused_store_args(const char *fn, int32_t L, int64_t T, int32_t H,
                           const int64_t *positions, const int64_t *const *slots,
                           const uint16_t *cos_sin, int64_t max_position, uint16_t *const *caches,
                           int32_t num_blocks, int32_t block_size, float eps, int64_t rows,
                           int32_t *err, uint16_t *kv_out, rc::FusedStore *fs,
                           const int64_t *layer_rows = nullptr)
{
    if (L > rc::kMaxFusedLayers)
        return fail(RC_ERR_UNSUPPORTED, "%s: L=%d above %d", fn, L, rc::kMaxFusedLayers);
    if (!slots || !caches)
        return fail(RC_ERR_INVALID_ARG, "%s: slots and caches must not be NULL", fn);
    if (kv_out && !aligned(kv_out, 16))
        return fail(RC_ERR_INVALID_ARG, "%s: kv_out must be 16-byte aligned", fn);
    if (L < 1)
        return fail(RC_ERR_INVALID_ARG, "%s: L=%d below 1", fn, L);
    for (int32_t l = 0; l < L; ++l) {
        const int64_t r = layer_rows ? layer_rows[l] : rows;
        if (r < 0 || r > T)
            return fail(RC_ERR_INVALID_ARG, "%s: rows=%lld (layer %d) outside [0, T]", fn,
                        (long long)r, l);
    }
    if (num_blocks < 1 || block_size < 1 || (int64_t)num_blocks * block_size >= (1LL << 31))
        return fail(RC_ERR_INVALID_ARG,
                    "%s: need num_blocks, block_size >= 1 and num_blocks*block_size < 2^31", fn);
    if (cos_sin) {
        if (!positions || !aligned(positions, 8))
            return fail(RC_ERR_INVALID_ARG, "%s: RoPE needs 8-byte aligned positions", fn);
        if (max_position < 1)
            return fail(RC_ERR_INVALID_ARG, "%s: max_position must be >= 1 with a table", fn);
        if (!aligned(cos_sin, 16))
            return fail(RC_ERR_INVALID_ARG, "%s: cos_sin must be 16-byte aligned", fn);
    }
    *fs = rc::FusedStore{};
    for (int32_t l = 0; l < L; ++l) {
        if (slots[l]) {
            if (!aligned(slots[l], 8))
                return fail(RC_ERR_INVALID_ARG, "%s: slots[%d] must be 8-byte aligned", fn, l);
            if (!caches[l] || !aligned(caches[l], 16))
                return fail(RC_ERR_INVALID_ARG, "%s: caches[%d] must be a 16-byte aligned pointer", fn, l);
        }
        fs->slots[l] = slots[l];
        fs->caches[l] = caches[l];
    }
    fs->positions = positions;
    fs->cos_sin = cos_sin;
    fs->max_position = max_position;
    fs->capacity = (int64_t)num_blocks * block_size;
    fs->block_size = block_size;
    fs->H = H;
    for (int32_t l = 0; l < L; ++l)
        fs->rows[l] = (int32_t)(layer_rows ? layer_rows[l] : rows);
    fs->eps = eps;
    fs->err = err;
    fs->kv_out = kv_out;
    return RC_OK;
}

bool supported_heads(int32_t H) {
    return H == 1 || H == 2 || H == 4 || H == 8 || H == 16 || H == 32;
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// Bytes the whole-chain call keeps ahead of the split-K partials.
size_t context_kv_fixed_bytes(bool pair, int32_t L, int64_t T, int32_t D) {
    return pair ? round256((size_t)T * D * 2) + round256((size_t)T * 4)
                : round256((size_t)L * T * D * 2);
}

}  // namespace

namespace {

// rc_kv_project_store and rc_kv_project_store_rows.
rc_status kv_project_store_impl(const char *fn, const uint16_t *normed, const uint16_t *W,
                                int32_t w_layout, int32_t L, int64_t T, int32_t D, int32_t H,
                                const int64_t *positions, const int64_t *const *slots,
                                const uint16_t *cos_sin, int64_t max_position,
                                uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                                float eps, const int64_t *layer_rows, int64_t rows, int32_t *err,
                                uint16_t *kv_out, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream)
{
    if (!supported_heads(H))
        return fail(RC_ERR_UNSUPPORTED, "%s: H=%d is not a power of two <= 32", fn, H);
    const int32_t N = 2 * H * rc::kHeadDim;
    rc_status st = check_project_sizes(L, T, D, N);
    if (st != RC_OK)
        return st;
    if (w_layout != RC_W_KN && w_layout != RC_W_NK)
        return fail(RC_ERR_INVALID_ARG, "%s: unknown weight layout %d", fn, w_layout);
    if (!normed || !W)
        return fail(RC_ERR_INVALID_ARG, "%s: normed and W must not be NULL", fn);
    if (!aligned(normed, 16) || !aligned(W, 16) || (workspace && !aligned(workspace, 16)))
        return fail(RC_ERR_INVALID_ARG, "%s: normed, W and workspace must be 16-byte aligned", fn);
    rc::FusedStore fs;
    st = fused_store_args(fn, L, T, H, positions, slots, cos_sin, max_position, caches, num_blocks,
                          block_size, eps, rows, err, kv_out, &fs, layer_rows);
    if (st != RC_OK)
        return st;
    if (T == 0)
        return ok();
    if (kv_out && overlap(kv_out, (size_t)L * T * N * 2, normed, (size_t)L * T * D * 2))
        return fail(RC_ERR_INVALID_ARG, "%s: kv_out overlaps normed", fn);
    const int sms = num_sms_current();
    if (sms <= 0)
        return fail(RC_ERR_CUDA, "%s: no current CUDA device", fn);
    const rc::ProjectPlan plan =
        rc::plan_kv_project(L, T, D, N, sms, workspace ? workspace_bytes : 0);
    if (plan.splits == 1 && !plan.pair && !kv_out)
        return fail(RC_ERR_INVALID_ARG,
                    "%s: at these sizes the store reads the projection from kv_out; "
                    "pass kv_out or a workspace of rc_kv_project_workspace_size() bytes", fn);
    const char *why = "launch";
    const cudaError_t e = rc::launch_kv_project_store(normed, W, w_layout == RC_W_NK, L, T, D, N, plan,
                                                      static_cast<float *>(workspace), fs, stream, &why);
    if (e != cudaSuccess)
        return cuda_fail(e, why);
    return ok();
}

}  // namespace

extern "C" {

rc_status rc_kv_project_store(const uint16_t *normed, const uint16_t *W, int32_t w_layout,
                              int32_t L, int64_t T, int32_t D, int32_t H,
                              const int64_t *positions, const int64_t *const *slots,
                              const uint16_t *cos_sin, int64_t max_position,
                              uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                              float eps, int64_t rows, int32_t *err, uint16_t *kv_out,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return kv_project_store_impl("rc_kv_project_store", normed, W, w_layout, L, T, D, H, positions,
                                 slots, cos_sin, max_position, caches, num_blocks, block_size, eps,
                                 nullptr, rows, err, kv_out, workspace, workspace_bytes, stream);
}

rc_status rc_kv_project_store_rows(const uint16_t *normed, const uint16_t *W, int32_t w_layout,
                                   int32_t L, int64_t T, int32_t D, int32_t H,
                                   const int64_t *positions, const int64_t *const *slots,
                                   const uint16_t *cos_sin, int64_t max_position,
                                   uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                                   float eps, const int64_t *layer_rows, int32_t *err,
                                   uint16_t *kv_out, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream)
{
    if (!layer_rows)
        return fail(RC_ERR_INVALID_ARG, "rc_kv_project_store_rows: layer_rows must not be NULL");
    return kv_project_store_impl("rc_kv_project_store_rows", normed, W, w_layout, L, T, D, H,
                                 positions, slots, cos_sin, max_position, caches, num_blocks,
                                 block_size, eps, layer_rows, 0, err, kv_out, workspace,
                                 workspace_bytes, stream);
}

namespace {

// The whole-chain calls run the forming projection, which takes every tile
// itself: their plans have no tail launch (the workspace holds split-K
// partials, or the persistent kernel's tile counter).
rc::ProjectPlan whole_chain_plan(int32_t L, int64_t T, int32_t D, int32_t N, int sms,
                                 size_t workspace_bytes) {
    return rc::plan_kv_project(L, T, D, N, sms, workspace_bytes, false);
}

}  // namespace

size_t rc_context_kv_workspace_size(int32_t L, int64_t T, int32_t D, int32_t H)
{
    if (!supported_heads(H) || D != rc::kHidden || L < 1 || L > rc::kMaxFusedLayers)
        return 0;
    const int32_t N = 2 * H * rc::kHeadDim;
    if (check_project_sizes(L, T, D, N) != RC_OK || T == 0)
        return 0;
    const int sms = num_sms_current();
    if (sms <= 0)
        return 0;
    const rc::ProjectPlan plan = whole_chain_plan(L, T, D, N, sms, SIZE_MAX);
    return context_kv_fixed_bytes(plan.pair, L, T, D) + plan.workspace;
}

rc_status rc_context_kv(const uint16_t *x, int64_t T, int32_t D, const uint16_t *hidden_w,
                        const uint16_t *pre_w, int32_t L, float eps, const uint16_t *W,
                        int32_t w_layout, int32_t H, const int64_t *positions,
                        const int64_t *const *slots, const uint16_t *cos_sin, int64_t max_position,
                        uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                        int64_t rows, int32_t *err, uint16_t *kv_out, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream)
{
    const char *fn = "rc_context_kv";
    if (D != rc::kHidden)
        return fail(RC_ERR_UNSUPPORTED, "%s: D=%d, the row norm takes D=8192", fn, D);
    if (!supported_heads(H))
        return fail(RC_ERR_UNSUPPORTED, "%s: H=%d is not a power of two <= 32", fn, H);
    const int32_t N = 2 * H * rc::kHeadDim;
    rc_status st = check_project_sizes(L, T, D, N);
    if (st != RC_OK)
        return st;
    if (w_layout != RC_W_KN && w_layout != RC_W_NK)
        return fail(RC_ERR_INVALID_ARG, "%s: unknown weight layout %d", fn, w_layout);
    if (!x || !W || !workspace)
        return fail(RC_ERR_INVALID_ARG, "%s: x, W and workspace must not be NULL", fn);
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(workspace, 256) ||
        (hidden_w && !aligned(hidden_w, 16)) || (pre_w && !aligned(pre_w, 16)))
        return fail(RC_ERR_INVALID_ARG,
                    "%s: x, W and weights must be 16-byte aligned, workspace 256-byte aligned", fn);
    rc::FusedStore fs;
    st = fused_store_args(fn, L, T, H, positions, slots, cos_sin, max_position, caches, num_blocks,
                          block_size, eps, rows, err, kv_out, &fs);
    if (st != RC_OK)
        return st;
    if (T == 0)
        return ok();
    const int sms = num_sms_current();
    if (sms <= 0)
        return fail(RC_ERR_CUDA, "%s: no current CUDA device", fn);
    const bool pair = rc::plan_kv_project(L, T, D, N, sms, 0).pair;
    const size_t fixed = context_kv_fixed_bytes(pair, L, T, D);
    if (workspace_bytes < fixed)
        return fail(RC_ERR_INVALID_ARG, "%s: the workspace needs at least %zu bytes (%zu given)", fn,
                    fixed, workspace_bytes);
    char *wsb = static_cast<char *>(workspace);
    float *partials = reinterpret_cast<float *>(wsb + fixed);
    const rc::ProjectPlan plan = whole_chain_plan(L, T, D, N, sms, workspace_bytes - fixed);
    const char *why = "launch";
    cudaError_t e;
    if (plan.pair) {
        uint16_t *z = reinterpret_cast<uint16_t *>(wsb);
        float *r2 = reinterpret_cast<float *>(wsb + round256((size_t)T * D * 2));
        e = rc::launch_row_prep(x, T, hidden_w, eps, z, r2, stream);
        if (e == cudaSuccess)
            e = rc::launch_kv_from_rows(z, r2, T, pre_w, W, w_layout == RC_W_NK, L, N, plan, partials,
                                        fs, stream, &why);
    } else {
        if (plan.splits == 1 && !kv_out)
            return fail(RC_ERR_INVALID_ARG,
                        "%s: at these sizes the store reads the projection from kv_out; pass kv_out "
                        "or a workspace of rc_context_kv_workspace_size() bytes", fn);
        uint16_t *normed = reinterpret_cast<uint16_t *>(wsb);
        e = rc::launch_context_norms(x, T, hidden_w, pre_w, L, eps, eps, normed, stream);
        if (e == cudaSuccess)
            e = rc::launch_kv_project_store(normed, W, w_layout == RC_W_NK, L, T, D, N, plan, partials,
                                            fs, stream, &why);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, why);
    return ok();
}

rc_status rc_context_rows(const uint16_t *x, int64_t T, int32_t D, const uint16_t *hidden_w,
                          float eps, uint16_t *z, float *r2, cudaStream_t stream)
{
    const char *fn = "rc_context_rows";
    if (D != rc::kHidden)
        return fail(RC_ERR_UNSUPPORTED, "%s: D=%d, the row norm takes D=8192", fn, D);
    if (T < 0 || T > 0x7FFFFFFFLL)
        return fail(RC_ERR_INVALID_ARG, "%s: T=%lld outside [0, 2^31)", fn, (long long)T);
    if (!x || !z || !r2)
        return fail(RC_ERR_INVALID_ARG, "%s: x, z and r2 must not be NULL", fn);
    if (!aligned(x, 16) || !aligned(z, 16) || !aligned(r2, 4) || (hidden_w && !aligned(hidden_w, 16)))
        return fail(RC_ERR_INVALID_ARG, "%s: x, z and hidden_w must be 16-byte aligned", fn);
    if (T > 0 && overlap(x, (size_t)T * D * 2, z, (size_t)T * D * 2))
        return fail(RC_ERR_INVALID_ARG, "%s: z overlaps x", fn);
    if (T == 0)
        return ok();
    const cudaError_t e = rc::launch_row_prep(x, T, hidden_w, eps, z, r2, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "rc_context_rows launch");
    return ok();
}

rc_status rc_context_kv_from_rows(const uint16_t *z, const float *r2, int64_t T, int32_t D,
                                  const uint16_t *pre_w, int32_t L, float eps, const uint16_t *W,
                                  int32_t w_layout, int32_t H, const int64_t *positions,
                                  const int64_t *const *slots, const uint16_t *cos_sin,
                                  int64_t max_position, uint16_t *const *caches,
                                  int32_t num_blocks, int32_t block_size, int64_t rows,
                                  int32_t *err, uint16_t *kv_out, void *workspace,
                                  size_t workspace_bytes, cudaStream_t stream)
{
    const char *fn = "rc_context_kv_from_rows";
    if (D != rc::kHidden)
        return fail(RC_ERR_UNSUPPORTED, "%s: D=%d, the rows are 8192 wide", fn, D);
    if (!supported_heads(H))
        return fail(RC_ERR_UNSUPPORTED, "%s: H=%d is not a power of two <= 32", fn, H);
    const int32_t N = 2 * H * rc::kHeadDim;
    rc_status st = check_project_sizes(L, T, D, N);
    if (st != RC_OK)
        return st;
    if (w_layout != RC_W_KN && w_layout != RC_W_NK)
        return fail(RC_ERR_INVALID_ARG, "%s: unknown weight layout %d", fn, w_layout);
    if (!z || !r2 || !W)
        return fail(RC_ERR_INVALID_ARG, "%s: z, r2 and W must not be NULL", fn);
    if (!aligned(z, 16) || !aligned(W, 16) || !aligned(r2, 4) || (pre_w && !aligned(pre_w, 16)) ||
        (workspace && !aligned(workspace, 16)))
        return fail(RC_ERR_INVALID_ARG, "%s: z, W, pre_w and workspace must be 16-byte aligned", fn);
    rc::FusedStore fs;
    st = fused_store_args(fn, L, T, H, positions, slots, cos_sin, max_position, caches, num_blocks,
                          block_size, eps, rows, err, kv_out, &fs);
    if (st != RC_OK)
        return st;
    if (T == 0)
        return ok();
    const int sms = num_sms_current();
    if (sms <= 0)
        return fail(RC_ERR_CUDA, "%s: no current CUDA device", fn);
    const rc::ProjectPlan plan = whole_chain_plan(L, T, D, N, sms, workspace ? workspace_bytes : 0);
    if (!plan.pair)
        return fail(RC_ERR_UNSUPPORTED,
                    "%s: needs T > 128 and H >= 2 (CTA-pair tiles); use rc_context_kv", fn);
    const char *why = "launch";
    const cudaError_t e = rc::launch_kv_from_rows(z, r2, T, pre_w, W, w_layout == RC_W_NK, L, N, plan,
                                                  static_cast<float *>(workspace), fs, stream, &why);
    if (e != cudaSuccess)
        return cuda_fail(e, why);
    return ok();
}

}  // extern "C"

namespace {

constexpr int32_t kMaxChunks = 16;
constexpr size_t kChunkCounterBytes = 256;     // one chunk's tile counter
// The automatic count: at most 4 chunks of 12 rounds of tiles or more each.
// Each chunk adds a partly idle last round and a start, which the overlap of
// the norms pays for only on long chunks (measured on one GB300: workload 5,
// 54 rounds, 4 chunks 2.8 % faster than one; workload 4, 34 rounds, 2
// chunks 1.7 % faster, 4 chunks 2 % slower).
constexpr int32_t kAutoChunks = 4;
constexpr int64_t kAutoChunkRounds = 12;
// With x in host memory the norms of a chunk wait for its rows to cross the
// host link: the count is chosen by the score in plan_row_chunks, in which a
// 256-row block of the first chunk costs as much as kHostBlockRounds idle
// rounds of tiles (fitted on GB300 to eight end-to-end steps, workloads 4
// and 5 at 2-12 chunks: the first chunk's rows cross the link at about
// 0.06 us a row, an idle round costs about 59 us).  An explicit request
// gets equal-sized chunks.
constexpr double kHostBlockRounds = 0.26;

// The first chunk's norms run alone (nothing to overlap them with), so the
// first chunk is about 1 / kFirstChunkDiv of the others' size (measured at
// workload 5: a half 1.9-3 % faster than equal chunks; a third, a quarter
// or a sixth no better than a half).
constexpr int64_t kFirstChunkDiv = 2;
// Chunk sizes snapped to whole rounds of tiles (measured: workload 5 1.4 %,
// workload 4 1.8 % faster than unsnapped halves).
constexpr bool kSnapRounds = true;

// Row chunks of rc_context_kv_chunked: chunk c holds rows [row0[c],
// row0[c + 1]), each boundary a multiple of 256.  More than one chunk only
// where every chunk's projection runs as persistent CTA pairs that need no
// workspace but their tile counter (no split-K partials, no tail launch);
// with the automatic count (requested <= 0) only where every chunk after the
// first also has eight rounds of tiles or more (dynamic tile order).
struct RowChunks {
    int32_t count;
    int64_t row0[kMaxChunks + 1];
};

RowChunks plan_row_chunks(int32_t L, int64_t T, int32_t D, int32_t N, int sms, int32_t requested,
                          bool x_on_host)
{
    const int64_t pairs = std::max(1, sms / 2);
    const int64_t blocks = (T + 255) / 256;
    int32_t most = std::min(requested, kMaxChunks);
    if (requested <= 0) {
        const int64_t tiles = (int64_t)L * blocks * (N / 256);
        most = (int32_t)std::min<int64_t>(kAutoChunks, tiles / (kAutoChunkRounds * pairs));
    }
    // x read over the host link: a chunk's norms take about as long as the
    // projection of an equal chunk, so the first chunk is not made smaller
    // (nor snapped larger), and chunks need not be long enough for the
    // dynamic tile order
    const int64_t div = x_on_host ? 1 : kFirstChunkDiv;
    auto fits = [&](int64_t rows, bool need_dyn) {
        const rc::ProjectPlan p = rc::plan_kv_project(L, rows, D, N, sms, kChunkCounterBytes);
        return p.pair && p.splits == 1 && p.tail_tiles == 0 && (!need_dyn || p.tile_ctr_offset >= 0);
    };
    // A chunk of b 256-row blocks has L * b * (N / 256) tiles; with b a
    // multiple of q its last round is full (no pair idle while the chunk
    // ends).  A chunk size snaps to the nearest multiple of q within a
    // quarter of it.
    const int64_t q = pairs / std::gcd(pairs, (int64_t)L * (N / 256));
    auto snap = [&](int64_t b) {
        const int64_t m = std::max<int64_t>(q, (b + q / 2) / q * q);
        return kSnapRounds && 4 * (m > b ? m - b : b - m) <= b ? m : b;
    };
    RowChunks out{};
    if (x_on_host && requested <= 0 && blocks >= 2) {
        // x over the host link: equal chunks, their count chosen to spend the
        // least on the first chunk, whose rows cross the link with nothing
        // to overlap them (kHostBlockRounds rounds of tiles per 256-row
        // block), plus the partly idle last round of every chunk's
        // projection
        // one chunk: every row crosses the link before its projection, which
        // then runs with split-K partials (no idle round) or as persistent
        // pairs (the idle part of its last round)
        const rc::ProjectPlan whole = rc::plan_kv_project(L, T, D, N, sms, SIZE_MAX);
        const int64_t whole_tiles = (int64_t)L * blocks * (N / 256);
        double best = kHostBlockRounds * (double)blocks +
                      (whole.splits > 1 || !whole.pair ? 0.0
                       : (double)((whole_tiles + pairs - 1) / pairs) - (double)whole_tiles / (double)pairs);
        for (int32_t n = 2; n <= kMaxChunks && n <= blocks; ++n) {
            const int64_t even = (blocks + n - 1) / n;
            RowChunks cand{};
            int32_t count = 0;
            int64_t b0 = 0;
            double score = kHostBlockRounds * (double)even;
            bool ok = true;
            while (b0 < blocks && ok) {
                const int64_t b = std::min(even, blocks - b0);
                const int64_t tiles = (int64_t)L * b * (N / 256);
                score += (double)((tiles + pairs - 1) / pairs) - (double)tiles / (double)pairs;
                ok = fits(std::min(T, (b0 + b) * 256) - b0 * 256, false);
                b0 += b;
                cand.row0[++count] = std::min(T, b0 * 256);
            }
            if (ok && count >= 2 && score < best - 1e-9) {
                cand.count = count;
                out = cand;
                best = score;
            }
        }
        if (out.count >= 2)
            return out;
        out = RowChunks{};
    }
    for (int32_t n = blocks >= 2 ? most : 1; n >= 2; --n) {
        // a first chunk of about per / div blocks, then n - 1 chunks sharing
        // the rest; the snapped size only where it leaves the last chunk
        // between half and one and a half of the others
        const int64_t per = (blocks * div + (n - 1) * div) / ((n - 1) * div + 1);
        const int64_t first0 = std::max<int64_t>(1, per / div);
        const int64_t first = std::min(blocks - 1, x_on_host ? first0 : snap(first0));
        const int64_t rest = blocks - first;
        const int64_t even = (rest + n - 2) / (n - 1);
        int64_t mid = snap(even);
        const int64_t last_snapped = rest - (int64_t)(n - 2) * mid;
        if (mid != even && !(2 * last_snapped >= mid && 2 * last_snapped <= 3 * mid))
            mid = even;
        int32_t count = 0;
        int64_t b0 = 0;
        out.row0[0] = 0;
        while (b0 < blocks && count < kMaxChunks) {
            int64_t b = std::max<int64_t>(1, count == 0 ? first : mid);
            if (count == n - 1 || b0 + b >= blocks)
                b = blocks - b0;                     // the last chunk takes the rest
            b0 += b;
            out.row0[++count] = std::min(T, b0 * 256);
        }
        bool ok = count >= 2 && b0 >= blocks;
        for (int32_t c = 0; ok && c < count; ++c)
            ok = fits(out.row0[c + 1] - out.row0[c], requested <= 0 && !x_on_host && c > 0);
        if (ok) {
            out.count = count;
            return out;
        }
    }
    out.count = 1;
    out.row0[0] = 0;
    out.row0[1] = T;
    return out;
}

rc_status chunked_sizes(const char *fn, int32_t L, int64_t T, int32_t D, int32_t H) {
    if (D != rc::kHidden)
        return fail(RC_ERR_UNSUPPORTED, "%s: D=%d, the row norm takes D=8192", fn, D);
    if (!supported_heads(H))
        return fail(RC_ERR_UNSUPPORTED, "%s: H=%d is not a power of two <= 32", fn, H);
    if (L < 1 || L > rc::kMaxFusedLayers)
        return fail(RC_ERR_UNSUPPORTED, "%s: L=%d outside [1, %d]", fn, L, rc::kMaxFusedLayers);
    return check_project_sizes(L, T, D, 2 * H * rc::kHeadDim);
}

// Workspace of rc_context_kv_chunked: the normed rows, then room for a tile
// counter per chunk (the most chunks a call makes) or the projection's
// workspace (one chunk), whichever is larger: the same for x in device or
// host memory.
size_t chunked_workspace(int32_t L, int64_t T, int32_t D, int32_t N, int sms) {
    const size_t normed = round256((size_t)L * T * D * 2);
    const rc::ProjectPlan p = rc::plan_kv_project(L, T, D, N, sms, SIZE_MAX);
    // single CTAs without a K split store from a bf16 copy of the projection
    const size_t kv = p.splits == 1 && !p.pair ? round256((size_t)L * T * N * 2) : 0;
    return normed + std::max({kChunkCounterBytes * kMaxChunks, p.workspace, kv});
}

// Whether x is page-locked host memory (read by the norms over the host
// link).
bool on_host(const void *x) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, x) != cudaSuccess) {
        cudaGetLastError();                       // not sticky: clear it
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// rc_context_kv_chunked and rc_context_kv_chunked_ex: the norms given by d,
// then the projection + store with the K-norm's eps, by row chunks; layer l
// stores its first layer_rows[l] rows (`rows` for every layer when NULL).
rc_status chunked_impl(const char *fn, const uint16_t *x, int64_t T, int32_t D,
                       const rc::NormDesc d[2], int32_t L, float eps, const uint16_t *W,
                       int32_t w_layout, int32_t H, const int64_t *positions,
                       const int64_t *const *slots, const uint16_t *cos_sin, int64_t max_position,
                       uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                       const int64_t *layer_rows, int64_t rows, int32_t *err, int32_t chunks,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    rc_status st = chunked_sizes(fn, L, T, D, H);
    if (st != RC_OK)
        return st;
    const int32_t N = 2 * H * rc::kHeadDim;
    if (w_layout != RC_W_KN && w_layout != RC_W_NK)
        return fail(RC_ERR_INVALID_ARG, "%s: unknown weight layout %d", fn, w_layout);
    if (!x || !W || !workspace)
        return fail(RC_ERR_INVALID_ARG, "%s: x, W and workspace must not be NULL", fn);
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(workspace, 256))
        return fail(RC_ERR_INVALID_ARG, "%s: x and W must be 16-byte aligned, workspace 256-byte "
                    "aligned", fn);
    rc::FusedStore fs;
    st = fused_store_args(fn, L, T, H, positions, slots, cos_sin, max_position, caches, num_blocks,
                          block_size, eps, rows, err, nullptr, &fs, layer_rows);
    if (st != RC_OK)
        return st;
    if (T == 0)
        return ok();
    const int sms = num_sms_current();
    if (sms <= 0)
        return fail(RC_ERR_CUDA, "%s: no current CUDA device", fn);
    const bool x_on_host = on_host(x);
    // With x in device memory, norm options beyond the default kernel's keep
    // one chunk unless more are asked for: below 16384 rows the option
    // kernel reads each weight row from L2 once per row (the kernel that
    // stages them takes 64 KB of shared memory and so cannot run beside a
    // projection CTA), and beside the projection that costs more than the
    // overlap gains (workload 5 with FP32 gains: 3398-3410 us in 4 chunks,
    // 3159-3169 us in one).
    if (chunks <= 0 && !x_on_host && !(plain_norm(d[0]) && plain_norm(d[1])))
        chunks = 1;
    const RowChunks rcn = plan_row_chunks(L, T, D, N, sms, chunks, x_on_host);
    const size_t nbytes = round256((size_t)L * T * D * 2);
    const size_t need = rcn.count > 1 ? nbytes + kChunkCounterBytes * rcn.count : nbytes;
    if (workspace_bytes < need)
        return fail(RC_ERR_INVALID_ARG, "%s: the workspace needs at least %zu bytes (%zu given)", fn,
                    need, workspace_bytes);
    if (overlap(workspace, workspace_bytes, x, (size_t)T * D * 2) ||
        overlap(workspace, workspace_bytes, W, (size_t)L * D * N * 2))
        return fail(RC_ERR_INVALID_ARG, "%s: the workspace overlaps x or W", fn);
    char *wsb = static_cast<char *>(workspace);
    uint16_t *normed = reinterpret_cast<uint16_t *>(wsb);
    const bool nk = w_layout == RC_W_NK;
    const char *why = "launch";
    cudaError_t e;
    if (rcn.count == 1) {
        const size_t avail = workspace_bytes - nbytes;
        const rc::ProjectPlan plan = rc::plan_kv_project(L, T, D, N, sms, avail);
        if (plan.splits == 1 && !plan.pair) {
            // single CTAs without a K split: the projection goes through a
            // bf16 copy in the workspace, which the store kernel then reads
            const size_t kvb = round256((size_t)L * T * N * 2);
            if (avail < kvb)
                return fail(RC_ERR_INVALID_ARG,
                            "%s: the workspace needs at least %zu bytes (%zu given)", fn,
                            nbytes + kvb, workspace_bytes);
            fs.kv_out = reinterpret_cast<uint16_t *>(wsb + nbytes);
        }
        e = launch_norms(x, T, d, L, normed, stream);
        if (e == cudaSuccess)
            e = rc::launch_kv_project_store(normed, W, nk, L, T, D, N, plan,
                                            reinterpret_cast<float *>(wsb + nbytes), fs, stream, &why);
        if (e != cudaSuccess)
            return cuda_fail(e, why);
        return ok();
    }
    // Chunk c's norms run beside chunk c - 1's projection: launched right
    // behind it (PDL), they take the registers its persistent CTAs leave on
    // each SM.  Rows of different chunks share no buffer, so only the
    // projection of a chunk waits for that chunk's norms; the counters of
    // all chunks are zeroed first, so no memset separates the kernels.
    char *ctrs = wsb + nbytes;
    e = cudaMemsetAsync(ctrs, 0, kChunkCounterBytes * rcn.count, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "tile counter memset");
    for (int32_t c = 0; c < rcn.count; ++c) {
        const int64_t r0 = rcn.row0[c];
        const int64_t tc = rcn.row0[c + 1] - r0;
        uint16_t *normed_c = normed + (size_t)L * r0 * D;     // [L, tc, D]
        e = launch_norms(x + r0 * D, tc, d, L, normed_c, stream, c > 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "norms launch");
        rc::FusedStore fc = fs;
        if (fs.positions)
            fc.positions = fs.positions + r0;
        for (int32_t l = 0; l < L; ++l) {
            if (fs.slots[l])
                fc.slots[l] = fs.slots[l] + r0;
            fc.rows[l] = (int32_t)std::min<int64_t>(std::max<int64_t>(fs.rows[l] - r0, 0), tc);
        }
        rc::ProjectPlan plan = rc::plan_kv_project(L, tc, D, N, sms, kChunkCounterBytes);
        plan.ctr_zeroed = true;
        e = rc::launch_kv_project_store(normed_c, W, nk, L, tc, D, N, plan,
                                        reinterpret_cast<float *>(ctrs + kChunkCounterBytes * c), fc,
                                        stream, &why);
        if (e != cudaSuccess)
            return cuda_fail(e, why);
    }
    return ok();
}

}  // namespace

extern "C" {

int32_t rc_context_kv_chunks(int32_t L, int64_t T, int32_t D, int32_t H, int32_t chunks,
                             int32_t x_on_host, int32_t num_sms, int64_t *row0)
{
    if (chunked_sizes("rc_context_kv_chunks", L, T, D, H) != RC_OK || T == 0 || num_sms < 2)
        return 0;
    const RowChunks rcn =
        plan_row_chunks(L, T, D, 2 * H * rc::kHeadDim, num_sms, chunks, x_on_host != 0);
    if (row0)
        for (int32_t c = 0; c <= rcn.count; ++c)
            row0[c] = rcn.row0[c];
    return rcn.count;
}

size_t rc_context_kv_chunked_workspace_size(int32_t L, int64_t T, int32_t D, int32_t H,
                                            int32_t chunks)
{
    if (chunked_sizes("rc_context_kv_chunked_workspace_size", L, T, D, H) != RC_OK || T == 0)
        return 0;
    const int sms = num_sms_current();
    if (sms <= 0)
        return 0;
    (void)chunks;                                 // every chunk plan fits the same workspace
    return chunked_workspace(L, T, D, 2 * H * rc::kHeadDim, sms);
}

rc_status rc_context_kv_chunked(const uint16_t *x, int64_t T, int32_t D, const uint16_t *hidden_w,
                                const uint16_t *pre_w, int32_t L, float eps, const uint16_t *W,
                                int32_t w_layout, int32_t H, const int64_t *positions,
                                const int64_t *const *slots, const uint16_t *cos_sin,
                                int64_t max_position, uint16_t *const *caches, int32_t num_blocks,
                                int32_t block_size, int64_t rows, int32_t *err, int32_t chunks,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    const char *fn = "rc_context_kv_chunked";
    if ((hidden_w && !aligned(hidden_w, 16)) || (pre_w && !aligned(pre_w, 16)))
        return fail(RC_ERR_INVALID_ARG, "%s: weights must be 16-byte aligned", fn);
    // bf16 output-scale weights (or none), gain centre 0, one eps
    const rc::NormDesc d[2] = {{hidden_w, 0, 0, 0.0f, eps}, {pre_w, 0, 0, 0.0f, eps}};
    return chunked_impl(fn, x, T, D, d, L, eps, W, w_layout, H, positions, slots, cos_sin,
                        max_position, caches, num_blocks, block_size, nullptr, rows, err, chunks,
                        workspace, workspace_bytes, stream);
}

rc_status rc_context_kv_chunked_ex(const uint16_t *x, int64_t T, int32_t D,
                                   const rc_norm_params *hidden, const rc_norm_params *pre,
                                   int32_t L, const uint16_t *W, int32_t w_layout, int32_t H,
                                   const int64_t *positions, const int64_t *const *slots,
                                   const uint16_t *cos_sin, int64_t max_position,
                                   uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                                   float eps, const int64_t *layer_rows, int32_t *err,
                                   int32_t chunks, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream)
{
    const char *fn = "rc_context_kv_chunked_ex";
    if (!hidden || !pre)
        return fail(RC_ERR_INVALID_ARG, "%s: hidden and pre must not be NULL", fn);
    rc::NormDesc d[2];
    const rc_status st = norm_descs(fn, hidden, pre, d);
    if (st != RC_OK)
        return st;
    return chunked_impl(fn, x, T, D, d, L, eps, W, w_layout, H, positions, slots, cos_sin,
                        max_position, caches, num_blocks, block_size, layer_rows, T, err, chunks,
                        workspace, workspace_bytes, stream);
}

rc_status rc_device_address(const void *p, const void **dev)
{
    if (!p || !dev)
        return fail(RC_ERR_INVALID_ARG, "rc_device_address: p and dev must not be NULL");
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();                       // not sticky: clear it
        return fail(RC_ERR_INVALID_ARG, "rc_device_address: %p: %s", p, cudaGetErrorString(e));
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *dev = p;
        return ok();
    }
    if (a.type != cudaMemoryTypeHost)
        return fail(RC_ERR_INVALID_ARG,
                    "rc_device_address: %p is not device memory or page-locked host memory", p);
    void *d = nullptr;
    e = cudaHostGetDevicePointer(&d, const_cast<void *>(p), 0);
    if (e != cudaSuccess) {
        cudaGetLastError();                       // not sticky: clear it
        return fail(RC_ERR_INVALID_ARG,
                    "rc_device_address: page-locked memory at %p is not mapped for the device (%s)",
                    p, cudaGetErrorString(e));
    }
    *dev = d;
    return ok();
}

rc_status rc_read_device_faults(uint32_t *flags, int32_t clear)
{
    if (!flags)
        return fail(RC_ERR_INVALID_ARG, "rc_read_device_faults: flags must not be NULL");
    uint32_t project = 0, front = 0;
    cudaError_t e = rc::read_project_faults(&project, clear != 0);
    if (e == cudaSuccess)
        e = rc::read_front_faults(&front, clear != 0);
    if (e != cudaSuccess)
        return cuda_fail(e, "rc_read_device_faults");
    *flags = project | (front << 8);
    return ok();
}

rc_status rc_qkv_front(const uint16_t *hidden, int32_t M, int32_t D, const uint16_t *W,
                       int32_t num_heads, int32_t num_kv_heads, const int64_t *positions,
                       const uint16_t *cos_sin, int64_t max_position, const int64_t *slots,
                       uint16_t *cache, int32_t num_blocks, int32_t block_size, float eps,
                       uint16_t *out, uint16_t *raw_out, int32_t *err, cudaStream_t stream)
{
    const char *fn = "rc_qkv_front";
    if (M < 0 || M > 16)
        return fail(RC_ERR_UNSUPPORTED, "%s: M=%d outside [0, 16] (the decode front takes 1 to 16 "
                    "tokens)", fn, M);
    if (D < 64 || D % 64 != 0)
        return fail(RC_ERR_UNSUPPORTED, "%s: D=%d is not a positive multiple of 64", fn, D);
    if (num_heads < 1 || num_kv_heads < 1 || num_heads > 4096 || num_kv_heads > 4096)
        return fail(RC_ERR_INVALID_ARG, "%s: num_heads=%d, num_kv_heads=%d outside [1, 4096]", fn,
                    num_heads, num_kv_heads);
    if (!hidden || !W || !out)
        return fail(RC_ERR_INVALID_ARG, "%s: hidden, W and out must not be NULL", fn);
    if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(out, 16) || (raw_out && !aligned(raw_out, 16)))
        return fail(RC_ERR_INVALID_ARG, "%s: hidden, W, out and raw_out must be 16-byte aligned", fn);
    if (cos_sin) {
        if (!positions || !aligned(positions, 8))
            return fail(RC_ERR_INVALID_ARG, "%s: RoPE needs 8-byte aligned positions", fn);
        if (max_position < 1)
            return fail(RC_ERR_INVALID_ARG, "%s: max_position must be >= 1 with a table", fn);
        if (!aligned(cos_sin, 2))
            return fail(RC_ERR_INVALID_ARG, "%s: cos_sin must be 2-byte aligned", fn);
    }
    if (slots) {
        if (!aligned(slots, 8) || !cache || !aligned(cache, 4))
            return fail(RC_ERR_INVALID_ARG, "%s: slots need 8-byte alignment and a 4-byte aligned "
                        "cache", fn);
        if (num_blocks < 1 || block_size < 1 || (int64_t)num_blocks * block_size >= (1LL << 31))
            return fail(RC_ERR_INVALID_ARG,
                        "%s: need num_blocks, block_size >= 1 and num_blocks*block_size < 2^31", fn);
    }
    const int64_t N = 64LL * (2 * num_heads + 2 * num_kv_heads);
    if (overlap(out, (size_t)M * N * 2, W, (size_t)N * D * 2) ||
        overlap(out, (size_t)M * N * 2, hidden, (size_t)M * D * 2) ||
        (raw_out && overlap(raw_out, (size_t)M * N * 2, out, (size_t)M * N * 2)))
        return fail(RC_ERR_INVALID_ARG, "%s: out (or raw_out) overlaps an input or the other output", fn);
    if (M == 0)
        return ok();
    const int sms = num_sms_current();
    if (sms <= 0)
        return fail(RC_ERR_CUDA, "%s: no current CUDA device", fn);
    const char *why = "launch";
    const cudaError_t e = rc::launch_qkv_front(hidden, M, D, W, num_heads, num_kv_heads, positions,
                                               cos_sin, max_position, slots, cache,
                                               slots ? num_blocks : 1, slots ? block_size : 1, eps,
                                               out, raw_out, err, sms, stream, &why);
    if (e != cudaSuccess)
        return cuda_fail(e, why);
    return ok();
}

}  // extern "C"
