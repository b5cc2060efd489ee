// C-ABI entry points of liblidx: host-side argument validation, kernel
// dispatch and error reporting.  Nothing here allocates device memory or
// synchronises, except idx_device_status(), which is documented to.
#include <stdarg.h>
#include <stdio.h>

#include <cmath>
#include <mutex>
#include <string>

#include "lidx_internal.cuh"

namespace lidx {
namespace {

thread_local std::string t_last_error;

idx_status fail(idx_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

idx_status from_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return IDX_OK;
    if (e == cudaErrorNotSupported) return fail(IDX_ERR_UNSUPPORTED, "%s: unsupported shape", what);
    return fail(IDX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// device status word: first data-dependent fault any kernel recorded
__device__ int g_device_status = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// device address of g_device_status on the current device (looked up once per device)
int* status_ptr() {
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

bool valid_dtype(int t) { return t == IDX_F32 || t == IDX_F16 || t == IDX_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

idx_status check_batch(const idx_batch& b, const char* what) {
    if (b.n_seq < 0) return fail(IDX_ERR_INVALID_ARG, "%s: n_seq < 0", what);
    if (b.n_q_per_seq < 1) return fail(IDX_ERR_INVALID_ARG, "%s: n_q_per_seq < 1", what);
    if (b.max_n_kv < 0) return fail(IDX_ERR_INVALID_ARG, "%s: max_n_kv < 0", what);
    if (b.n_seq > 0 && !b.n_kv) return fail(IDX_ERR_INVALID_ARG, "%s: n_kv is NULL", what);
    if (!b.kv_start && b.kv_seq_stride < 0)
        return fail(IDX_ERR_INVALID_ARG, "%s: kv_seq_stride < 0", what);
    if ((int64_t)b.n_seq * b.n_q_per_seq > (int64_t)INT32_MAX)
        return fail(IDX_ERR_INVALID_ARG, "%s: more than 2^31-1 query rows", what);
    if (b.page_table) {
        if (b.page_size < 1) return fail(IDX_ERR_INVALID_ARG, "%s: page_size < 1 with a page table", what);
        if (b.page_table_stride < ((int64_t)b.max_n_kv + b.page_size - 1) / b.page_size)
            return fail(IDX_ERR_INVALID_ARG, "%s: page_table_stride < pages of max_n_kv", what);
    }
    return IDX_OK;
}

Geom make_geom(const idx_batch& b) {
    Geom g;
    g.B = b.n_seq;
    g.T = b.n_q_per_seq;
    g.n_kv = b.n_kv;
    g.kv_start = b.kv_start;
    g.kv_seq_stride = b.kv_seq_stride;
    g.q_pos = b.q_pos;
    g.max_n_kv = b.max_n_kv;
    g.page_table = b.page_table;
    g.page_table_stride = b.page_table_stride;
    g.page_size = b.page_table ? b.page_size : 0;
    g.status = status_ptr();
    return g;
}

idx_status attn_common(const char* what, const void* q, idx_dtype dtype, int32_t Hq, int32_t Hkv,
                       int32_t dk, int32_t dv, const void* k, const void* v, int64_t kv_row_stride,
                       int64_t v_row_stride, int64_t kv_rows, idx_batch batch, const int32_t* idx,
                       int64_t idx_row_stride, const int32_t* n_sel, float scale, void* out,
                       idx_dtype out_dtype, void* ws, size_t ws_bytes, cudaStream_t st) {
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (!valid_dtype(dtype)) return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (out_dtype != IDX_F32 && out_dtype != IDX_BF16)
        return fail(IDX_ERR_INVALID_ARG, "%s: out_dtype must be F32 or BF16", what);
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
        return fail(IDX_ERR_INVALID_ARG, "%s: need Hq, Hkv >= 1 and Hq %% Hkv == 0", what);
    if (dk < 1 || dk > 576 || dv < 1 || dv > 512)
        return fail(IDX_ERR_INVALID_ARG, "%s: need 1 <= dk <= 576 and 1 <= dv <= 512", what);
    if (!v && (Hkv != 1 || dv > dk))
        return fail(IDX_ERR_INVALID_ARG, "%s: latent form (v == NULL) needs Hkv == 1, dv <= dk", what);
    if (kv_row_stride < (int64_t)Hkv * dk)
        return fail(IDX_ERR_INVALID_ARG, "%s: kv_row_stride < Hkv*dk", what);
    if (v && v_row_stride < (int64_t)Hkv * dv)
        return fail(IDX_ERR_INVALID_ARG, "%s: v_row_stride < Hkv*dv", what);
    if (kv_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: kv_rows < 0", what);
    if (idx_row_stride < 1) return fail(IDX_ERR_INVALID_ARG, "%s: idx_row_stride < 1", what);
    if (!std::isfinite(scale)) return fail(IDX_ERR_INVALID_ARG, "%s: scale not finite", what);
    if (rows == 0) return IDX_OK;
    if (!q || !k || !idx || !n_sel || !out)
        return fail(IDX_ERR_INVALID_ARG, "%s: NULL q/k/idx/n_sel/out", what);
    const Geom g = make_geom(batch);
    if (mla_tc_supported(dtype, Hq, Hkv, dk, dv, k, v, kv_row_stride, kv_rows, q, out)) {
        const size_t need = mla_workspace_bytes(rows, idx_row_stride);
        if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
            return fail(IDX_ERR_INVALID_ARG,
                        "%s: needs a 16-byte aligned workspace of %zu bytes (idx_workspace_size)", what, need);
        return from_cuda(launch_attn_mla_tc(q, k, kv_row_stride, kv_rows, g, idx, idx_row_stride, n_sel, scale,
                                            out, out_dtype, ws, ws_bytes, st),
                         what);
    }
    if (gqa_tc_supported(dtype, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, q)) {
        const cudaError_t e = launch_attn_gqa_tc(q, dtype, Hq, Hkv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                                                 idx_row_stride, n_sel, scale, out, out_dtype, ws,
                                                 ws ? ws_bytes : 0, st);
        if (e != cudaErrorNotSupported) return from_cuda(e, what);
    }
    return from_cuda(launch_attn_generic(q, dtype, Hq, Hkv, dk, dv, k, v, kv_row_stride,
                                         v_row_stride, kv_rows, g, idx, idx_row_stride, n_sel,
                                         scale, out, out_dtype, ws, ws_bytes, st),
                     what);
}

}  // namespace

// for entry points defined in other files: record the calling thread's message
idx_status record_error(idx_status s, const char* msg) { return fail(s, "%s", msg); }

// for entry points defined in other files: the kernels' view of a validated batch
Geom geom_of(const idx_batch& b) { return make_geom(b); }

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace lidx

using namespace lidx;

extern "C" {

idx_status idx_hadamard(const void* x, void* y, idx_dtype dtype, int64_t n_rows, int32_t d,
                        int64_t row_stride, idx_stream_t stream) {
    const char* what = "idx_hadamard";
    if (!valid_dtype(dtype)) return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (n_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: n_rows < 0", what);
    if (d != 32 && d != 64 && d != 128 && d != 256)
        return fail(IDX_ERR_INVALID_ARG, "%s: d must be 32, 64, 128 or 256", what);
    if (row_stride < d) return fail(IDX_ERR_INVALID_ARG, "%s: row_stride < d", what);
    if (n_rows == 0) return IDX_OK;
    if (!x || !y) return fail(IDX_ERR_INVALID_ARG, "%s: x or y is NULL", what);
    if (!aligned16(x) || !aligned16(y) || (row_stride * (int64_t)dtype_size(dtype)) % 16 != 0)
        return fail(IDX_ERR_INVALID_ARG, "%s: x, y and rows must be 16-byte aligned", what);
    return from_cuda(launch_hadamard(x, y, dtype, n_rows, d, row_stride, (cudaStream_t)stream), what);
}

idx_status idx_score(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads,
                     int32_t head_dim, const void* k, idx_dtype k_dtype, int64_t k_row_stride,
                     int64_t k_rows, idx_batch batch, int32_t block_size, float* scores,
                     int64_t score_row_stride, void* workspace, size_t workspace_bytes,
                     idx_stream_t stream) {
    const char* what = "idx_score";
    (void)workspace;
    (void)workspace_bytes;
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    if (!valid_dtype(q_dtype) || !valid_dtype(k_dtype))
        return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (n_heads < 1 || n_heads > 64)
        return fail(IDX_ERR_UNSUPPORTED, "%s: n_heads must be in [1, 64]", what);
    if (head_dim < 1 || head_dim > 256)
        return fail(IDX_ERR_UNSUPPORTED, "%s: head_dim must be in [1, 256]", what);
    if (block_size < 0) return fail(IDX_ERR_INVALID_ARG, "%s: block_size < 0", what);
    if (block_size > 1 && batch.page_table)
        return fail(IDX_ERR_UNSUPPORTED, "%s: pooled block keys are addressed without a page table", what);
    if (k_row_stride < head_dim) return fail(IDX_ERR_INVALID_ARG, "%s: k_row_stride < head_dim", what);
    if (k_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: k_rows < 0", what);
    const int32_t max_keys = block_size > 1 ? batch.max_n_kv / block_size : batch.max_n_kv;
    if (score_row_stride < max_keys)
        return fail(IDX_ERR_INVALID_ARG, "%s: score_row_stride < keys per row", what);
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (rows == 0 || max_keys == 0) return IDX_OK;
    if (!q || !w || !k || !scores) return fail(IDX_ERR_INVALID_ARG, "%s: NULL q/w/k/scores", what);
    const Geom g = make_geom(batch);
    const cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaErrorNotSupported;
    // tensor cores when q converts exactly to the key type (same type, or bf16 q with F16
    // keys: bf16's 8-bit significand fits f16's 11 bits inside f16's normal range)
    const bool q_exact = q_dtype == k_dtype || (q_dtype == IDX_BF16 && k_dtype == IDX_F16);
    if (n_heads == 64 && head_dim == 128 && k_dtype != IDX_F32 && block_size <= 1 && q_exact)
        e = launch_score_tc(q, q_dtype, w, n_heads, head_dim, k, k_dtype, k_row_stride, k_rows, g,
                            block_size, scores, score_row_stride, st);
    if (e == cudaErrorNotSupported)
        e = launch_score_generic(q, q_dtype, w, n_heads, head_dim, k, k_dtype, k_row_stride, k_rows,
                                 g, block_size, scores, score_row_stride, st);
    return from_cuda(e, what);
}

idx_status idx_quantize_rows(const void* x, idx_dtype x_dtype, int64_t n_rows, int32_t d, int64_t x_row_stride,
                             int8_t* q8, int64_t q8_row_stride, float* scale, idx_stream_t stream) {
    const char* what = "idx_quantize_rows";
    if (!valid_dtype(x_dtype)) return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (n_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: n_rows < 0", what);
    if (d < 1 || d > 1024) return fail(IDX_ERR_INVALID_ARG, "%s: d must be in [1, 1024]", what);
    if (x_row_stride < d || q8_row_stride < d) return fail(IDX_ERR_INVALID_ARG, "%s: row stride < d", what);
    if (n_rows == 0) return IDX_OK;
    if (!x || !q8) return fail(IDX_ERR_INVALID_ARG, "%s: NULL x/q8", what);
    if (!aligned16(q8) || q8_row_stride % 16 != 0)
        return fail(IDX_ERR_INVALID_ARG, "%s: q8 / q8_row_stride not 16-byte aligned", what);
    if (!scale && (d % 4 != 0 || q8_row_stride < d + 4))
        return fail(IDX_ERR_INVALID_ARG, "%s: inline scales need d %% 4 == 0 and q8_row_stride >= d + 4", what);
    return from_cuda(launch_quantize_rows(x, x_dtype, n_rows, d, x_row_stride, q8, q8_row_stride, scale,
                                          (cudaStream_t)stream),
                     what);
}

idx_status idx_score_q8(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                        const int8_t* k8, int64_t k_row_stride, const float* k_scale, int64_t k_rows,
                        idx_batch batch, int32_t block_size, float* scores, int64_t score_row_stride,
                        void* workspace, size_t workspace_bytes, idx_stream_t stream) {
    const char* what = "idx_score_q8";
    (void)workspace;
    (void)workspace_bytes;
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    if (!valid_dtype(q_dtype)) return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (n_heads < 1 || n_heads > 64)
        return fail(IDX_ERR_UNSUPPORTED, "%s: n_heads must be in [1, 64]", what);
    if (head_dim < 1 || head_dim > 256)
        return fail(IDX_ERR_UNSUPPORTED, "%s: head_dim must be in [1, 256]", what);
    if (block_size < 0 || block_size > 1)
        return fail(IDX_ERR_UNSUPPORTED, "%s: token keys only (block_size 0 or 1)", what);
    if (k_row_stride < head_dim) return fail(IDX_ERR_INVALID_ARG, "%s: k_row_stride < head_dim", what);
    if (k_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: k_rows < 0", what);
    if (score_row_stride < batch.max_n_kv)
        return fail(IDX_ERR_INVALID_ARG, "%s: score_row_stride < keys per row", what);
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (rows == 0 || batch.max_n_kv == 0) return IDX_OK;
    if (!q || !w || !k8 || !scores) return fail(IDX_ERR_INVALID_ARG, "%s: NULL q/w/k8/scores", what);
    if (!k_scale && (head_dim % 4 != 0 || k_row_stride < head_dim + 4 || k_row_stride % 4 != 0))
        return fail(IDX_ERR_INVALID_ARG, "%s: inline scales need head_dim %% 4 == 0 and a row stride >= head_dim + 4",
                    what);
    const Geom g = make_geom(batch);
    const cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaErrorNotSupported;
    if (n_heads == 64 && head_dim == 128)
        e = launch_score_tc_q8(q, q_dtype, w, k8, k_row_stride, k_scale, k_rows, g, scores, score_row_stride, st);
    if (e == cudaErrorNotSupported)
        e = launch_score_generic(q, q_dtype, w, n_heads, head_dim, k8, IDX_I8_ROWSCALE, k_row_stride, k_rows, g, 0,
                                 scores, score_row_stride, st, k_scale);
    return from_cuda(e, what);
}

static idx_status block_pool_common(const char* what, const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride,
                                    int64_t k_rows, idx_batch batch, const int32_t* n_pooled,
                                    const int32_t* stale_pos, int32_t block_size, int32_t head_dim, float* pooled,
                                    int64_t pool_seq_stride, idx_stream_t stream) {
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    if (!valid_dtype(k_dtype)) return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (block_size < 1) return fail(IDX_ERR_INVALID_ARG, "%s: block_size < 1", what);
    const int64_t row_bytes = (int64_t)head_dim * dtype_size(k_dtype);
    if (head_dim < 1 || row_bytes % 16 != 0 || row_bytes > 2048)
        return fail(IDX_ERR_UNSUPPORTED, "%s: head_dim*size must be a multiple of 16 bytes, <= 2048", what);
    if (k_row_stride < head_dim || (k_row_stride * (int64_t)dtype_size(k_dtype)) % 16 != 0)
        return fail(IDX_ERR_INVALID_ARG, "%s: k_row_stride < head_dim or not 16-byte aligned", what);
    if (pool_seq_stride < batch.max_n_kv / block_size)
        return fail(IDX_ERR_INVALID_ARG, "%s: pool_seq_stride < max_n_kv / block_size", what);
    if (k_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: k_rows < 0", what);
    if (batch.n_seq == 0 || batch.max_n_kv / block_size == 0) return IDX_OK;
    if (!k_raw || !pooled) return fail(IDX_ERR_INVALID_ARG, "%s: NULL k_raw/pooled", what);
    if (!aligned16(k_raw)) return fail(IDX_ERR_INVALID_ARG, "%s: k_raw not 16-byte aligned", what);
    const Geom g = make_geom(batch);
    return from_cuda(launch_block_pool(k_raw, k_dtype, k_row_stride, k_rows, g, block_size, head_dim, pooled,
                                       pool_seq_stride, n_pooled, stale_pos, (cudaStream_t)stream),
                     what);
}

idx_status idx_block_pool(const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride,
                          int64_t k_rows, idx_batch batch, int32_t block_size, int32_t head_dim,
                          float* pooled, int64_t pool_seq_stride, idx_stream_t stream) {
    return block_pool_common("idx_block_pool", k_raw, k_dtype, k_row_stride, k_rows, batch, nullptr, nullptr,
                             block_size, head_dim, pooled, pool_seq_stride, stream);
}

idx_status idx_block_pool_update(const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride,
                                 int64_t k_rows, idx_batch batch, const int32_t* n_pooled,
                                 const int32_t* stale_pos, int32_t block_size, int32_t head_dim,
                                 float* pooled, int64_t pool_seq_stride, idx_stream_t stream) {
    return block_pool_common("idx_block_pool_update", k_raw, k_dtype, k_row_stride, k_rows, batch, n_pooled,
                             stale_pos, block_size, head_dim, pooled, pool_seq_stride, stream);
}

idx_status idx_topk(const float* scores, int64_t score_row_stride, idx_batch batch, int32_t top_k,
                    int32_t block_size, int32_t* idx, int64_t idx_row_stride, int32_t* n_sel,
                    void* workspace, size_t workspace_bytes, idx_stream_t stream) {
    const char* what = "idx_topk";
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    if (top_k == -1) top_k = IDX_DEFAULT_TOP_K;   // the model's configured indexer top_k
    if (top_k < 1) return fail(IDX_ERR_INVALID_ARG, "%s: top_k < 1 (or -1 for the default)", what);
    if (block_size < 0) return fail(IDX_ERR_INVALID_ARG, "%s: block_size < 0", what);
    const bool blocks = block_size > 1;
    const int64_t cap = blocks ? (int64_t)(top_k / block_size) * block_size + block_size - 1 : top_k;
    if (idx_row_stride < cap)
        return fail(IDX_ERR_INVALID_ARG, "%s: idx_row_stride < output capacity %lld", what,
                    (long long)cap);
    const int32_t max_keys = blocks ? batch.max_n_kv / block_size : batch.max_n_kv;
    if (score_row_stride < max_keys)
        return fail(IDX_ERR_INVALID_ARG, "%s: score_row_stride < candidates per row", what);
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (rows == 0) return IDX_OK;
    if (!idx || (!scores && max_keys > 0)) return fail(IDX_ERR_INVALID_ARG, "%s: NULL scores/idx", what);
    const Geom g = make_geom(batch);
    if (workspace && !aligned16(workspace))
        return fail(IDX_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", what);
    return from_cuda(launch_topk(scores, score_row_stride, g, top_k, block_size, idx, idx_row_stride,
                                 n_sel, workspace, workspace ? workspace_bytes : 0, (cudaStream_t)stream),
                     what);
}

idx_status idx_block_score_topk(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                                const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride, int64_t k_rows,
                                idx_batch batch, const int32_t* n_pooled, const int32_t* stale_pos,
                                int32_t block_size, float* pooled, int64_t pool_seq_stride, int32_t top_k,
                                float* scores, int64_t score_row_stride, int32_t* idx, int64_t idx_row_stride,
                                int32_t* n_sel, idx_stream_t stream) {
    const char* what = "idx_block_score_topk";
    if (top_k == -1) top_k = IDX_DEFAULT_TOP_K;   // the model's configured indexer top_k
    // the pooled keys are addressed by pool_seq_stride alone (as idx_score addresses them)
    idx_batch pb = batch;
    pb.kv_start = nullptr;
    pb.kv_seq_stride = pool_seq_stride;
    pb.page_table = nullptr;
    pb.page_table_stride = 0;
    pb.page_size = 0;
    // one launch when every argument is valid for the three calls and the shape fits it
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    const int64_t row_bytes = (int64_t)head_dim * (valid_dtype(k_dtype) ? dtype_size(k_dtype) : 0);
    const bool ok = check_batch(batch, what) == IDX_OK && valid_dtype(q_dtype) && valid_dtype(k_dtype) &&
                    top_k >= 1 && block_size > 1 && n_heads >= 1 && n_heads <= 64 && head_dim >= 1 &&
                    head_dim <= 256 && row_bytes % 16 == 0 && row_bytes <= 2048 && k_row_stride >= head_dim &&
                    (k_row_stride * (int64_t)dtype_size(k_dtype)) % 16 == 0 && k_rows >= 0 &&
                    pool_seq_stride >= batch.max_n_kv / block_size &&
                    score_row_stride >= batch.max_n_kv / block_size &&
                    idx_row_stride >= (int64_t)(top_k / block_size) * block_size + block_size - 1 && rows > 0 &&
                    q && w && k_raw && aligned16(k_raw) && pooled && scores && idx;
    if (ok) {
        cudaError_t e = launch_block_score_topk(q, q_dtype, w, n_heads, head_dim, k_raw, k_dtype, k_row_stride, k_rows,
                                                make_geom(batch), block_size, n_pooled, stale_pos, pooled,
                                                pool_seq_stride, top_k, scores, score_row_stride, idx, idx_row_stride,
                                                n_sel, (cudaStream_t)stream);
        if (e != cudaErrorNotSupported) return from_cuda(e, what);
    }
    // otherwise the three calls, with the same results (and their argument errors)
    idx_status s = idx_block_pool_update(k_raw, k_dtype, k_row_stride, k_rows, batch, n_pooled, stale_pos, block_size,
                                         head_dim, pooled, pool_seq_stride, stream);
    if (s != IDX_OK) return s;
    s = idx_score(q, q_dtype, w, n_heads, head_dim, pooled, IDX_F32, head_dim,
                  (int64_t)batch.n_seq * pool_seq_stride, pb, block_size, scores, score_row_stride, nullptr, 0, stream);
    if (s != IDX_OK) return s;
    return idx_topk(scores, score_row_stride, batch, top_k, block_size, idx, idx_row_stride, n_sel, nullptr, 0,
                    stream);
}

idx_status idx_score_topk(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                          const void* k, idx_dtype k_dtype, int64_t k_row_stride, int64_t k_rows, idx_batch batch,
                          int32_t top_k, float* scores, int64_t score_row_stride, int32_t* idx,
                          int64_t idx_row_stride, int32_t* n_sel, void* workspace, size_t workspace_bytes,
                          idx_stream_t stream) {
    const char* what = "idx_score_topk";
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    if (top_k == -1) top_k = IDX_DEFAULT_TOP_K;   // the model's configured indexer top_k
    if (top_k < 1) return fail(IDX_ERR_INVALID_ARG, "%s: top_k < 1 (or -1 for the default)", what);
    if (!valid_dtype(q_dtype) || !valid_dtype(k_dtype)) return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (n_heads < 1 || n_heads > 64) return fail(IDX_ERR_UNSUPPORTED, "%s: n_heads must be in [1, 64]", what);
    if (head_dim < 1 || head_dim > 256) return fail(IDX_ERR_UNSUPPORTED, "%s: head_dim must be in [1, 256]", what);
    if (k_row_stride < head_dim) return fail(IDX_ERR_INVALID_ARG, "%s: k_row_stride < head_dim", what);
    if (k_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: k_rows < 0", what);
    if (score_row_stride < batch.max_n_kv)
        return fail(IDX_ERR_INVALID_ARG, "%s: score_row_stride < keys per row", what);
    if (idx_row_stride < top_k) return fail(IDX_ERR_INVALID_ARG, "%s: idx_row_stride < top_k", what);
    if (workspace && !aligned16(workspace))
        return fail(IDX_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", what);
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (rows == 0) return IDX_OK;
    if (!q || !w || !k || !scores || !idx) return fail(IDX_ERR_INVALID_ARG, "%s: NULL q/w/k/scores/idx", what);
    const cudaStream_t st = (cudaStream_t)stream;
    // fused: decode rows on the tensor-core scorer, few enough for the multi-CTA select
    const bool q_exact = q_dtype == k_dtype || (q_dtype == IDX_BF16 && k_dtype == IDX_F16);
    if (n_heads == 64 && head_dim == 128 && k_dtype != IDX_F32 && q_exact && batch.n_q_per_seq == 1 &&
        batch.max_n_kv > 0 && rows < 2 * (int64_t)sm_count() && rows <= 1024 && workspace &&
        workspace_bytes >= topk_fused_workspace_bytes(rows)) {
        const Geom g = make_geom(batch);
        const FusedArrays fa = topk_fused_arrays(workspace, rows);
        cudaError_t e = launch_score_tc(q, q_dtype, w, n_heads, head_dim, k, k_dtype, k_row_stride, k_rows, g, 0,
                                        scores, score_row_stride, st, fa.hist, fa.cnt);
        if (e == cudaSuccess)
            return from_cuda(launch_topk_fused(scores, score_row_stride, g, top_k, idx, idx_row_stride, n_sel,
                                               workspace, st),
                             what);
        if (e != cudaErrorNotSupported) return from_cuda(e, what);
    }
    // otherwise the two calls, with the same results
    s = idx_score(q, q_dtype, w, n_heads, head_dim, k, k_dtype, k_row_stride, k_rows, batch, 0, scores,
                  score_row_stride, nullptr, 0, stream);
    if (s != IDX_OK) return s;
    return idx_topk(scores, score_row_stride, batch, top_k, 0, idx, idx_row_stride, n_sel, workspace,
                    workspace_bytes, stream);
}

idx_status sparse_attn_decode(const void* q, idx_dtype dtype, int32_t n_q_heads, int32_t n_kv_heads,
                              int32_t dk, int32_t dv, const void* k, const void* v,
                              int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows,
                              idx_batch batch, const int32_t* idx, int64_t idx_row_stride,
                              const int32_t* n_sel, float scale, void* out, idx_dtype out_dtype,
                              void* workspace, size_t workspace_bytes, idx_stream_t stream) {
    return attn_common("sparse_attn_decode", q, dtype, n_q_heads, n_kv_heads, dk, dv, k, v,
                       kv_row_stride, v_row_stride, kv_rows, batch, idx, idx_row_stride, n_sel,
                       scale, out, out_dtype, workspace, workspace_bytes, (cudaStream_t)stream);
}

idx_status sparse_attn_prefill(const void* q, idx_dtype dtype, int32_t n_q_heads, int32_t n_kv_heads,
                               int32_t dk, int32_t dv, const void* k, const void* v,
                               int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows,
                               idx_batch batch, const int32_t* idx, int64_t idx_row_stride,
                               const int32_t* n_sel, float scale, void* out, idx_dtype out_dtype,
                               void* workspace, size_t workspace_bytes, idx_stream_t stream) {
    return attn_common("sparse_attn_prefill", q, dtype, n_q_heads, n_kv_heads, dk, dv, k, v,
                       kv_row_stride, v_row_stride, kv_rows, batch, idx, idx_row_stride, n_sel,
                       scale, out, out_dtype, workspace, workspace_bytes, (cudaStream_t)stream);
}

idx_status sparse_decode_step(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                              const void* k, idx_dtype k_dtype, int64_t k_row_stride, int64_t k_rows,
                              idx_batch batch, int32_t top_k, float* scores, int64_t score_row_stride, int32_t* idx,
                              int64_t idx_row_stride, int32_t* n_sel, const void* q_attn, idx_dtype attn_dtype,
                              int32_t n_q_heads, int32_t n_kv_heads, int32_t dk, int32_t dv, const void* k_attn,
                              const void* v_attn, int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows,
                              float scale, void* out, idx_dtype out_dtype, void* workspace, size_t workspace_bytes,
                              idx_stream_t stream) {
    const char* what = "sparse_decode_step";
    idx_status s = check_batch(batch, what);
    if (s != IDX_OK) return s;
    if (top_k == -1) top_k = IDX_DEFAULT_TOP_K;
    if (top_k < 1) return fail(IDX_ERR_INVALID_ARG, "%s: top_k < 1 (or -1 for the default)", what);
    if (!valid_dtype(q_dtype) || !valid_dtype(k_dtype) || !valid_dtype(attn_dtype))
        return fail(IDX_ERR_INVALID_ARG, "%s: bad dtype", what);
    if (out_dtype != IDX_F32 && out_dtype != IDX_BF16)
        return fail(IDX_ERR_INVALID_ARG, "%s: out_dtype must be F32 or BF16", what);
    if (n_heads < 1 || n_heads > 64) return fail(IDX_ERR_UNSUPPORTED, "%s: n_heads must be in [1, 64]", what);
    if (head_dim < 1 || head_dim > 256) return fail(IDX_ERR_UNSUPPORTED, "%s: head_dim must be in [1, 256]", what);
    if (k_row_stride < head_dim) return fail(IDX_ERR_INVALID_ARG, "%s: k_row_stride < head_dim", what);
    if (k_rows < 0 || kv_rows < 0) return fail(IDX_ERR_INVALID_ARG, "%s: k_rows or kv_rows < 0", what);
    if (score_row_stride < batch.max_n_kv)
        return fail(IDX_ERR_INVALID_ARG, "%s: score_row_stride < keys per row", what);
    if (idx_row_stride < top_k) return fail(IDX_ERR_INVALID_ARG, "%s: idx_row_stride < top_k", what);
    if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads != 0)
        return fail(IDX_ERR_INVALID_ARG, "%s: need Hq, Hkv >= 1 and Hq %% Hkv == 0", what);
    if (dk < 1 || dk > 576 || dv < 1 || dv > 512)
        return fail(IDX_ERR_INVALID_ARG, "%s: need 1 <= dk <= 576 and 1 <= dv <= 512", what);
    if (!v_attn && (n_kv_heads != 1 || dv > dk))
        return fail(IDX_ERR_INVALID_ARG, "%s: latent form (v == NULL) needs Hkv == 1, dv <= dk", what);
    if (kv_row_stride < (int64_t)n_kv_heads * dk) return fail(IDX_ERR_INVALID_ARG, "%s: kv_row_stride < Hkv*dk", what);
    if (v_attn && v_row_stride < (int64_t)n_kv_heads * dv)
        return fail(IDX_ERR_INVALID_ARG, "%s: v_row_stride < Hkv*dv", what);
    if (!std::isfinite(scale)) return fail(IDX_ERR_INVALID_ARG, "%s: scale not finite", what);
    if (workspace && !aligned16(workspace))
        return fail(IDX_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", what);
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (rows == 0) return IDX_OK;
    if (!q || !w || !k || !scores || !idx || !n_sel || !q_attn || !k_attn || !out)
        return fail(IDX_ERR_INVALID_ARG, "%s: NULL q/w/k/scores/idx/n_sel/q_attn/k_attn/out", what);
    const cudaStream_t st = (cudaStream_t)stream;
    // one launch for few short decode rows with the 128-head MLA attention
    const bool q_exact = q_dtype == k_dtype || (q_dtype == IDX_BF16 && k_dtype == IDX_F16);
    if (n_heads == 64 && head_dim == 128 && k_dtype != IDX_F32 && q_exact && batch.n_q_per_seq == 1 &&
        aligned16(q) && aligned16(k) && (k_row_stride * 2) % 16 == 0 && batch.max_n_kv > 0 &&
        mla_tc_supported(attn_dtype, n_q_heads, n_kv_heads, dk, dv, k_attn, v_attn, kv_row_stride, kv_rows, q_attn,
                         out) &&
        fused_decode_fits(rows, batch.max_n_kv, top_k, idx_row_stride)) {
        const size_t need = fused_decode_workspace_bytes(rows, idx_row_stride);
        if (workspace && workspace_bytes >= need) {
            const Geom g = make_geom(batch);
            const cudaError_t e = launch_decode_fused(q, q_dtype, w, k, k_dtype, k_row_stride, k_rows, g, top_k, scores,
                                                      score_row_stride, idx, idx_row_stride, n_sel, k_attn,
                                                      kv_row_stride, kv_rows, q_attn, scale, out, out_dtype, workspace,
                                                      workspace_bytes, st);
            if (e == cudaSuccess) return IDX_OK;
            // a grid the device cannot hold at once (or a shape the launch declines) runs unfused
            if (e != cudaErrorNotSupported && e != cudaErrorCooperativeLaunchTooLarge)
                return from_cuda(e, what);
            cudaGetLastError();
        }
    }
    // otherwise the two calls, with the same results
    s = idx_score_topk(q, q_dtype, w, n_heads, head_dim, k, k_dtype, k_row_stride, k_rows, batch, top_k, scores,
                       score_row_stride, idx, idx_row_stride, n_sel, workspace, workspace_bytes, stream);
    if (s != IDX_OK) return s;
    return sparse_attn_decode(q_attn, attn_dtype, n_q_heads, n_kv_heads, dk, dv, k_attn, v_attn, kv_row_stride,
                              v_row_stride, kv_rows, batch, idx, idx_row_stride, n_sel, scale, out, out_dtype,
                              workspace, workspace_bytes, stream);
}

int32_t sparse_decode_step_fused(int64_t n_rows, int32_t n_q_per_seq, int32_t max_n_kv, int32_t top_k,
                                 int64_t idx_row_stride) {
    if (top_k == -1) top_k = IDX_DEFAULT_TOP_K;
    return n_q_per_seq == 1 && max_n_kv > 0 && top_k >= 1 && idx_row_stride >= top_k &&
                   fused_decode_fits(n_rows, max_n_kv, top_k, idx_row_stride)
               ? 1
               : 0;
}

size_t idx_workspace_size(int32_t op, int64_t n_rows, int32_t max_n_kv, int32_t top_k,
                          int32_t n_q_heads, int32_t dv) {
    (void)max_n_kv;
    if (top_k == -1) top_k = IDX_DEFAULT_TOP_K;
    if (n_rows <= 0 || top_k <= 0) return 0;
    if (op == IDX_OP_ATTN_DECODE || op == IDX_OP_ATTN_PREFILL) {
        // 128 heads x 512: the tensor-core MLA path's split partials (if such a call runs on the CUDA
        // cores instead, it uses as many key splits as this fits); otherwise the CUDA-core path's
        if (n_q_heads == 128 && dv == 512) return mla_workspace_bytes(n_rows, top_k);
        return generic_attn_workspace_bytes(n_rows, top_k, n_q_heads, dv);
    }
    if (op == IDX_OP_TOPK) return topk_workspace_bytes(n_rows, top_k);
    if (op == IDX_OP_DECODE_STEP) {
        // the larger of the two calls' (they run one after the other on the same buffer); the
        // fused launch needs the attention's split partials only
        const size_t a = idx_workspace_size(IDX_OP_SCORE_TOPK, n_rows, max_n_kv, top_k, 0, 0);
        const size_t b = idx_workspace_size(IDX_OP_ATTN_DECODE, n_rows, max_n_kv, top_k, n_q_heads, dv);
        const size_t c = n_q_heads == 128 && dv == 512 && n_rows <= 32 ? fused_decode_workspace_bytes(n_rows, top_k) : 0;
        return a > b ? (a > c ? a : c) : (b > c ? b : c);
    }
    if (op == IDX_OP_SCORE_TOPK) {
        int sms = sm_count();
        if (sms < 2) sms = 152;
        return n_rows < 2 * (int64_t)sms ? topk_fused_workspace_bytes(n_rows) : topk_workspace_bytes(n_rows, top_k);
    }
    return 0;
}

const char* idx_last_error(void) { return t_last_error.c_str(); }

idx_status idx_device_status(int32_t reset) {
    int* p = status_ptr();
    if (!p) return fail(IDX_ERR_CUDA, "idx_device_status: no device status word");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "idx_device_status: %s", cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && reset) e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) return fail(IDX_ERR_CUDA, "idx_device_status: %s", cudaGetErrorString(e));
    if (v != 0) fail((idx_status)v, "a kernel recorded device fault code %d", v);
    return (idx_status)v;
}

}  // extern "C"
