// sparse_attn_decode_noalloc: the 128-head MLA decode attention for callers
// that cannot allocate device memory.
//
// Who needs it: a host program that owns every byte of device memory through
// its own pool or arena (a serving engine's memory planner, a framework that
// embeds this library as a plugin) may not call cudaMalloc: an allocation
// outside its pool breaks its accounting, and cudaMalloc can block while the
// driver maps memory and can synchronise the device.  Such a caller cannot
// provide the key-split workspace sparse_attn_decode asks for when there are
// few query rows.  This entry point keeps that scratch in a fixed array that
// is part of the library itself, so the caller passes only inputs and outputs.
//
// Costs and rules:
//  - The array is kScratchBytes (20,000,768 bytes = 76 key-split units of
//    128 heads x (512 + 2) floats): enough for every split count the
//    attention chooses on a device with at most 152 SMs (a GB300) when each
//    row selects at most 2048 keys.  The split policy reads the SM count at
//    run time and uses at most SMs/2 units for such rows, so a device with
//    more SMs, or rows selecting more keys (always split, rows x splits
//    units), can need more: such calls are rejected, never truncated.
//    Every GPU that loads the library holds it until the process exits.
//  - A call whose key-split partials would not fit is rejected with
//    IDX_ERR_INVALID_ARG before anything is launched.
//  - All calls share the one array, and it keeps the contents of the last
//    call.  Nothing in it has to start at zero: every partial the merge step
//    reads is written earlier by the same call.  Calls whose work overlaps
//    on the GPU (other streams, other threads) race on the array and must be
//    serialised by the caller.
//  - The device address of the array is looked up once per device, by the
//    first call made with that device current.  Make that first call before
//    any stream capture begins.
#include <mutex>

#include "lidx_internal.cuh"

namespace lidx {
namespace {

constexpr size_t kScratchBytes = (size_t)76 * 128 * (512 + 2) * sizeof(float);

// the key-split partials (O, then m and l) of every call of this entry point
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// device address of g_attn_scratch on the current device; looked up once per device
idx_status scratch_ptr(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return record_error(IDX_ERR_CUDA, "sparse_attn_decode_noalloc: no usable current device");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress((void**)&p, g_attn_scratch);
        if (e != cudaSuccess || !p)
            return record_error(IDX_ERR_CUDA, "sparse_attn_decode_noalloc: cannot locate the static scratch array");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return IDX_OK;
}

}  // namespace
}  // namespace lidx

using namespace lidx;

extern "C" idx_status sparse_attn_decode_noalloc(const void* q, idx_dtype dtype, int32_t n_q_heads,
                                                 int32_t n_kv_heads, int32_t dk, int32_t dv, const void* k,
                                                 int64_t kv_row_stride, int64_t kv_rows, idx_batch batch,
                                                 const int32_t* idx, int64_t idx_row_stride,
                                                 const int32_t* n_sel, float scale, void* out,
                                                 idx_dtype out_dtype, idx_stream_t stream) {
    if (batch.n_seq < 0 || batch.n_q_per_seq < 1 || batch.max_n_kv < 0 || (batch.n_seq > 0 && !batch.n_kv) ||
        (!batch.kv_start && batch.kv_seq_stride < 0) ||
        (batch.page_table && (batch.page_size < 1 || batch.page_table_stride <
                                                       ((int64_t)batch.max_n_kv + batch.page_size - 1) / batch.page_size)))
        return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: invalid batch geometry");
    if (out_dtype != IDX_F32 && out_dtype != IDX_BF16)
        return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: out_dtype must be F32 or BF16");
    if (idx_row_stride < 1 || !(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
        return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: bad idx_row_stride or scale");
    const int64_t rows = (int64_t)batch.n_seq * batch.n_q_per_seq;
    if (rows > (int64_t)INT32_MAX)
        return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: too many query rows");
    if (rows == 0) return IDX_OK;
    if (!q || !k || !idx || !n_sel || !out)
        return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: NULL q/k/idx/n_sel/out");
    // the same row-stride rule as sparse_attn_decode: a latent row must not
    // overlap the next one (this also rules out zero and negative strides)
    if (n_kv_heads < 1 || dk < 1 || kv_row_stride < (int64_t)n_kv_heads * dk)
        return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: kv_row_stride < Hkv*dk");
    if (kv_rows < 0) return record_error(IDX_ERR_INVALID_ARG, "sparse_attn_decode_noalloc: kv_rows < 0");
    if (!mla_tc_supported(dtype, n_q_heads, n_kv_heads, dk, dv, k, nullptr, kv_row_stride, kv_rows, q, out))
        return record_error(IDX_ERR_UNSUPPORTED,
                            "sparse_attn_decode_noalloc: serves only bf16 MLA latent attention with 128 query "
                            "heads, dk 576, dv 512, 16-byte aligned q/k/out and kv_row_stride % 8 == 0");
    const size_t need = mla_workspace_bytes(rows, idx_row_stride);
    if (need > kScratchBytes)
        return record_error(IDX_ERR_INVALID_ARG,
                            "sparse_attn_decode_noalloc: the key-split partials of this call exceed the "
                            "20,000,768-byte static scratch array (sized for devices with at most 152 SMs "
                            "and rows selecting at most 2048 keys); use sparse_attn_decode with a workspace");
    void* scratch = nullptr;
    if (need > 0) {
        const idx_status s = scratch_ptr(&scratch);
        if (s != IDX_OK) return s;
    }
    const cudaError_t e = launch_attn_mla_tc(q, k, kv_row_stride, kv_rows, geom_of(batch), idx, idx_row_stride,
                                             n_sel, scale, out, out_dtype, scratch, kScratchBytes,
                                             (cudaStream_t)stream);
    if (e != cudaSuccess)
        return record_error(IDX_ERR_CUDA, cudaGetErrorString(e));
    return IDX_OK;
}
