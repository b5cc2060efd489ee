// Internal declarations shared by the kernels and the C-ABI layer of liblidx.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "lidx.h"

namespace lidx {

// ---------------------------------------------------------------------------
// batch geometry as the kernels see it (a by-value copy of idx_batch plus the
// device status word every kernel reports data-dependent faults to)
// ---------------------------------------------------------------------------
struct Geom {
    int32_t B;
    int32_t T;
    const int32_t* n_kv;
    const int32_t* kv_start;
    int64_t kv_seq_stride;
    const int32_t* q_pos;
    int32_t max_n_kv;
    const int32_t* page_table;   // paged caches (NULL: kv_start / kv_seq_stride)
    int64_t page_table_stride;
    int32_t page_size;
    int* status;  // device int: first fault code recorded, 0 = none
};

// Programmatic dependent launch along the decode chain (scorer -> top-k ->
// attention -> next step's scorer).  Each kernel of the chain lets the next
// one launch as soon as all of its CTAs have started (pdl_trigger), and every
// CTA waits for the previous grid to complete, its writes visible
// (pdl_wait), before it reads or writes anything another kernel produces or
// consumes.  Completion therefore stays transitive along the chain; only
// launch latency and work on pure inputs overlap.  Launched without the
// attribute, both instructions are no-ops.
// A chained kernel's pointers to what its predecessor writes (scores,
// histograms, selections, split partials) carry no __restrict__: a restricted
// read-only pointer lets the compiler treat the data as invariant for the
// whole kernel, so its loads may move above pdl_wait or take the
// non-coherent read-only path, and would then see the predecessor's data
// before it is written.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void flag(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// cached tokens of sequence b, clamped to [0, max_n_kv] (a violation is flagged)
__device__ __forceinline__ int seq_n_kv(const Geom& g, int b) {
    int n = g.n_kv[b];
    if (n < 0 || n > g.max_n_kv) {
        flag(g.status, IDX_ERR_DEVICE_BOUNDS);
        n = n < 0 ? 0 : g.max_n_kv;
    }
    return n;
}

// keys visible to query row r: min(q_pos + 1, n_kv) under the causal mask, else n_kv
__device__ __forceinline__ int row_n_vis(const Geom& g, int64_t r) {
    int b = (int)(r / g.T);
    int n = seq_n_kv(g, b);
    if (g.q_pos) {
        int p = g.q_pos[r];
        int lim = p < 0 ? 0 : (p >= n ? n : p + 1);
        n = lim;
    }
    return n;
}

// cache row of position 0 of sequence b (contiguous caches)
__device__ __forceinline__ int64_t seq_row0(const Geom& g, int b) {
    return g.kv_start ? (int64_t)g.kv_start[b] : (int64_t)b * g.kv_seq_stride;
}

// cache row of position j of sequence b: through the page table when there is
// one; a negative page index gives a negative row, which callers reject
__device__ __forceinline__ int64_t key_row(const Geom& g, int b, int64_t j) {
    if (g.page_table) {
        const int64_t pg = j / g.page_size;
        const int32_t phys = g.page_table[(int64_t)b * g.page_table_stride + pg];
        return (int64_t)phys * g.page_size + (j - pg * g.page_size);
    }
    return seq_row0(g, b) + j;
}

// ---------------------------------------------------------------------------
// element conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(int8_t x) { return (float)x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float load_any(const void* p, int64_t i, int dtype) {
    switch (dtype) {
        case IDX_F16: return __half2float(static_cast<const __half*>(p)[i]);
        case IDX_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
        default: return static_cast<const float*>(p)[i];
    }
}

// order-preserving map of an f32 score to uint32 (larger score -> larger key);
// -0 is folded onto +0 first so that equal scores have equal keys
__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

inline size_t dtype_size(int t) { return t == IDX_F32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// launchers (one per kernel family); each returns cudaGetLastError()
// ---------------------------------------------------------------------------
cudaError_t launch_hadamard(const void* x, void* y, int dtype, int64_t n_rows, int d,
                            int64_t row_stride, cudaStream_t st);

// k_dtype IDX_I8_ROWSCALE: int8 key rows with per-row f32 scales k_scale
constexpr int IDX_I8_ROWSCALE = 100;
cudaError_t launch_score_generic(const void* q, int q_dtype, const float* w, int H, int d,
                                 const void* k, int k_dtype, int64_t k_row_stride, int64_t k_rows,
                                 const Geom& g, int block_size, float* scores,
                                 int64_t score_row_stride, cudaStream_t st, const float* k_scale = nullptr);

cudaError_t launch_quantize_rows(const void* x, int x_dtype, int64_t n_rows, int d, int64_t x_row_stride,
                                 int8_t* q8, int64_t q8_row_stride, float* scale, cudaStream_t st);

// tensor-core scorer for H = 64, d = 128, 16-bit keys; returns cudaErrorNotSupported
// when the shape is not one it handles (the caller then uses the generic scorer)
// hist (decode rows only, T = 1, at most 1024 rows): also count each row's scores into
// hist[row][2048] by the top 11 bits of their order key; the launch zeroes hist and cnt[rows]
cudaError_t launch_score_tc(const void* q, int q_dtype, const float* w, int H, int d,
                            const void* k, int k_dtype, int64_t k_row_stride, int64_t k_rows,
                            const Geom& g, int block_size, float* scores, int64_t score_row_stride,
                            cudaStream_t st, uint32_t* hist = nullptr, uint32_t* cnt = nullptr);

// tensor-core decode scorer over int8 keys with per-row scales (H = 64, d = 128,
// T = 1, 16-bit q); k_scale NULL: each row's f32 scale sits in its bytes 128..131
// (row stride >= 144); cudaErrorNotSupported for anything else
cudaError_t launch_score_tc_q8(const void* q, int q_dtype, const float* w, const int8_t* k8, int64_t k_row_stride,
                               const float* k_scale, int64_t k_rows, const Geom& g, float* scores,
                               int64_t score_row_stride, cudaStream_t st);

// n_pooled / stale_pos (device, may be NULL): pool only blocks from
// min(n_pooled[b], stale_pos[b] / C) on (incremental maintenance)
cudaError_t launch_block_pool(const void* k_raw, int k_dtype, int64_t k_row_stride, int64_t k_rows,
                              const Geom& g, int C, int d, float* pooled, int64_t pool_seq_stride,
                              const int32_t* n_pooled, const int32_t* stale_pos, cudaStream_t st);

// pool update + pooled-key scores + block selection in one launch (k_block_select.cu);
// cudaErrorNotSupported for shapes it does not take
cudaError_t launch_block_score_topk(const void* q, int q_dtype, const float* w, int H, int d, const void* k_raw,
                                    int k_dtype, int64_t k_row_stride, int64_t k_rows, const Geom& g, int C,
                                    const int32_t* n_pooled, const int32_t* stale_pos, float* pooled,
                                    int64_t pool_seq_stride, int top_k, float* scores, int64_t score_row_stride,
                                    int32_t* idx, int64_t idx_row_stride, int32_t* n_sel, cudaStream_t st);

// few rows with a workspace of topk_workspace_bytes(): multi-CTA passes; else one CTA per row
cudaError_t launch_topk(const float* scores, int64_t score_row_stride, const Geom& g, int top_k,
                        int block_size, int32_t* idx, int64_t idx_row_stride, int32_t* n_sel, void* ws,
                        size_t ws_bytes, cudaStream_t st);
size_t topk_workspace_bytes(int64_t n_rows, int top_k);

// fused score + top-k: the scorer counts each row's scores into the workspace's histograms (and
// zeroes the select's counters); the select reads them (filter + finish kernels)
size_t topk_fused_workspace_bytes(int64_t n_rows);
// the fused workspace's arrays the scorer writes: histograms, candidate counters
struct FusedArrays {
    uint32_t* hist;
    uint32_t* cnt;
};
FusedArrays topk_fused_arrays(void* ws, int64_t n_rows);
cudaError_t launch_topk_fused(const float* scores, int64_t score_row_stride, const Geom& g, int top_k, int32_t* idx,
                              int64_t idx_row_stride, int32_t* n_sel, void* ws, cudaStream_t st);

// CUDA-core attention (any head counts and widths); with few rows the selected keys are split
// over CTAs, and the partials need generic_attn_workspace_bytes() of the workspace (without it,
// or with less, fewer splits are used)
int generic_attn_splits(int64_t n_rows, int64_t cap);
size_t generic_attn_workspace_bytes(int64_t n_rows, int64_t cap, int Hq, int dv);
cudaError_t launch_attn_generic(const void* q, int dtype, int Hq, int Hkv, int dk, int dv,
                                const void* k, const void* v, int64_t kv_row_stride,
                                int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                                const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
                                float scale, void* out, int out_dtype, void* ws, size_t ws_bytes,
                                cudaStream_t st);

// merge of the CUDA-core layout's key-split partials ([row, split, head] x dv, then (m, l) in
// natural-log units)
cudaError_t launch_attn_generic_combine(const float* part_o, const float* part_ml, int splits, int64_t n_rows, int Hq,
                                        int dv, void* out, int out_dtype, cudaStream_t st);

// tcgen05 sparse GQA attention (16-bit K/V, dk = dv = 128, at most 16 query heads per kv head);
// splits write the CUDA-core layout's partials into ws (fewer splits when it is smaller);
// cudaErrorNotSupported when the selection needs more splits than the workspace holds
bool gqa_tc_supported(int dtype, int Hq, int Hkv, int dk, int dv, const void* k, const void* v,
                      int64_t kv_row_stride, int64_t v_row_stride, const void* q);
cudaError_t launch_attn_gqa_tc(const void* q, int dtype, int Hq, int Hkv, const void* k, const void* v,
                               int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                               const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel, float scale,
                               void* out, int out_dtype, void* ws, size_t ws_bytes, cudaStream_t st);

// tcgen05 sparse MLA attention (128 heads, 576/512 bf16 latent); the caller
// checks mla_tc_supported() first; splits > 1 needs mla_workspace_bytes()
bool mla_tc_supported(int dtype, int Hq, int Hkv, int dk, int dv, const void* k, const void* v,
                      int64_t kv_row_stride, int64_t kv_rows, const void* q, const void* out);
int mla_splits(int64_t n_rows, int64_t cap);
size_t mla_workspace_bytes(int64_t n_rows, int64_t cap);
cudaError_t launch_attn_mla_tc(const void* q, const void* lat, int64_t kv_row_stride, int64_t kv_rows,
                               const Geom& g, const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
                               float scale, void* out, int out_dtype, void* ws, size_t ws_bytes,
                               cudaStream_t st);

// fused decode step (scores + top-k + MLA attention in one cooperative launch) for few short
// decode rows: whether a batch fits, its workspace, the launch (cudaErrorNotSupported when the
// device cannot hold the grid at once)
bool fused_decode_fits(int64_t n_rows, int max_n_kv, int top_k, int64_t idx_row_stride);
size_t fused_decode_workspace_bytes(int64_t n_rows, int64_t idx_row_stride);
cudaError_t launch_decode_fused(const void* qi, int qi_dtype, const float* w, const void* k, int k_dtype,
                                int64_t k_row_stride, int64_t k_rows, const Geom& g, int top_k, float* scores,
                                int64_t score_row_stride, int32_t* idx, int64_t idx_row_stride, int32_t* n_sel,
                                const void* lat, int64_t lat_row_stride, int64_t kv_rows, const void* qa, float scale,
                                void* out, int out_dtype, void* ws, size_t ws_bytes, cudaStream_t st);

// TMA tensor maps over 16-bit caches (128-byte swizzle); false if encoding fails
bool make_key_tmap(CUtensorMap* m, const void* k, bool bf16, int64_t k_row_stride, int64_t k_rows, int box_rows);
bool make_q3d_tmap(CUtensorMap* m, const void* q, bool bf16, int64_t rows);
bool make_w_tmap(CUtensorMap* m, const float* w, int64_t rows);
// [rows, payload] int8 keys (128 codes, or 144 bytes with the scale inline): boxes of
// payload bytes x box_rows rows, unswizzled or (128-byte rows) in the 128-byte swizzle
bool make_key8_tmap(CUtensorMap* m, const int8_t* k, int64_t row_bytes, int64_t k_rows, int box_rows,
                    int payload, bool swizzle128 = false);

// number of SMs of the current device (cached per device)
int sm_count();

// launch with programmatic stream serialisation (see pdl_trigger / pdl_wait)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// set idx_last_error() for the calling thread and return s
idx_status record_error(idx_status s, const char* msg);

// kernel geometry of a batch (with the device status word of the current device)
Geom geom_of(const idx_batch& b);

}  // namespace lidx
