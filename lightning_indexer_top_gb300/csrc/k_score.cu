// Lightning-indexer score on the CUDA cores, any head count / head size:
//     s[r, j] = sum_h w[r, h] * max(0, q[r, h, :] . k[j, :])
// (ik_llama_opt commit log, "openpangu: DSA lightning indexer + SWA schedule";
// ReLU per head before the head sum, llama.cpp commit c88c916636, QSA commit
// message).  Used for small head counts and for pooled block keys, where the
// work per key is small; H = 64 x d = 128 on 16-bit keys goes to the tensor
// core scorer instead.
//
// Grid (query rows, key tiles of 128).  The CTA stages its row's q (converted
// to f32) and w in shared memory; thread j owns key j of the tile, streams
// that key row in chunks of 8 elements and keeps one f32 accumulator per
// head in registers.  The head count is rounded up to a power of two (a
// template parameter, so the accumulators stay in registers) and the padding
// heads get q = 0, w = 0.  Pooled block keys (few per row) with 16 or more
// heads take score_split_kernel instead: four threads per key, each over a
// quarter of the heads.
#include "block_ops.cuh"

namespace lidx {
namespace {

constexpr int kTile = 128;

template <typename TK, int HH>
__global__ void __launch_bounds__(kTile) score_generic_kernel(
    const void* q, int q_dtype, const float* __restrict__ w, int H, int d,
    const TK* k, int64_t k_row_stride, int64_t k_rows, Geom g, int block_size,
    float* __restrict__ scores, int64_t score_row_stride, const float* k_scale) {
    extern __shared__ float smem[];
    pdl_trigger();
    pdl_wait();
    float* qs = smem;            // [HH][d], heads >= H zero
    float* ws = smem + HH * d;   // [HH],    heads >= H zero

    // grid.x = query rows (no 65535 limit); grid.y strides over key tiles
    const int64_t r = blockIdx.x;
    const int b = (int)(r / g.T);
    int n_keys = row_n_vis(g, r);
    if (block_size > 1) n_keys /= block_size;
    if ((int)blockIdx.y * kTile >= n_keys) return;

    for (int i = threadIdx.x; i < HH * d; i += blockDim.x)
        qs[i] = (i < H * d) ? load_any(q, r * (int64_t)H * d + i, q_dtype) : 0.f;
    for (int i = threadIdx.x; i < HH; i += blockDim.x) ws[i] = (i < H) ? w[r * H + i] : 0.f;
    __syncthreads();

    for (int j0 = blockIdx.y * kTile; j0 < n_keys; j0 += gridDim.y * kTile) {
        const int j = j0 + threadIdx.x;
        if (j >= n_keys) continue;
        const int64_t row = key_row(g, b, j);
        if (row < 0 || row >= k_rows) {
            flag(g.status, IDX_ERR_DEVICE_BOUNDS);
            continue;
        }
        const TK* kr = k + row * k_row_stride;

        float acc[HH];
#pragma unroll
        for (int h = 0; h < HH; ++h) acc[h] = 0.f;
        for (int c0 = 0; c0 < d; c0 += 8) {
            float kv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) kv[i] = (c0 + i < d) ? to_f32(kr[c0 + i]) : 0.f;
#pragma unroll
            for (int h = 0; h < HH; ++h) {
                const float* qh = qs + h * d + c0;
                float a = acc[h];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (c0 + i < d) a = fmaf(qh[i], kv[i], a);
                acc[h] = a;
            }
        }
        // quantized keys: the dot with the dequantized key is scale * (dot with the codes)
        float ks = 1.f;
        if constexpr (sizeof(TK) == 1)   // int8 codes: scale array, or inline after the row's d codes
            ks = k_scale ? k_scale[row] : *reinterpret_cast<const float*>(kr + d);
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < HH; ++h) s = fmaf(ws[h], fmaxf(ks * acc[h], 0.f), s);
        scores[r * score_row_stride + j] = s + 0.0f;  // -0 + +0 = +0
    }
}

// Few keys per row and many heads (the pooled block keys of a decode step): four threads per key,
// each summing HH/4 heads, so a row's keys spread over 4x the threads; the four partial head sums
// of a key are added by shuffles.  q sits in shared memory head-fastest ([d][HH]), so a thread
// reads its heads' values at one dimension with 16-byte loads and the four head groups of a warp
// hit different banks; key rows are read with 16-byte loads (the four threads of a key share the
// lines in L1).  Grid (query rows, tiles of 32 keys).
constexpr int kSplitKeys = 32;

template <typename TK, int HH>
__global__ void __launch_bounds__(128) score_split_kernel(
    const void* q, int q_dtype, const float* __restrict__ w, int H, int d,
    const TK* k, int64_t k_row_stride, int64_t k_rows, Geom g, int block_size,
    float* __restrict__ scores, int64_t score_row_stride, bool vec) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) float smem[];
    float* qs = smem;            // [d][HH], heads >= H zero
    float* ws = smem + HH * d;   // [HH]
    const int64_t r = blockIdx.x;
    const int b = (int)(r / g.T);
    int n_keys = row_n_vis(g, r);
    if (block_size > 1) n_keys /= block_size;
    if ((int)blockIdx.y * kSplitKeys >= n_keys) return;
    blk::load_q_split<HH>(q, q_dtype, w, H, d, r, qs, ws);
    __syncthreads();
    const int hg = threadIdx.x & 3;
    const int j = blockIdx.y * kSplitKeys + (threadIdx.x >> 2);
    bool valid = j < n_keys;
    int64_t row = 0;
    if (valid) {
        row = key_row(g, b, j);
        if (row < 0 || row >= k_rows) {
            flag(g.status, IDX_ERR_DEVICE_BOUNDS);
            valid = false;
        }
    }
    const float part = blk::score_split_sum(valid ? blk::score_split_part<TK, HH>(qs, ws, k + row * k_row_stride, d, hg, vec) : 0.f);
    if (valid && hg == 0) scores[r * score_row_stride + j] = part;
}

template <typename TK>
cudaError_t run(const void* q, int q_dtype, const float* w, int H, int d, const TK* k,
                int64_t k_row_stride, int64_t k_rows, const Geom& g, int block_size,
                float* scores, int64_t score_row_stride, cudaStream_t st, const float* k_scale) {
    int max_keys = g.max_n_kv;
    if (block_size > 1) max_keys /= block_size;
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (max_keys <= 0 || n_rows == 0) return cudaSuccess;
    int HH = 1;
    while (HH < H) HH <<= 1;
    size_t sm = (size_t)(HH * d + HH) * sizeof(float);
    // pooled block keys with many heads: four threads per key
    if (block_size > 1 && HH >= 16 && sizeof(TK) != 1 && max_keys <= 65535 * kSplitKeys) {
        dim3 sgrid((unsigned)n_rows, (unsigned)((max_keys + kSplitKeys - 1) / kSplitKeys));
        auto kern = HH == 16 ? score_split_kernel<TK, 16> : (HH == 32 ? score_split_kernel<TK, 32> : score_split_kernel<TK, 64>);
        if (sm > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        const bool vec = !(reinterpret_cast<uintptr_t>(k) & 15u) && (k_row_stride * (int64_t)sizeof(TK)) % 16 == 0;
        return launch_pdl(kern, sgrid, dim3(128), sm, st, q, q_dtype, w, H, d, k, k_row_stride, k_rows, g,
                          block_size, scores, score_row_stride, vec);
    }
    const int tiles = (max_keys + kTile - 1) / kTile;
    dim3 grid((unsigned)n_rows, (unsigned)(tiles < 65535 ? tiles : 65535));
#define LIDX_SCORE_CASE(N)                                                                     \
    case N: {                                                                                  \
        auto kern = score_generic_kernel<TK, N>;                                               \
        if (sm > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm); \
        return launch_pdl(kern, grid, dim3(kTile), sm, st, q, q_dtype, w, H, d, k, k_row_stride, \
                          k_rows, g, block_size, scores, score_row_stride, k_scale);           \
    }
    switch (HH) {
        LIDX_SCORE_CASE(1)
        LIDX_SCORE_CASE(2)
        LIDX_SCORE_CASE(4)
        LIDX_SCORE_CASE(8)
        LIDX_SCORE_CASE(16)
        LIDX_SCORE_CASE(32)
        LIDX_SCORE_CASE(64)
        default: return cudaErrorNotSupported;
    }
#undef LIDX_SCORE_CASE
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_generic(const void* q, int q_dtype, const float* w, int H, int d,
                                 const void* k, int k_dtype, int64_t k_row_stride, int64_t k_rows,
                                 const Geom& g, int block_size, float* scores,
                                 int64_t score_row_stride, cudaStream_t st, const float* k_scale) {
    switch (k_dtype) {
        case IDX_F16:
            return run(q, q_dtype, w, H, d, static_cast<const __half*>(k), k_row_stride, k_rows, g,
                       block_size, scores, score_row_stride, st, nullptr);
        // (k_scale NULL with int8 keys: the scale is stored inline after each row's codes)
        case IDX_BF16:
            return run(q, q_dtype, w, H, d, static_cast<const __nv_bfloat16*>(k), k_row_stride,
                       k_rows, g, block_size, scores, score_row_stride, st, nullptr);
        case IDX_I8_ROWSCALE:
            return run(q, q_dtype, w, H, d, static_cast<const int8_t*>(k), k_row_stride, k_rows, g,
                       block_size, scores, score_row_stride, st, k_scale);
        default:
            return run(q, q_dtype, w, H, d, static_cast<const float*>(k), k_row_stride, k_rows, g,
                       block_size, scores, score_row_stride, st, nullptr);
    }
}

}  // namespace lidx
