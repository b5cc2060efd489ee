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
#include "lidx_internal.cuh"

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
    constexpr int HG = HH / 4;   // heads per thread
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
    if (q_dtype != IDX_F32 && d % 8 == 0 && !(reinterpret_cast<uintptr_t>(q) & 15u)) {
        // 16-bit q: 8 elements per 16-byte load, a thread's loads issued together
        constexpr int kQB = 8;
        const int n8 = HH * d / 8;
        for (int i0 = threadIdx.x; i0 < n8; i0 += kQB * blockDim.x) {
            uint4 raw[kQB];
#pragma unroll
            for (int u = 0; u < kQB; ++u) {
                const int i = i0 + u * blockDim.x;
                const int h = (i * 8) / d, c = (i * 8) % d;
                raw[u] = (i < n8 && h < H)
                             ? *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(q) + (r * H + h) * (int64_t)d + c)
                             : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kQB; ++u) {
                const int i = i0 + u * blockDim.x;
                if (i >= n8) break;
                const int h = (i * 8) / d, c = (i * 8) % d;
                const uint16_t* e = reinterpret_cast<const uint16_t*>(&raw[u]);
#pragma unroll
                for (int x = 0; x < 8; ++x)
                    qs[(c + x) * HH + h] = q_dtype == IDX_BF16 ? __bfloat162float(__ushort_as_bfloat16(e[x]))
                                                               : __half2float(__ushort_as_half(e[x]));
            }
        }
    } else {
        for (int i = threadIdx.x; i < HH * d; i += blockDim.x) {
            const int h = i % HH, c = i / HH;
            qs[i] = h < H ? load_any(q, (r * H + h) * (int64_t)d + c, q_dtype) : 0.f;
        }
    }
    for (int i = threadIdx.x; i < HH; i += blockDim.x) ws[i] = (i < H) ? w[r * H + i] : 0.f;
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
    float part = 0.f;
    if (valid) {
        const TK* kr = k + row * k_row_stride;
        float acc[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) acc[h] = 0.f;
        // 32 dimensions of the key row in flight at a time (8 loads of 4), then their products
        constexpr int kKB = 32;
        for (int c00 = 0; c00 < d; c00 += kKB) {
            float kv[kKB];
            if (vec && sizeof(TK) == 4 && c00 + kKB <= d) {
#pragma unroll
                for (int u = 0; u < kKB / 4; ++u) {
                    const float4 x = *reinterpret_cast<const float4*>(kr + c00 + 4 * u);
                    kv[4 * u] = x.x;
                    kv[4 * u + 1] = x.y;
                    kv[4 * u + 2] = x.z;
                    kv[4 * u + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < kKB; ++i) kv[i] = (c00 + i < d) ? to_f32(kr[c00 + i]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kKB; ++i) {
                if (c00 + i >= d) break;
                const float4* qc = reinterpret_cast<const float4*>(qs + (c00 + i) * HH + hg * HG);
#pragma unroll
                for (int h4 = 0; h4 < HG / 4; ++h4) {
                    const float4 qq = qc[h4];
                    acc[4 * h4] = fmaf(qq.x, kv[i], acc[4 * h4]);
                    acc[4 * h4 + 1] = fmaf(qq.y, kv[i], acc[4 * h4 + 1]);
                    acc[4 * h4 + 2] = fmaf(qq.z, kv[i], acc[4 * h4 + 2]);
                    acc[4 * h4 + 3] = fmaf(qq.w, kv[i], acc[4 * h4 + 3]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) part = fmaf(ws[hg * HG + h], fmaxf(acc[h], 0.f), part);
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    if (valid && hg == 0) scores[r * score_row_stride + j] = part + 0.0f;
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
