// Walsh-Hadamard rotation of d-element rows: y = H_d x with the
// orthonormal Sylvester matrix (natural order).  Score preserving because
// (Hq).(Hk) = q.k (ik_llama.cpp PR #2058, commit "Add GLM-5.2/DeepSeek-V3.2
// DSA lightning indexer"); the cached indexer key is stored rotated (commit
// "decode-correct via persistent indexer-K cache").
//
// One warp per row.  Lane l holds the M = d/32 consecutive elements
// [l*M, l*M + M).  Butterfly stage h pairs element e with e ^ h: for h < M
// both live in the same lane, otherwise the partner lane is l ^ (h/M) and the
// value travels by shuffle.  Work is log2(d) add/sub stages in f32, then one
// scale by 1/sqrt(d) and one rounding to the storage type.  HBM-bound: one
// read and one write of each row.
#include "lidx_internal.cuh"

namespace lidx {
namespace {

template <typename T, int M>
__global__ void __launch_bounds__(256) hadamard_kernel(const T* x, T* y, int64_t n_rows,
                                                       int64_t row_stride, float inv_sqrt_d) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= n_rows) return;
    const T* p = x + row * row_stride + lane * M;
    T* o = y + row * row_stride + lane * M;
    float v[M];
#pragma unroll
    for (int i = 0; i < M; ++i) v[i] = to_f32(p[i]);

    // stages inside a lane
#pragma unroll
    for (int h = 1; h < M; h <<= 1) {
#pragma unroll
        for (int i = 0; i < M; ++i) {
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
        }
    }
    // stages across lanes
#pragma unroll
    for (int hl = 1; hl < 32; hl <<= 1) {
        const bool upper = (lane & hl) != 0;
#pragma unroll
        for (int i = 0; i < M; ++i) {
            float other = __shfl_xor_sync(0xffffffffu, v[i], hl);
            v[i] = upper ? other - v[i] : v[i] + other;
        }
    }
#pragma unroll
    for (int i = 0; i < M; ++i) o[i] = from_f32<T>(v[i] * inv_sqrt_d);
}

template <typename T>
cudaError_t run(const T* x, T* y, int64_t n_rows, int d, int64_t row_stride, cudaStream_t st) {
    const int warps = 8;
    dim3 grid((unsigned)((n_rows + warps - 1) / warps));
    const float s = (float)(1.0 / sqrt((double)d));
    switch (d) {
        case 32: hadamard_kernel<T, 1><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s); break;
        case 64: hadamard_kernel<T, 2><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s); break;
        case 128: hadamard_kernel<T, 4><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s); break;
        case 256: hadamard_kernel<T, 8><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hadamard(const void* x, void* y, int dtype, int64_t n_rows, int d,
                            int64_t row_stride, cudaStream_t st) {
    if (n_rows == 0) return cudaSuccess;
    switch (dtype) {
        case IDX_F16:
            return run(static_cast<const __half*>(x), static_cast<__half*>(y), n_rows, d, row_stride, st);
        case IDX_BF16:
            return run(static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), n_rows, d,
                       row_stride, st);
        default:
            return run(static_cast<const float*>(x), static_cast<float*>(y), n_rows, d, row_stride, st);
    }
}

}  // namespace lidx
