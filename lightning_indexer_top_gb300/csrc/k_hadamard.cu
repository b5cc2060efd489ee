// Walsh-Hadamard rotation of d-element rows: y = H_d x with the
// orthonormal Sylvester matrix (natural order), stored as the exact rotation
// rounded once (nearest even) to the storage type.  Score preserving because
// (Hq).(Hk) = q.k (ik_llama.cpp PR #2058, commit "Add GLM-5.2/DeepSeek-V3.2
// DSA lightning indexer"); the cached indexer key is stored rotated (commit
// "decode-correct via persistent indexer-K cache").
//
// One warp per row.  Lane l holds the M = d/32 consecutive elements
// [l*M, l*M + M).  Butterfly stage h pairs element e with e ^ h: for h < M
// both live in the same lane, otherwise the partner lane is l ^ (h/M) and the
// value travels by shuffle.  After log2(d) stages element e holds
//     sum_j (-1)^popcount(e & j) x_j.
//
// Rounding once, for 16-bit storage: the butterflies run in f32, and the f32
// result y of each element is certified.  Each output is a +-sum of all d
// inputs formed by a tree of log2(d) rounded additions, so its error is at
// most log2(d) * 2^-24 * sum_j |x_j|; the scaling by f32(1/sqrt(d)) and its
// rounding add two more units, and forming y -+ err one more.  The bound used,
// (log2(d) + 6) * 2^-24 * sum|x| / sqrt(d), covers all of these.  If y - err
// and y + err round to the same storage value, the exact rotation rounds to
// it too (rounding is monotonic).  The rare elements whose interval straddles
// a rounding boundary are recomputed by the whole warp in f64 (each lane sums
// its M signed inputs, then a shuffle tree), divided by sqrt(d) in f64 and
// rounded once.  f32 storage runs every stage in f64 and rounds once.
//
// HBM-bound: one read and one write of each row.
#include "lidx_internal.cuh"

namespace lidx {
namespace {

__device__ __forceinline__ uint16_t bits_of(__half x) { return __half_as_ushort(x); }
__device__ __forceinline__ uint16_t bits_of(__nv_bfloat16 x) { return __bfloat16_as_ushort(x); }

// f64 -> 16-bit storage with one rounding to nearest even
__device__ __forceinline__ __half round_once(double v, __half*) { return __double2half(v); }
__device__ __forceinline__ __nv_bfloat16 round_once(double v, __nv_bfloat16*) { return __double2bfloat16(v); }

template <typename T, int M>
__global__ void __launch_bounds__(256) hadamard_kernel(const T* x, T* y, int64_t n_rows, int64_t row_stride,
                                                       float inv_sqrt_d, double sqrt_d64, int log2d) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= n_rows) return;   // warp-uniform
    const T* p = x + row * row_stride + lane * M;
    T* o = y + row * row_stride + lane * M;
    float x0[M];
#pragma unroll
    for (int i = 0; i < M; ++i) x0[i] = to_f32(p[i]);

    if constexpr (sizeof(T) == 4) {
        // f32 storage: every stage in f64, one rounding at the end
        double v[M];
#pragma unroll
        for (int i = 0; i < M; ++i) v[i] = (double)x0[i];
#pragma unroll
        for (int h = 1; h < M; h <<= 1) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                if ((i & h) == 0) {
                    const double a = v[i], b = v[i + h];
                    v[i] = a + b;
                    v[i + h] = a - b;
                }
            }
        }
#pragma unroll
        for (int hl = 1; hl < 32; hl <<= 1) {
            const bool upper = (lane & hl) != 0;
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const double other = __shfl_xor_sync(0xffffffffu, v[i], hl);
                v[i] = upper ? other - v[i] : v[i] + other;
            }
        }
#pragma unroll
        for (int i = 0; i < M; ++i) o[i] = (T)(v[i] / sqrt_d64);
    } else {
        float v[M];
        float l1 = 0.f;
#pragma unroll
        for (int i = 0; i < M; ++i) {
            v[i] = x0[i];
            l1 += fabsf(x0[i]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        // stages inside a lane
#pragma unroll
        for (int h = 1; h < M; h <<= 1) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                if ((i & h) == 0) {
                    const float a = v[i], b = v[i + h];
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
                const float other = __shfl_xor_sync(0xffffffffu, v[i], hl);
                v[i] = upper ? other - v[i] : v[i] + other;
            }
        }
        // certify each rounding (see the header); the bound is taken 1% larger for its own roundings
        const float err = (float)(log2d + 6) * 5.9604645e-8f * l1 * inv_sqrt_d * 1.01f;
        T out[M];
        uint32_t unsure = 0;
#pragma unroll
        for (int i = 0; i < M; ++i) {
            const float yv = v[i] * inv_sqrt_d;
            out[i] = from_f32<T>(yv);
            const uint16_t b = bits_of(out[i]);
            if (bits_of(from_f32<T>(yv - err)) != b || bits_of(from_f32<T>(yv + err)) != b) unsure |= 1u << i;
        }
        // exact recomputation of the uncertain elements, one at a time, by the whole warp
        uint32_t lanes = __ballot_sync(0xffffffffu, unsure != 0);
        while (lanes) {
            const int src = __ffs(lanes) - 1;
            uint32_t m = __shfl_sync(0xffffffffu, unsure, src);
            while (m) {
                const int i = __ffs(m) - 1;
                m &= m - 1;
                const int e = src * M + i;   // element index in the row
                double part = 0.0;
#pragma unroll
                for (int k = 0; k < M; ++k) {
                    const int j = lane * M + k;
                    part += (__popc(e & j) & 1) ? -(double)x0[k] : (double)x0[k];
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
                if (lane == src) {
#pragma unroll
                    for (int k = 0; k < M; ++k)
                        if (k == i) out[k] = round_once(part / sqrt_d64, (T*)nullptr);
                }
            }
            lanes &= lanes - 1;
        }
#pragma unroll
        for (int i = 0; i < M; ++i) o[i] = out[i];
    }
}

template <typename T>
cudaError_t run(const T* x, T* y, int64_t n_rows, int d, int64_t row_stride, cudaStream_t st) {
    const int warps = 8;
    dim3 grid((unsigned)((n_rows + warps - 1) / warps));
    const double s64 = sqrt((double)d);
    const float s = (float)(1.0 / s64);
    switch (d) {
        case 32: hadamard_kernel<T, 1><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, s64, 5); break;
        case 64: hadamard_kernel<T, 2><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, s64, 6); break;
        case 128: hadamard_kernel<T, 4><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, s64, 7); break;
        case 256: hadamard_kernel<T, 8><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, s64, 8); break;
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
