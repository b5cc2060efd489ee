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
// result y of each element is certified.  Each output is a +-sum of the d
// inputs formed by a tree of rounded additions; an addition's rounding error
// is at most 2^-24 of its computed result and reaches the output with weight
// +-1, so the error is at most 2^-24 times the sum E of |result| over the
// tree's additions, which the kernel tracks alongside the butterflies (about
// five times tighter than log2(d) * 2^-24 * sum|x|).  Scaling by f32(1/sqrt d),
// its rounding and forming y -+ err add a few units of |y|.  If y - err and
// y + err round to the same storage value, the exact rotation rounds to it
// too (rounding is monotonic).  The rare elements whose interval straddles
// a rounding boundary are recomputed by the whole warp in double-word f32
// arithmetic (error-free two-sums: each lane sums its M signed inputs, then a
// shuffle tree of (hi, lo) pairs; an exact product with 1/sqrt(d) as an f32
// pair), about 2^-44 relative, and rounded once with the halfway cases decided
// by the low word.  (f64 would do, but GB300's f64 rate makes those few
// recomputations dominate the kernel.)  f32 storage runs every stage in f64.
//
// HBM-bound: one read and one write of each row.
#include "lidx_internal.cuh"

namespace lidx {
namespace {

__device__ __forceinline__ uint16_t bits_of(__half x) { return __half_as_ushort(x); }
__device__ __forceinline__ uint16_t bits_of(__nv_bfloat16 x) { return __bfloat16_as_ushort(x); }

__device__ __forceinline__ __half half_of_bits(uint16_t b) { return __ushort_as_half(b); }
__device__ __forceinline__ __nv_bfloat16 bf16_of_bits(uint16_t b) { return __ushort_as_bfloat16(b); }
template <typename T> __device__ __forceinline__ T of_bits(uint16_t b);
template <> __device__ __forceinline__ __half of_bits<__half>(uint16_t b) { return half_of_bits(b); }
template <> __device__ __forceinline__ __nv_bfloat16 of_bits<__nv_bfloat16>(uint16_t b) { return bf16_of_bits(b); }

// a + b = s + e exactly (Knuth's two-sum, no contraction)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) renormalised so that hi = fl(hi + lo), |a| >= |b| assumed
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// The value y = hi + lo (|lo| <= half an f32 ulp of hi) rounded once to nearest even in T.
// Rounding hi alone is right unless hi lies exactly halfway between two T values (the halfway
// points of T are f32 numbers): then the sign of lo decides, and lo == 0 is a true tie.
template <typename T>
__device__ __forceinline__ T round_pair(float hi, float lo) {
    const T r = from_f32<T>(hi);
    const float t = to_f32(r);
    if (t == hi || lo == 0.f || !isfinite(hi)) return r;
    // the T neighbour of r on hi's side of it
    const uint16_t u = bits_of(r);
    const bool up = hi > t;                       // the neighbour is the larger value
    const uint16_t mag = u & 0x7fffu, sgn = u & 0x8000u;
    uint16_t nb;
    if (mag == 0) nb = (uint16_t)(up ? 0x0001u : 0x8001u);      // across zero: the smallest subnormal
    else nb = (uint16_t)(((up != (sgn != 0)) ? mag + 1 : mag - 1) | sgn);
    const float nt = to_f32(of_bits<T>(nb));
    if (!isfinite(nt) || 0.5f * (t + nt) != hi) return r;        // not halfway: r is right
    const bool toward_larger = lo > 0.f;
    return (toward_larger == (nt > t)) ? of_bits<T>(nb) : r;
}

template <typename T, int M>
__global__ void __launch_bounds__(256) hadamard_kernel(const T* x, T* y, int64_t n_rows, int64_t row_stride,
                                                       float inv_sqrt_d, float inv_hi, float inv_lo, double sqrt_d64, int log2d) {
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
        // v: the butterfly values; E: for each position, the sum of |value| over every addition in
        // the tree that produced it (the leaves are exact inputs).  Rounding errors of additions
        // pass to the output with weight +-1, and each is at most 2^-24 of its (computed) result,
        // so 2^-24 * E bounds the output's error.
        float v[M], E[M];
#pragma unroll
        for (int i = 0; i < M; ++i) {
            v[i] = x0[i];
            E[i] = 0.f;
        }
        // stages inside a lane
#pragma unroll
        for (int h = 1; h < M; h <<= 1) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                if ((i & h) == 0) {
                    const float a = v[i], b = v[i + h];
                    v[i] = a + b;
                    v[i + h] = a - b;
                    const float eab = E[i] + E[i + h];
                    E[i] = eab + fabsf(v[i]);
                    E[i + h] = eab + fabsf(v[i + h]);
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
                const float eo = __shfl_xor_sync(0xffffffffu, E[i], hl);
                v[i] = upper ? other - v[i] : v[i] + other;
                E[i] = E[i] + eo + fabsf(v[i]);
            }
        }
        (void)log2d;
        T out[M];
        uint32_t unsure = 0;
#pragma unroll
        for (int i = 0; i < M; ++i) {
            // certify the rounding (see the header): the additions' bound (1% larger for the
            // roundings of E itself), plus 4 units of |v| for 1/sqrt(d)'s own error, the scaling
            // product and forming y -+ err
            const float err = 5.9604645e-8f * inv_sqrt_d * (1.01f * E[i] + 4.f * fabsf(v[i]));
            const float yv = v[i] * inv_sqrt_d;
            out[i] = from_f32<T>(yv);
            const uint16_t b = bits_of(out[i]);
            if (bits_of(from_f32<T>(yv - err)) != b || bits_of(from_f32<T>(yv + err)) != b) unsure |= 1u << i;
        }
        // the uncertain elements, one at a time, by the whole warp in double-word f32 arithmetic:
        // each lane sums its M signed inputs with exact two-sums, the warp adds the (hi, lo) pairs,
        // the pair is scaled by 1/sqrt(d) = c_hi + c_lo with an exact product, and rounded once
        uint32_t lanes = __ballot_sync(0xffffffffu, unsure != 0);
        while (lanes) {
            const int src = __ffs(lanes) - 1;
            uint32_t m = __shfl_sync(0xffffffffu, unsure, src);
            while (m) {
                const int i = __ffs(m) - 1;
                m &= m - 1;
                const int e = src * M + i;   // element index in the row
                float hi = 0.f, lo = 0.f;
#pragma unroll
                for (int k = 0; k < M; ++k) {
                    const int j = lane * M + k;
                    float sv, ev;
                    two_sum(hi, (__popc(e & j) & 1) ? -x0[k] : x0[k], sv, ev);
                    hi = sv;
                    lo = __fadd_rn(lo, ev);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float oh = __shfl_xor_sync(0xffffffffu, hi, off), ol = __shfl_xor_sync(0xffffffffu, lo, off);
                    float sv, ev;
                    two_sum(hi, oh, sv, ev);
                    const float l2 = __fadd_rn(__fadd_rn(lo, ol), ev);
                    fast_two_sum(sv, l2, hi, lo);
                }
                if (lane == src) {
                    const float p = __fmul_rn(hi, inv_hi);
                    const float pe = fmaf(hi, inv_hi, -p);                          // exact product error
                    const float t = fmaf(hi, inv_lo, fmaf(lo, inv_hi, pe));
                    float yh, yl;
                    fast_two_sum(p, t, yh, yl);
#pragma unroll
                    for (int k = 0; k < M; ++k)
                        if (k == i) out[k] = round_pair<T>(yh, yl);
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
    const double inv = 1.0 / s64;
    const float s = (float)inv;
    const float ih = (float)inv, il = (float)(inv - (double)ih);   // 1/sqrt(d) as an f32 pair
    switch (d) {
        case 32: hadamard_kernel<T, 1><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, ih, il, s64, 5); break;
        case 64: hadamard_kernel<T, 2><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, ih, il, s64, 6); break;
        case 128: hadamard_kernel<T, 4><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, ih, il, s64, 7); break;
        case 256: hadamard_kernel<T, 8><<<grid, warps * 32, 0, st>>>(x, y, n_rows, row_stride, s, ih, il, s64, 8); break;
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
