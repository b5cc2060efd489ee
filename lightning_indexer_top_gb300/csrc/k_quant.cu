// Per-row symmetric 8-bit code of key rows, the storage format of a quantized
// indexer key cache ("GLM-DSA: allow for quantized indexer cache", ik_llama_opt
// commit log):
//     scale[r] = max_c |x[r, c]| / 127,   q8[r, c] = clamp(rint(x[r, c] / scale[r]), -127, 127)
// in f32 with IEEE round-to-nearest-even division (so a CPU in f32 takes the
// same integer decisions).  The scale goes to its own array, or (scale NULL)
// into bytes d .. d+3 of the code row.  One warp per row; a cache-write op,
// off the scan.
#include "lidx_internal.cuh"

namespace lidx {
namespace {

constexpr int kWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) quantize_rows_kernel(const T* __restrict__ x, int64_t n_rows, int d,
                                                                   int64_t x_row_stride, int8_t* __restrict__ q8,
                                                                   int64_t q8_row_stride, float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (r >= n_rows) return;
    const T* xr = x + r * x_row_stride;
    float amax = 0.f;
    for (int c = lane; c < d; c += 32) amax = fmaxf(amax, fabsf(to_f32(xr[c])));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 127.f);
    int8_t* qr = q8 + r * q8_row_stride;
    for (int c = lane; c < d; c += 32) {
        float v = 0.f;
        if (s > 0.f) v = fminf(fmaxf(rintf(__fdiv_rn(to_f32(xr[c]), s)), -127.f), 127.f);
        qr[c] = (int8_t)(int)v;
    }
    if (lane == 0) {
        if (scale) scale[r] = s;
        else *reinterpret_cast<float*>(qr + d) = s;   // inline: the row's bytes d .. d+3
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const void* x, int x_dtype, int64_t n_rows, int d, int64_t x_row_stride,
                                 int8_t* q8, int64_t q8_row_stride, float* scale, cudaStream_t st) {
    if (n_rows == 0) return cudaSuccess;
    const int64_t blocks = (n_rows + kWarps - 1) / kWarps;
    if (blocks > INT32_MAX) return cudaErrorNotSupported;
    const dim3 grid((unsigned)blocks);
    switch (x_dtype) {
        case IDX_F16:
            quantize_rows_kernel<<<grid, kWarps * 32, 0, st>>>(static_cast<const __half*>(x), n_rows, d, x_row_stride,
                                                               q8, q8_row_stride, scale);
            break;
        case IDX_BF16:
            quantize_rows_kernel<<<grid, kWarps * 32, 0, st>>>(static_cast<const __nv_bfloat16*>(x), n_rows, d,
                                                               x_row_stride, q8, q8_row_stride, scale);
            break;
        default:
            quantize_rows_kernel<<<grid, kWarps * 32, 0, st>>>(static_cast<const float*>(x), n_rows, d, x_row_stride,
                                                               q8, q8_row_stride, scale);
    }
    return cudaGetLastError();
}

}  // namespace lidx
