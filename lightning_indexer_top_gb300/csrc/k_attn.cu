// Softmax attention of each query row over only its selected keys, on the
// CUDA cores:
//     l[h, j] = scale * q[r, h] . K[j, g(h)],  p = softmax_j(l),
//     out[r, h] = sum_j p[h, j] * V[j, g(h)]
// for j in the row's selected positions ("Gather OpenPangu DSA decode reads"
// and "Gather OpenPangu sparse prefill attention", ik_llama_opt commit log).
// With v == NULL the MLA latent form applies: one shared 576-wide latent row
// per token, and the value is its first dv columns ("openpangu: MLA-latent KV
// cache", same log).
//
// Grid (query rows, kv heads x head chunks).  A CTA of 4 warps serves one
// query row, one kv head and HC = 4*HPW of its query heads.  Per tile of 32
// selected keys it gathers the K (and V) rows into shared memory as f32;
// warp w then owns heads w, w+4, ...: lane l computes the logit of key l,
// the warp keeps a running max and sum (online softmax), and each lane
// accumulates dv/32 output columns.  Unselected lanes and invalid indices
// contribute p = 0 explicitly; no -inf enters any arithmetic.  The selected
// set may come in any order; padding entries (-1) are never read because only
// the first n_sel[r] entries are used.
#include <float.h>

#include "lidx_internal.cuh"

namespace lidx {
namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 32;

template <typename T, int HPW, int DVL>
__global__ void __launch_bounds__(kThreads) attn_generic_kernel(
    const T* __restrict__ q, int Hq, int Hkv, int dk, int dv, const T* __restrict__ k,
    const T* __restrict__ v, int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, Geom g,
    const int32_t* __restrict__ idx, int64_t idx_row_stride, const int32_t* __restrict__ n_sel,
    float scale, void* __restrict__ out, int out_dtype, int n_chunks) {
    constexpr int HC = 4 * HPW;
    extern __shared__ __align__(16) unsigned char sm_raw[];
    int64_t* rows_s = reinterpret_cast<int64_t*>(sm_raw);            // [kKeys] cache rows, -1 invalid
    float* qs = reinterpret_cast<float*>(sm_raw + kKeys * sizeof(int64_t));  // [HC][dk], pre-scaled
    float* ks = qs + HC * dk;                    // [kKeys][dk+1]
    float* vs = ks + kKeys * (dk + 1);           // [kKeys][dv] (GQA only)

    const int64_t r = blockIdx.x;
    const int gkv = blockIdx.y / n_chunks;       // kv head
    const int chunk = blockIdx.y % n_chunks;
    const int G = Hq / Hkv;
    const int h_base = gkv * G + chunk * HC;     // first query head of this CTA
    const int n_heads = min(HC, G - chunk * HC);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = (int)(r / g.T);
    const int n_kv_b = seq_n_kv(g, b);
    int ns = n_sel[r];
    if (ns < 0 || ns > idx_row_stride) {
        flag(g.status, IDX_ERR_DEVICE_BOUNDS);
        ns = ns < 0 ? 0 : (int)idx_row_stride;
    }

    for (int i = threadIdx.x; i < HC * dk; i += kThreads) {
        const int hl = i / dk, c = i % dk;
        qs[i] = hl < n_heads ? scale * to_f32(q[(r * Hq + h_base + hl) * (int64_t)dk + c]) : 0.f;
    }

    float o[HPW][DVL];
    float m_run[HPW], l_run[HPW];
    bool has_m[HPW];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        m_run[hh] = 0.f;
        l_run[hh] = 0.f;
        has_m[hh] = false;
#pragma unroll
        for (int i = 0; i < DVL; ++i) o[hh][i] = 0.f;
    }

    for (int t0 = 0; t0 < ns; t0 += kKeys) {
        __syncthreads();  // previous tile fully consumed (and qs written, first time)
        if (threadIdx.x < kKeys) {
            const int j = t0 + threadIdx.x;
            int64_t row = -1;
            if (j < ns) {
                const int pos = idx[r * idx_row_stride + j];
                const int64_t rr = (pos >= 0 && pos < n_kv_b) ? key_row(g, b, pos) : -1;
                if (rr >= 0 && rr < kv_rows) {
                    row = rr;
                } else {
                    flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                }
            }
            rows_s[threadIdx.x] = row;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kKeys * dk; e += kThreads) {
            const int key = e / dk, c = e % dk;
            const int64_t row = rows_s[key];
            ks[key * (dk + 1) + c] = row >= 0 ? to_f32(k[row * kv_row_stride + (int64_t)gkv * dk + c]) : 0.f;
        }
        if (v) {
            for (int e = threadIdx.x; e < kKeys * dv; e += kThreads) {
                const int key = e / dv, c = e % dv;
                const int64_t row = rows_s[key];
                vs[key * dv + c] = row >= 0 ? to_f32(v[row * v_row_stride + (int64_t)gkv * dv + c]) : 0.f;
            }
        }
        __syncthreads();

        const bool valid = rows_s[lane] >= 0;
        const float* vrow_base = v ? vs : ks;
        const int vstride = v ? dv : dk + 1;
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
            const int hl = warp + 4 * hh;
            if (hl >= n_heads) continue;  // warp-uniform
            const float* qh = qs + hl * dk;
            const float* kr = ks + lane * (dk + 1);
            float logit = 0.f;
            for (int c = 0; c < dk; ++c) logit = fmaf(qh[c], kr[c], logit);
            float tmax = valid ? logit : -FLT_MAX;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            if (__ballot_sync(0xffffffffu, valid) == 0u) continue;  // whole tile invalid
            const float m_new = has_m[hh] ? fmaxf(m_run[hh], tmax) : tmax;
            const float corr = has_m[hh] ? expf(m_run[hh] - m_new) : 0.f;
            const float p = valid ? expf(logit - m_new) : 0.f;
            float psum = p;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l_run[hh] = l_run[hh] * corr + psum;
#pragma unroll
            for (int i = 0; i < DVL; ++i) o[hh][i] *= corr;
            for (int key = 0; key < kKeys; ++key) {
                const float pk = __shfl_sync(0xffffffffu, p, key);
                const float* vr = vrow_base + key * vstride;
#pragma unroll
                for (int i = 0; i < DVL; ++i) {
                    const int c = lane + 32 * i;
                    if (c < dv) o[hh][i] = fmaf(pk, vr[c], o[hh][i]);
                }
            }
            m_run[hh] = m_new;
            has_m[hh] = true;
        }
    }

#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        const int hl = warp + 4 * hh;
        if (hl >= n_heads) continue;
        const float inv = l_run[hh] > 0.f ? 1.f / l_run[hh] : 0.f;
        const int64_t base = (r * Hq + h_base + hl) * (int64_t)dv;
#pragma unroll
        for (int i = 0; i < DVL; ++i) {
            const int c = lane + 32 * i;
            if (c >= dv) continue;
            const float val = o[hh][i] * inv;
            if (out_dtype == IDX_BF16)
                static_cast<__nv_bfloat16*>(out)[base + c] = __float2bfloat16_rn(val);
            else
                static_cast<float*>(out)[base + c] = val;
        }
    }
}

template <typename T, int HPW>
cudaError_t run_dv(const T* q, int Hq, int Hkv, int dk, int dv, const T* k, const T* v,
                   int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                   const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel, float scale,
                   void* out, int out_dtype, int n_chunks, cudaStream_t st) {
    constexpr int HC = 4 * HPW;
    const int64_t n_rows = (int64_t)g.B * g.T;
    dim3 grid((unsigned)n_rows, (unsigned)(Hkv * n_chunks));
    size_t sm = (size_t)(HC * dk + kKeys * (dk + 1) + (v ? kKeys * dv : 0)) * sizeof(float) +
                kKeys * sizeof(int64_t);
    const int dvl = (dv + 31) / 32;
#define LIDX_ATTN_CASE(N)                                                                       \
    if (dvl <= N) {                                                                             \
        auto kern = attn_generic_kernel<T, HPW, N>;                                             \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);       \
        kern<<<grid, kThreads, sm, st>>>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, \
                                         kv_rows, g, idx, idx_row_stride, n_sel, scale, out,    \
                                         out_dtype, n_chunks);                                  \
        return cudaGetLastError();                                                              \
    }
    LIDX_ATTN_CASE(1)
    LIDX_ATTN_CASE(2)
    LIDX_ATTN_CASE(4)
    LIDX_ATTN_CASE(8)
    LIDX_ATTN_CASE(16)
#undef LIDX_ATTN_CASE
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t run(const T* q, int Hq, int Hkv, int dk, int dv, const T* k, const T* v,
                int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel, float scale,
                void* out, int out_dtype, cudaStream_t st) {
    const int G = Hq / Hkv;
    if ((int64_t)g.B * g.T == 0) return cudaSuccess;
    if (G <= 4)
        return run_dv<T, 1>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                            idx_row_stride, n_sel, scale, out, out_dtype, 1, st);
    if (G <= 8)
        return run_dv<T, 2>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                            idx_row_stride, n_sel, scale, out, out_dtype, 1, st);
    return run_dv<T, 4>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                        idx_row_stride, n_sel, scale, out, out_dtype, (G + 15) / 16, st);
}

}  // namespace

cudaError_t launch_attn_generic(const void* q, int dtype, int Hq, int Hkv, int dk, int dv,
                                const void* k, const void* v, int64_t kv_row_stride,
                                int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                                const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
                                float scale, void* out, int out_dtype, cudaStream_t st) {
    switch (dtype) {
        case IDX_F16:
            return run(static_cast<const __half*>(q), Hq, Hkv, dk, dv, static_cast<const __half*>(k),
                       static_cast<const __half*>(v), kv_row_stride, v_row_stride, kv_rows, g, idx,
                       idx_row_stride, n_sel, scale, out, out_dtype, st);
        case IDX_BF16:
            return run(static_cast<const __nv_bfloat16*>(q), Hq, Hkv, dk, dv,
                       static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                       kv_row_stride, v_row_stride, kv_rows, g, idx, idx_row_stride, n_sel, scale,
                       out, out_dtype, st);
        default:
            return run(static_cast<const float*>(q), Hq, Hkv, dk, dv, static_cast<const float*>(k),
                       static_cast<const float*>(v), kv_row_stride, v_row_stride, kv_rows, g, idx,
                       idx_row_stride, n_sel, scale, out, out_dtype, st);
    }
}

}  // namespace lidx
