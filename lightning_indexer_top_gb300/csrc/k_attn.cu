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
// Grid (query rows, kv heads x head chunks, key splits).  A CTA of 4 warps
// serves one query row, one kv head, HC = 4*HPW of its query heads and one
// split of the row's selected keys.  When the rows are few (a decode batch),
// the selection is split so that the CTAs cover the SMs; each split writes
// its unnormalised output with its running max and sum, and a combine kernel
// merges the splits (rescaling each by exp(m_s - max)).  Per tile of 32
// selected keys a CTA gathers the K (and V) rows into shared memory as f32
// (16-byte loads, all of a tile's in flight at once, when rows and head
// slices are 16-byte aligned);
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

// The K rows (dk elements from column kc0 of each row) and, with v, the V rows (dv elements from
// column vc0) of one tile of kKeys keys, copied as stored into shared memory: key `key` at
// ks[key * kp] and vs[key * vp].  Invalid keys (rows_s < 0) give zeros.  With `vec` each thread
// moves 16-byte pieces, all of a tile's loads issued before any store (one memory round trip per
// tile); otherwise element by element.
template <typename T>
__device__ __forceinline__ void gather_kv_tile(T* ks, T* vs, const T* __restrict__ k, const T* __restrict__ v,
                                               int64_t k_stride, int64_t v_stride, int64_t kc0, int64_t vc0, int dk,
                                               int dv, int kp, int vp, const int64_t* rows_s, bool vec) {
    if (vec) {
        constexpr int E = 16 / sizeof(T);      // elements per 16-byte piece
        constexpr int kBatch = 8;
        const int wk = dk / E, wv = v ? dv / E : 0;
        const int nk = kKeys * wk, total = nk + kKeys * wv;
        for (int e0 = threadIdx.x; e0 < total; e0 += kThreads * kBatch) {
            uint4 r[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int e = e0 + b * kThreads;
                r[b] = make_uint4(0u, 0u, 0u, 0u);
                if (e < total) {
                    const bool isk = e < nk;
                    const int ee = isk ? e : e - nk, w = isk ? wk : wv;
                    const int key = ee / w, c = (ee % w) * E;
                    const int64_t row = rows_s[key];
                    if (row >= 0)
                        r[b] = isk ? *reinterpret_cast<const uint4*>(k + row * k_stride + kc0 + c)
                                   : *reinterpret_cast<const uint4*>(v + row * v_stride + vc0 + c);
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int e = e0 + b * kThreads;
                if (e < total) {
                    const bool isk = e < nk;
                    const int ee = isk ? e : e - nk, w = isk ? wk : wv;
                    const int key = ee / w, c = (ee % w) * E;
                    *reinterpret_cast<uint4*>(isk ? ks + key * kp + c : vs + key * vp + c) = r[b];
                }
            }
        }
    } else {
        for (int e = threadIdx.x; e < kKeys * dk; e += kThreads) {
            const int key = e / dk, c = e % dk;
            const int64_t row = rows_s[key];
            ks[key * kp + c] = row >= 0 ? k[row * k_stride + kc0 + c] : from_f32<T>(0.f);
        }
        if (v) {
            for (int e = threadIdx.x; e < kKeys * dv; e += kThreads) {
                const int key = e / dv, c = e % dv;
                const int64_t row = rows_s[key];
                vs[key * vp + c] = row >= 0 ? v[row * v_stride + vc0 + c] : from_f32<T>(0.f);
            }
        }
    }
}

// eight consecutive shared-memory elements (16-byte aligned) widened to f32
template <typename T>
__device__ __forceinline__ void lds8(const T* p, float (&f)[8]) {
    if constexpr (sizeof(T) == 4) {
        const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = to_f32(e[i]);
    }
}

// two consecutive shared-memory elements (aligned to two elements) widened to f32
template <typename T>
__device__ __forceinline__ void lds2(const T* p, float& x, float& y) {
    if constexpr (sizeof(T) == 4) {
        const float2 a = *reinterpret_cast<const float2*>(p);
        x = a.x;
        y = a.y;
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        const T* e = reinterpret_cast<const T*>(&u);
        x = to_f32(e[0]);
        y = to_f32(e[1]);
    }
}

template <typename T, int HPW, int DV2>
__global__ void __launch_bounds__(kThreads, 4) attn_generic_kernel(
    const T* __restrict__ q, int Hq, int Hkv, int dk, int dv, const T* __restrict__ k,
    const T* __restrict__ v, int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, Geom g,
    const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
    float scale, void* __restrict__ out, int out_dtype, int n_chunks, bool vec, int splits, int kps,
    float* __restrict__ part_o, float* __restrict__ part_ml) {
    constexpr int HC = 4 * HPW;
    extern __shared__ __align__(16) unsigned char sm_raw[];
    // q as f32, rows of qp = dk rounded up to 8 (zero padding); K and V tiles as stored, K rows of
    // kp = qp + 16 bytes (16-byte aligned; the extra step spreads the 32 lanes' row reads over the
    // bank groups), V rows of vp elements (16-byte aligned)
    const int qp = (dk + 7) & ~7;
    const int kp = qp + 16 / (int)sizeof(T);
    const int vp = (dv + 15 / (int)sizeof(T)) / (16 / (int)sizeof(T)) * (16 / (int)sizeof(T));
    int64_t* rows_s = reinterpret_cast<int64_t*>(sm_raw);                     // [kKeys] cache rows, -1 invalid
    float* qs = reinterpret_cast<float*>(sm_raw + kKeys * sizeof(int64_t));   // [HC][qp], pre-scaled
    T* ks = reinterpret_cast<T*>(qs + HC * qp);                               // [kKeys][kp]
    T* vs = ks + kKeys * kp;                                                  // [kKeys][vp] (GQA only)

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

    for (int i = threadIdx.x; i < HC * qp; i += kThreads) {
        const int hl = i / qp, c = i % qp;
        qs[i] = (hl < n_heads && c < dk) ? scale * to_f32(q[(r * Hq + h_base + hl) * (int64_t)dk + c]) : 0.f;
    }
    // the K padding columns [dk, kp) are read (against zero q) and must hold finite values
    for (int i = threadIdx.x; i < kKeys * kp; i += kThreads) ks[i] = from_f32<T>(0.f);

    float o[HPW][2 * DV2];
    float m_run[HPW], l_run[HPW];
    bool has_m[HPW];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        m_run[hh] = 0.f;
        l_run[hh] = 0.f;
        has_m[hh] = false;
#pragma unroll
        for (int i = 0; i < 2 * DV2; ++i) o[hh][i] = 0.f;
    }

    const int split = blockIdx.z;
    const int t_end = min(ns, (split + 1) * kps);
    for (int t0 = split * kps; t0 < t_end; t0 += kKeys) {
        __syncthreads();  // previous tile fully consumed (and qs / padding written, first time)
        if (threadIdx.x < kKeys) {
            const int j = t0 + threadIdx.x;
            int64_t row = -1;
            if (j < t_end) {
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
        gather_kv_tile(ks, vs, k, v, kv_row_stride, v_row_stride, (int64_t)gkv * dk, (int64_t)gkv * dv, dk, dv, kp,
                       vp, rows_s, vec);
        __syncthreads();

        const bool valid = rows_s[lane] >= 0;
        if (__ballot_sync(0xffffffffu, valid) == 0u) continue;  // whole tile invalid (block-uniform)
        const T* vrow_base = v ? vs : ks;
        const int vstride = v ? vp : kp;
        // logits of this lane's key for the warp's heads: one 16-byte read of the key row per 8
        // dimensions, shared by the heads
        float logit[HPW];
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) logit[hh] = 0.f;
        const T* kr = ks + lane * kp;
        for (int c = 0; c < qp; c += 8) {
            float kv8[8];
            lds8(kr + c, kv8);
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) {
                const int hl = warp + 4 * hh;
                if (hl >= n_heads) continue;   // warp-uniform
                const float4 qa = *reinterpret_cast<const float4*>(qs + hl * qp + c);
                const float4 qb = *reinterpret_cast<const float4*>(qs + hl * qp + c + 4);
                float a = logit[hh];
                a = fmaf(qa.x, kv8[0], a);
                a = fmaf(qa.y, kv8[1], a);
                a = fmaf(qa.z, kv8[2], a);
                a = fmaf(qa.w, kv8[3], a);
                a = fmaf(qb.x, kv8[4], a);
                a = fmaf(qb.y, kv8[5], a);
                a = fmaf(qb.z, kv8[6], a);
                a = fmaf(qb.w, kv8[7], a);
                logit[hh] = a;
            }
        }
        float p[HPW];
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
            const int hl = warp + 4 * hh;
            p[hh] = 0.f;
            if (hl >= n_heads) continue;  // warp-uniform
            float tmax = valid ? logit[hh] : -FLT_MAX;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_new = has_m[hh] ? fmaxf(m_run[hh], tmax) : tmax;
            const float corr = has_m[hh] ? expf(m_run[hh] - m_new) : 0.f;
            p[hh] = valid ? expf(logit[hh] - m_new) : 0.f;
            float psum = p[hh];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l_run[hh] = l_run[hh] * corr + psum;
#pragma unroll
            for (int i = 0; i < 2 * DV2; ++i) o[hh][i] *= corr;
            m_run[hh] = m_new;
            has_m[hh] = true;
        }
        // o += p V: lane owns the column pairs 2*lane + 64*i; each pair is read once for all heads
        for (int key = 0; key < kKeys; ++key) {
            float pk[HPW];
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) pk[hh] = __shfl_sync(0xffffffffu, p[hh], key);
            const T* vr = vrow_base + key * vstride;
#pragma unroll
            for (int i = 0; i < DV2; ++i) {
                const int c = 2 * lane + 64 * i;
                if (c >= dv) continue;
                float x, y = 0.f;
                if (c + 1 < dv) {
                    lds2(vr + c, x, y);
                } else {
                    x = to_f32(vr[c]);
                }
#pragma unroll
                for (int hh = 0; hh < HPW; ++hh) {
                    o[hh][2 * i] = fmaf(pk[hh], x, o[hh][2 * i]);
                    o[hh][2 * i + 1] = fmaf(pk[hh], y, o[hh][2 * i + 1]);
                }
            }
        }
    }

    if (splits > 1) {
        // this split's unnormalised output, running max and sum (l = 0: no valid key)
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
            const int hl = warp + 4 * hh;
            if (hl >= n_heads) continue;
            const int64_t u = (r * splits + split) * (int64_t)Hq + h_base + hl;
#pragma unroll
            for (int i = 0; i < DV2; ++i) {
                const int c = 2 * lane + 64 * i;
                if (c < dv) part_o[u * dv + c] = o[hh][2 * i];
                if (c + 1 < dv) part_o[u * dv + c + 1] = o[hh][2 * i + 1];
            }
            if (lane == 0) {
                part_ml[2 * u] = has_m[hh] ? m_run[hh] : 0.f;
                part_ml[2 * u + 1] = l_run[hh];
            }
        }
        return;
    }
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        const int hl = warp + 4 * hh;
        if (hl >= n_heads) continue;
        const float inv = l_run[hh] > 0.f ? 1.f / l_run[hh] : 0.f;
        const int64_t base = (r * Hq + h_base + hl) * (int64_t)dv;
#pragma unroll
        for (int i = 0; i < DV2; ++i) {
            const int c = 2 * lane + 64 * i;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (c + e >= dv) continue;
                const float val = o[hh][2 * i + e] * inv;
                if (out_dtype == IDX_BF16)
                    static_cast<__nv_bfloat16*>(out)[base + c + e] = __float2bfloat16_rn(val);
                else
                    static_cast<float*>(out)[base + c + e] = val;
            }
        }
    }
}

// merges the key splits of one (row, head): o = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s
__global__ void __launch_bounds__(128) attn_generic_combine_kernel(const float* part_o, const float* part_ml,
                                                                   int splits, int Hq, int dv, void* __restrict__ out,
                                                                   int out_dtype) {
    const int64_t r = blockIdx.x;
    const int h = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    float M = 0.f;
    bool any = false;
    for (int s = 0; s < splits; ++s) {
        const int64_t u = (r * splits + s) * (int64_t)Hq + h;
        if (part_ml[2 * u + 1] > 0.f) {
            M = any ? fmaxf(M, part_ml[2 * u]) : part_ml[2 * u];
            any = true;
        }
    }
    float den = 0.f;
    for (int s = 0; s < splits; ++s) {
        const int64_t u = (r * splits + s) * (int64_t)Hq + h;
        const float l = part_ml[2 * u + 1];
        if (l > 0.f) den += expf(part_ml[2 * u] - M) * l;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int c = threadIdx.x; c < dv; c += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) {
            const int64_t u = (r * splits + s) * (int64_t)Hq + h;
            const float l = part_ml[2 * u + 1];
            if (l > 0.f) acc += expf(part_ml[2 * u] - M) * part_o[u * dv + c];
        }
        const int64_t o = (r * Hq + h) * (int64_t)dv + c;
        if (out_dtype == IDX_BF16)
            static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(acc * inv);
        else
            static_cast<float*>(out)[o] = acc * inv;
    }
}

template <typename T, int HPW>
cudaError_t run_dv(const T* q, int Hq, int Hkv, int dk, int dv, const T* k, const T* v,
                   int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                   const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel, float scale,
                   void* out, int out_dtype, int n_chunks, void* ws, size_t ws_bytes, cudaStream_t st) {
    constexpr int HC = 4 * HPW;
    const int64_t n_rows = (int64_t)g.B * g.T;
    const size_t per_split = (size_t)n_rows * Hq * (dv + 2) * sizeof(float);
    int splits = generic_attn_splits(n_rows, idx_row_stride);
    if (splits > 1 && (!ws || (reinterpret_cast<uintptr_t>(ws) & 15u))) splits = 1;
    if (splits > 1 && (size_t)splits * per_split > ws_bytes) splits = (int)(ws_bytes / per_split);
    if (splits < 1) splits = 1;
    const int kps = (int)(((idx_row_stride + splits - 1) / splits + kKeys - 1) / kKeys * kKeys);
    float* part_o = splits > 1 ? static_cast<float*>(ws) : nullptr;
    float* part_ml = splits > 1 ? part_o + (size_t)n_rows * splits * Hq * dv : nullptr;
    const size_t ts = sizeof(T);
    const bool vec = dk % 8 == 0 && dv % 8 == 0 && !(reinterpret_cast<uintptr_t>(k) & 15u) &&
                     !(reinterpret_cast<uintptr_t>(v) & 15u) && (kv_row_stride * ts) % 16 == 0 &&
                     (!v || (v_row_stride * ts) % 16 == 0) && (dk * ts) % 16 == 0 && (dv * ts) % 16 == 0;
    dim3 grid((unsigned)n_rows, (unsigned)(Hkv * n_chunks), (unsigned)splits);
    const int qp = (dk + 7) & ~7;
    const int el = 16 / (int)sizeof(T);
    const int kp = qp + el, vp = (dv + el - 1) / el * el;
    size_t sm = (size_t)HC * qp * sizeof(float) + (size_t)kKeys * (kp + (v ? vp : 0)) * sizeof(T) +
                kKeys * sizeof(int64_t);
    const int dv2 = (dv + 63) / 64;   // column pairs per lane
#define LIDX_ATTN_CASE(N)                                                                       \
    if (dv2 <= N) {                                                                             \
        auto kern = attn_generic_kernel<T, HPW, N>;                                             \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);       \
        kern<<<grid, kThreads, sm, st>>>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, \
                                         kv_rows, g, idx, idx_row_stride, n_sel, scale, out,    \
                                         out_dtype, n_chunks, vec, splits, kps, part_o, part_ml); \
        cudaError_t e = cudaGetLastError();                                                     \
        if (e != cudaSuccess || splits == 1) return e;                                          \
        return launch_attn_generic_combine(part_o, part_ml, splits, n_rows, Hq, dv, out, out_dtype, st); \
    }
    LIDX_ATTN_CASE(1)
    LIDX_ATTN_CASE(2)
    LIDX_ATTN_CASE(4)
    LIDX_ATTN_CASE(8)
#undef LIDX_ATTN_CASE
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t run(const T* q, int Hq, int Hkv, int dk, int dv, const T* k, const T* v,
                int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel, float scale,
                void* out, int out_dtype, void* ws, size_t ws_bytes, cudaStream_t st) {
    const int G = Hq / Hkv;
    if ((int64_t)g.B * g.T == 0) return cudaSuccess;
    if (G <= 4)
        return run_dv<T, 1>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                            idx_row_stride, n_sel, scale, out, out_dtype, 1, ws, ws_bytes, st);
    if (G <= 8)
        return run_dv<T, 2>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                            idx_row_stride, n_sel, scale, out, out_dtype, 1, ws, ws_bytes, st);
    return run_dv<T, 4>(q, Hq, Hkv, dk, dv, k, v, kv_row_stride, v_row_stride, kv_rows, g, idx,
                        idx_row_stride, n_sel, scale, out, out_dtype, (G + 15) / 16, ws, ws_bytes, st);
}

}  // namespace

// key splits per (row, kv head) for few rows: enough CTAs to cover the SMs twice, at least 128
// selected keys per split; many rows need none
int generic_attn_splits(int64_t n_rows, int64_t cap) {
    if (n_rows <= 0) return 1;
    int sms = sm_count();
    if (sms < 2) sms = 152;
    int64_t s = 2 * (int64_t)sms / n_rows;
    const int64_t by_keys = (cap + 127) / 128;
    if (s > by_keys) s = by_keys;
    if (s > 64) s = 64;
    return s < 1 ? 1 : (int)s;
}

cudaError_t launch_attn_generic_combine(const float* part_o, const float* part_ml, int splits, int64_t n_rows, int Hq,
                                        int dv, void* out, int out_dtype, cudaStream_t st) {
    return launch_pdl(attn_generic_combine_kernel, dim3((unsigned)n_rows, (unsigned)Hq), dim3(128), 0, st, part_o,
                      part_ml, splits, Hq, dv, out, out_dtype);
}

size_t generic_attn_workspace_bytes(int64_t n_rows, int64_t cap, int Hq, int dv) {
    const int s = generic_attn_splits(n_rows, cap);
    if (s <= 1 || Hq < 1 || dv < 1) return 0;
    return (size_t)n_rows * s * Hq * (dv + 2) * sizeof(float);
}

cudaError_t launch_attn_generic(const void* q, int dtype, int Hq, int Hkv, int dk, int dv,
                                const void* k, const void* v, int64_t kv_row_stride,
                                int64_t v_row_stride, int64_t kv_rows, const Geom& g,
                                const int32_t* idx, int64_t idx_row_stride, const int32_t* n_sel,
                                float scale, void* out, int out_dtype, void* ws, size_t ws_bytes,
                                cudaStream_t st) {
    switch (dtype) {
        case IDX_F16:
            return run(static_cast<const __half*>(q), Hq, Hkv, dk, dv, static_cast<const __half*>(k),
                       static_cast<const __half*>(v), kv_row_stride, v_row_stride, kv_rows, g, idx,
                       idx_row_stride, n_sel, scale, out, out_dtype, ws, ws_bytes, st);
        case IDX_BF16:
            return run(static_cast<const __nv_bfloat16*>(q), Hq, Hkv, dk, dv,
                       static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                       kv_row_stride, v_row_stride, kv_rows, g, idx, idx_row_stride, n_sel, scale,
                       out, out_dtype, ws, ws_bytes, st);
        default:
            return run(static_cast<const float*>(q), Hq, Hkv, dk, dv, static_cast<const float*>(k),
                       static_cast<const float*>(v), kv_row_stride, v_row_stride, kv_rows, g, idx,
                       idx_row_stride, n_sel, scale, out, out_dtype, ws, ws_bytes, st);
    }
}

}  // namespace lidx
