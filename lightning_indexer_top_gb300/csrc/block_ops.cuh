// Device building blocks of the block-pooled indexer, shared by the separate
// kernels (idx_block_pool[_update], idx_score over pooled keys, idx_topk in
// block mode) and by their one-launch form (idx_block_score_topk), so that
// both give bit-identical pooled keys, scores and selections.
//
//   pool_block        p[b, beta, :] = (1/C) * sum_{t < C} k_raw[row(b, beta*C + t), :]
//                     (llama.cpp commit c88c916636, QSA commit message: block
//                     keys are the mean of the block's raw keys)
//   score_split_part  one thread's share of a pooled key's score
//                     sum_h w_h * relu(q_h . k) (DeepSeek-V3.2 lightning indexer,
//                     eq. 1, with the block key in the token key's place)
//   block_rank_row    the best min(floor(top_k/C), n_cb) complete blocks (lower
//                     block index wins ties, -0 == +0), expanded to their
//                     positions in ascending order, then the tail tokens
#pragma once

#include "lidx_internal.cuh"

namespace lidx {
namespace blk {

// ---------------------------------------------------------------------------
// Block mean-pool.  Threads [0, kPoolThreads) of the CTA do the work; with
// 16-byte vector loads a row of d elements takes tpr = d*size/16 threads, so
// the group reads rp = kPoolThreads/tpr rows at once; each thread sums its rows
// (t = rg, rg + rp, ...) in order in f32, eight rows' loads in flight, and the
// rp partial sums are added in order in shared memory (part: rp*d floats).
// Every thread of the CTA must call it (it crosses two CTA barriers).
// ---------------------------------------------------------------------------
constexpr int kPoolThreads = 128;

template <typename T>
__device__ __forceinline__ void pool_block(const T* k, int64_t k_row_stride, int64_t k_rows, const Geom& g, int C,
                                           int d, int b, int beta, float* part, float* pooled_row) {
    constexpr int V = 16 / sizeof(T);
    const int tpr = d / V;               // threads per row
    const int rp = kPoolThreads / tpr;   // rows per pass
    const int rg = threadIdx.x / tpr, cv = threadIdx.x % tpr;
    if (threadIdx.x < kPoolThreads && rg < rp) {
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        constexpr int kBatch = 8;
        for (int t0 = rg; t0 < C; t0 += kBatch * rp) {
            uint4 raw[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                raw[u] = make_uint4(0u, 0u, 0u, 0u);
                const int t = t0 + u * rp;
                if (t < C) {
                    const int64_t row = key_row(g, b, (int64_t)beta * C + t);
                    if (row < 0 || row >= k_rows)
                        flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                    else
                        raw[u] = *reinterpret_cast<const uint4*>(k + row * k_row_stride + cv * V);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (t0 + u * rp >= C) break;
                const T* e = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += to_f32(e[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) part[rg * d + cv * V + i] = acc[i];
    }
    __syncthreads();
    if (threadIdx.x < kPoolThreads) {
        for (int c = threadIdx.x; c < d; c += kPoolThreads) {
            float sum = 0.f;
            for (int i = 0; i < rp; ++i) sum += part[i * d + c];
            pooled_row[c] = sum / (float)C;
        }
    }
    __syncthreads();
}

// first pooled block of sequence b to (re)write: after the current ones, and from the stale one on
__device__ __forceinline__ int pool_first_block(const int32_t* n_pooled, const int32_t* stale_pos, int b, int C,
                                                int n_cb) {
    int beta0 = 0;
    if (n_pooled) beta0 = max(n_pooled[b], 0);
    if (stale_pos) {
        const int sp = stale_pos[b];
        beta0 = min(beta0, sp < 0 ? 0 : sp / C);
    }
    return min(beta0, n_cb);
}

// ---------------------------------------------------------------------------
// Pooled-key scores, four threads per key: the row's q as f32 in shared memory
// transposed to qs[d][HH] (heads >= H zero) and its weights ws[HH]; thread hg
// of a key's four takes heads [hg*HH/4, (hg+1)*HH/4), sums over the d
// dimensions in order, and returns sum_h w_h * relu(acc_h) over its heads; the
// four partials are added by two xor shuffles (lanes 4i..4i+3 hold one key).
// ---------------------------------------------------------------------------
template <int HH>
__device__ __forceinline__ void load_q_split(const void* q, int q_dtype, const float* w, int H, int d, int64_t r,
                                             float* qs, float* ws) {
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
}

template <typename TK, int HH>
__device__ __forceinline__ float score_split_part(const float* qs, const float* ws, const TK* kr, int d, int hg,
                                                  bool vec) {
    constexpr int HG = HH / 4;   // heads per thread
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
    float part = 0.f;
#pragma unroll
    for (int h = 0; h < HG; ++h) part = fmaf(ws[hg * HG + h], fmaxf(acc[h], 0.f), part);
    return part;
}

// score_split_part for two keys at once (kr0, kr1), each with exactly its arithmetic (the same fmaf
// chain per key and head, in dimension order): the q values read from shared memory serve both keys
template <typename TK, int HH>
__device__ __forceinline__ void score_split_part2(const float* qs, const float* ws, const TK* kr0, const TK* kr1,
                                                  int d, int hg, bool vec, float& part0, float& part1) {
    constexpr int HG = HH / 4;
    float a0[HG], a1[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        a0[h] = 0.f;
        a1[h] = 0.f;
    }
    constexpr int kKB = 16;
    for (int c00 = 0; c00 < d; c00 += kKB) {
        float k0[kKB], k1[kKB];
        if (vec && sizeof(TK) == 4 && c00 + kKB <= d) {
#pragma unroll
            for (int u = 0; u < kKB / 4; ++u) {
                const float4 x = *reinterpret_cast<const float4*>(kr0 + c00 + 4 * u);
                const float4 y = *reinterpret_cast<const float4*>(kr1 + c00 + 4 * u);
                k0[4 * u] = x.x;
                k0[4 * u + 1] = x.y;
                k0[4 * u + 2] = x.z;
                k0[4 * u + 3] = x.w;
                k1[4 * u] = y.x;
                k1[4 * u + 1] = y.y;
                k1[4 * u + 2] = y.z;
                k1[4 * u + 3] = y.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < kKB; ++i) {
                k0[i] = (c00 + i < d) ? to_f32(kr0[c00 + i]) : 0.f;
                k1[i] = (c00 + i < d) ? to_f32(kr1[c00 + i]) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kKB; ++i) {
            if (c00 + i >= d) break;
            const float4* qc = reinterpret_cast<const float4*>(qs + (c00 + i) * HH + hg * HG);
#pragma unroll
            for (int h4 = 0; h4 < HG / 4; ++h4) {
                const float4 qq = qc[h4];
                a0[4 * h4] = fmaf(qq.x, k0[i], a0[4 * h4]);
                a0[4 * h4 + 1] = fmaf(qq.y, k0[i], a0[4 * h4 + 1]);
                a0[4 * h4 + 2] = fmaf(qq.z, k0[i], a0[4 * h4 + 2]);
                a0[4 * h4 + 3] = fmaf(qq.w, k0[i], a0[4 * h4 + 3]);
                a1[4 * h4] = fmaf(qq.x, k1[i], a1[4 * h4]);
                a1[4 * h4 + 1] = fmaf(qq.y, k1[i], a1[4 * h4 + 1]);
                a1[4 * h4 + 2] = fmaf(qq.z, k1[i], a1[4 * h4 + 2]);
                a1[4 * h4 + 3] = fmaf(qq.w, k1[i], a1[4 * h4 + 3]);
            }
        }
    }
    part0 = 0.f;
    part1 = 0.f;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        part0 = fmaf(ws[hg * HG + h], fmaxf(a0[h], 0.f), part0);
        part1 = fmaf(ws[hg * HG + h], fmaxf(a1[h], 0.f), part1);
    }
}

// the four partials of a key (lanes 4i..4i+3), added; every lane of the warp must call it
__device__ __forceinline__ float score_split_sum(float part) {
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    return part + 0.0f;   // (-0 -> +0)
}


// ---------------------------------------------------------------------------
// Block selection of one row with at most NT <= kRankMax complete blocks (the
// pooled keys of a decode step), by a CTA of NT threads (a power of two): the blocks are
// sorted in shared memory by the composite key (order key, then the complement
// of the block index), so that a larger composite is a better block and equal
// scores order the lower block first, with a bitonic network; the first K are
// kept and expanded in ascending block order to their C member positions, then
// the tail.  The same selection as select_row<true> (the lower block index wins
// ties, -0 == +0).  s: the row's n_vis / C block scores (global or shared).
// ---------------------------------------------------------------------------
constexpr int kRankMax = 1024;
constexpr int kRankThreads = 1024;

struct RankShared {
    uint64_t comp[kRankMax];
    uint32_t sel[kRankMax / 32];
    uint32_t pre[kRankMax / 32];
    int32_t blk[kRankMax];
};

template <int NT>
__device__ __forceinline__ void block_rank_row(const float* s, int n_vis, int top_k, int C, int32_t* out,
                                               int32_t* n_sel_r, RankShared& rs) {
    const int n = n_vis / C;
    const int K = min(top_k / C, n);
    const int cap = (top_k / C) * C + C - 1;
    const int tail0 = n * C;
    const int n_out = K * C + (n_vis - tail0);
    const int nw = (n + 31) >> 5;
    int n_pad = 2;
    while (n_pad < n) n_pad <<= 1;
    for (int i = threadIdx.x; i < n_pad; i += NT)
        rs.comp[i] = i < n ? ((uint64_t)order_key(s[i]) << 32) | (uint32_t)(0xffffffffu - (uint32_t)i) : 0ull;
    for (int i = threadIdx.x; i < nw; i += NT) rs.sel[i] = 0u;
    __syncthreads();
    if (K == n) {
        for (int i = threadIdx.x; i < n_vis; i += NT) out[i] = i;
    } else {
        if (K > 0) {
            // bitonic sort, descending, one element per thread: the pair (i, i ^ stride) of a run of
            // `size` keeps the larger value at the lower index when the run is an even one (the
            // smaller otherwise); partners closer than a warp trade by shuffles, farther ones
            // through shared memory
            const int i = threadIdx.x;
            uint64_t val = i < n_pad ? rs.comp[i] : 0ull;
            for (int size = 2; size <= n_pad; size <<= 1) {
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    uint64_t other;
                    if (stride >= 32) {
                        __syncthreads();
                        rs.comp[i] = val;
                        __syncthreads();
                        other = rs.comp[i ^ stride];
                    } else {
                        other = __shfl_xor_sync(0xffffffffu, val, stride);
                    }
                    const bool lower = (i & stride) == 0, down = (i & size) == 0;
                    val = (lower == down) ? (val > other ? val : other) : (val < other ? val : other);
                }
            }
            __syncthreads();
            rs.comp[i] = val;
            __syncthreads();
            for (int i = threadIdx.x; i < K; i += NT) {
                const int bidx = (int)(0xffffffffu - (uint32_t)rs.comp[i]);
                atomicOr(&rs.sel[bidx >> 5], 1u << (bidx & 31));
            }
            __syncthreads();
            if (threadIdx.x < 32) {   // exclusive prefix of selected blocks per 32-block word
                uint32_t carry = 0;
                for (int w0 = 0; w0 < nw; w0 += 32) {
                    const int w = w0 + threadIdx.x;
                    const uint32_t c = w < nw ? (uint32_t)__popc(rs.sel[w]) : 0u;
                    uint32_t x = c;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                        if ((int)threadIdx.x >= o) x += y;
                    }
                    if (w < nw) rs.pre[w] = carry + x - c;
                    carry += __shfl_sync(0xffffffffu, x, 31);
                }
            }
            __syncthreads();
            for (int b = threadIdx.x; b < n; b += NT) {
                const uint32_t word = rs.sel[b >> 5];
                if ((word >> (b & 31)) & 1u) rs.blk[rs.pre[b >> 5] + __popc(word & ((1u << (b & 31)) - 1u))] = b;
            }
            __syncthreads();
            for (int o = threadIdx.x; o < K * C; o += NT) out[o] = rs.blk[o / C] * C + o % C;
        }
        for (int i = threadIdx.x; i < n_vis - tail0; i += NT) out[K * C + i] = tail0 + i;
    }
    for (int i = n_out + threadIdx.x; i < cap; i += NT) out[i] = -1;
    if (n_sel_r && threadIdx.x == 0) *n_sel_r = n_out;
}

}  // namespace blk
}  // namespace lidx
