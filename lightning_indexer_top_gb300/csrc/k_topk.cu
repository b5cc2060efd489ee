// Per-row top-k selection of indexer scores, replacing a full argsort.
//
// Token mode: K = min(top_k, n_vis) positions with the largest scores, equal
// scores resolved toward the lower position ("ggml_top_k(min(top_k,
// n_tokens))", ik_llama.cpp PR #2058, commit "Add GLM-5.2/DeepSeek-V3.2 DSA
// lightning indexer").  Block mode: the same selection over complete-block
// scores with K = min(floor(top_k/C), n_cb), expanded to every member token,
// plus the incomplete tail (llama.cpp commit c88c916636, QSA commit message).
//
// One CTA per query row.
//   1. Each score becomes an order-preserving uint32 key (-0 folded onto +0).
//   2. Three radix rounds (11, 11, 10 bits, most significant first) build a
//      shared-memory histogram of the keys that still match the prefix found
//      so far and locate the bin holding the K-th largest key.  After the
//      third round the threshold key T is exact, and `need` = how many keys
//      equal to T are taken.
//   3. One ordered compaction pass writes, in ascending position order, every
//      position with key > T and the first `need` positions with key == T.
//      A block-wide scan of (count > T, count == T) per chunk gives each
//      thread its output offset, so equal scores go to the lower positions
//      deterministically.
// Rows with K == n_vis (every visible key kept, e.g. the first top_k rows of a
// causal prefill) skip the select and write 0..n_vis-1.
#include "lidx_internal.cuh"

namespace lidx {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 16;                 // consecutive positions per thread in one compaction chunk
constexpr int kChunk = kThreads * kPer;

struct Shared {
    uint32_t hist[2048];
    uint32_t warp_sums[kWarps];
    uint32_t sel_bin;
    uint32_t sel_above;
};

// exclusive prefix sum of v over the CTA; *total receives the CTA sum
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Shared& sh, uint32_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t s = lane < kWarps ? sh.warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) sh.warp_sums[lane] = s;
    }
    __syncthreads();
    const uint32_t before = wid > 0 ? sh.warp_sums[wid - 1] : 0u;
    *total = sh.warp_sums[kWarps - 1];
    __syncthreads();
    return before + x - v;
}

// One radix round over keys matching (prefix, mask): returns via shared memory
// the bin (of `bits` bits at `shift`) that holds the `need`-th largest key and
// the number of matching keys in higher bins.
__device__ __forceinline__ void radix_round(const float* __restrict__ s, int n, uint32_t prefix,
                                            uint32_t mask, int shift, int bits, uint32_t need,
                                            Shared& sh) {
    const int nbins = 1 << bits;
    for (int i = threadIdx.x; i < nbins; i += kThreads) sh.hist[i] = 0u;
    __syncthreads();
    // Scores crowd into few bins, so equal bins are combined across the warp
    // first (one shared-memory atomic per distinct bin per warp instruction).
    const int lane = threadIdx.x & 31;
    auto count = [&](uint32_t key, bool in) {
        const bool hit = in && (key & mask) == prefix;
        const uint32_t bin = hit ? (key >> shift) & (nbins - 1) : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (hit && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
    };
    if ((reinterpret_cast<uintptr_t>(s) & 15u) == 0) {
        const int n4 = n >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(s);
        // kBatch independent 16-byte loads in flight per thread before any is used
        constexpr int kBatch = 8;
        const int step = kThreads * kBatch;
        const int lim = (n4 + step - 1) / step * step;   // whole warps stay converged
        for (int i0 = threadIdx.x; i0 < lim; i0 += step) {
            float4 v[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = i0 + b * kThreads;
                v[b] = i < n4 ? s4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const bool in = i0 + b * kThreads < n4;
                count(order_key(v[b].x), in);
                count(order_key(v[b].y), in);
                count(order_key(v[b].z), in);
                count(order_key(v[b].w), in);
            }
        }
        if (threadIdx.x < 32) {   // the last n % 4 elements, by all lanes of warp 0
            const int j = (n4 << 2) + lane;
            const bool in = j < n;
            count(in ? order_key(s[j]) : 0u, in);
        }
    } else {
        const int lim = (n + kThreads - 1) / kThreads * kThreads;
        for (int j = threadIdx.x; j < lim; j += kThreads) {
            const bool in = j < n;
            count(in ? order_key(s[j]) : 0u, in);
        }
    }
    __syncthreads();
    // thread t owns nbins/kThreads consecutive bins, walked from the top
    const int per = nbins / kThreads;
    const int top = nbins - 1 - threadIdx.x * per;
    uint32_t local = 0;
    for (int i = 0; i < per; ++i) local += sh.hist[top - i];
    uint32_t tot;
    uint32_t c = block_excl_scan(local, sh, &tot);
    for (int i = 0; i < per; ++i) {
        const uint32_t h = sh.hist[top - i];
        if (c < need && need <= c + h) {
            sh.sel_bin = (uint32_t)(top - i);
            sh.sel_above = c;
        }
        c += h;
    }
    __syncthreads();
}

template <bool kBlocks>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ scores,
                                                        int64_t score_row_stride, Geom g, int top_k,
                                                        int C, int32_t* __restrict__ idx,
                                                        int64_t idx_row_stride,
                                                        int32_t* __restrict__ n_sel) {
    __shared__ Shared sh;
    const int64_t r = blockIdx.x;
    const int n_vis = row_n_vis(g, r);
    const float* s = scores + r * score_row_stride;
    int32_t* out = idx + r * idx_row_stride;

    // n = candidates (tokens or complete blocks), K = how many of them to take
    const int n = kBlocks ? n_vis / C : n_vis;
    const int K = kBlocks ? min(top_k / C, n) : min(top_k, n_vis);
    const int cap = kBlocks ? (top_k / C) * C + C - 1 : top_k;
    const int tail0 = kBlocks ? n * C : n_vis;  // first tail token (block mode)
    const int n_out = kBlocks ? K * C + (n_vis - tail0) : K;

    if (K == n) {
        // every candidate kept: the selection is all visible positions
        for (int i = threadIdx.x; i < n_vis; i += kThreads) out[i] = i;
    } else if (K > 0) {
        uint32_t prefix = 0u, mask = 0u, need = (uint32_t)K;
        const int shifts[3] = {21, 10, 0};
        const int bitsv[3] = {11, 11, 10};
#pragma unroll 1
        for (int round = 0; round < 3; ++round) {
            radix_round(s, n, prefix, mask, shifts[round], bitsv[round], need, sh);
            const uint32_t bin = sh.sel_bin, above = sh.sel_above;
            need -= above;
            prefix |= bin << shifts[round];
            mask |= ((1u << bitsv[round]) - 1u) << shifts[round];
            __syncthreads();
        }
        const uint32_t T = prefix;
        const bool aligned = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;

        uint32_t run_gt = 0, run_eq = 0;
#pragma unroll 1
        for (int base = 0; base < n; base += kChunk) {
            const int p0 = base + threadIdx.x * kPer;
            uint32_t key[kPer];
            uint32_t gt = 0, eq = 0;
            if (aligned && p0 + kPer <= n) {
                const float4* s4 = reinterpret_cast<const float4*>(s + p0);
                float4 v[kPer / 4];
#pragma unroll
                for (int q4 = 0; q4 < kPer / 4; ++q4) v[q4] = s4[q4];
#pragma unroll
                for (int q4 = 0; q4 < kPer / 4; ++q4) {
                    key[4 * q4] = order_key(v[q4].x);
                    key[4 * q4 + 1] = order_key(v[q4].y);
                    key[4 * q4 + 2] = order_key(v[q4].z);
                    key[4 * q4 + 3] = order_key(v[q4].w);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kPer; ++i) key[i] = (p0 + i < n) ? order_key(s[p0 + i]) : 0u;
            }
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const bool valid = p0 + i < n;
                gt += (valid && key[i] > T);
                eq += (valid && key[i] == T);
            }
            uint32_t tot;
            const uint32_t ex = block_excl_scan((eq << 16) | gt, sh, &tot);
            uint32_t eq_before = run_eq + (ex >> 16);
            uint32_t off = run_gt + (ex & 0xffffu) + min(eq_before, need);
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                if (p0 + i >= n) break;
                bool take = false;
                if (key[i] > T) {
                    take = true;
                } else if (key[i] == T) {
                    take = eq_before < need;
                    ++eq_before;
                }
                if (take) {
                    if (kBlocks) {
                        for (int c = 0; c < C; ++c) out[off * C + c] = (p0 + i) * C + c;
                    } else {
                        out[off] = p0 + i;
                    }
                    ++off;
                }
            }
            run_gt += tot & 0xffffu;
            run_eq += tot >> 16;
        }
        if (kBlocks) {
            for (int i = threadIdx.x; i < n_vis - tail0; i += kThreads) out[K * C + i] = tail0 + i;
        }
    } else if (kBlocks) {
        // no whole block fits the budget: the tail alone
        for (int i = threadIdx.x; i < n_vis - tail0; i += kThreads) out[i] = tail0 + i;
    }
    for (int i = n_out + threadIdx.x; i < cap; i += kThreads) out[i] = -1;
    if (n_sel && threadIdx.x == 0) n_sel[r] = n_out;
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t score_row_stride, const Geom& g, int top_k,
                        int block_size, int32_t* idx, int64_t idx_row_stride, int32_t* n_sel,
                        cudaStream_t st) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0) return cudaSuccess;
    if (block_size > 1)
        topk_kernel<true><<<(unsigned)n_rows, kThreads, 0, st>>>(scores, score_row_stride, g, top_k,
                                                                 block_size, idx, idx_row_stride,
                                                                 n_sel);
    else
        topk_kernel<false><<<(unsigned)n_rows, kThreads, 0, st>>>(scores, score_row_stride, g, top_k,
                                                                  1, idx, idx_row_stride, n_sel);
    return cudaGetLastError();
}

}  // namespace lidx
