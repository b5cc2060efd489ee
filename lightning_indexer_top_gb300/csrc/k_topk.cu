// Per-row top-k selection of indexer scores, replacing a full argsort.
//
// Token mode: K = min(top_k, n_vis) positions with the largest scores, equal
// scores resolved toward the lower position ("ggml_top_k(min(top_k,
// n_tokens))", ik_llama.cpp PR #2058, commit "Add GLM-5.2/DeepSeek-V3.2 DSA
// lightning indexer").  Block mode: the same selection over complete-block
// scores with K = min(floor(top_k/C), n_cb), expanded to every member token,
// plus the incomplete tail (llama.cpp commit c88c916636, QSA commit message).
//
// One CTA per query row.  Token-mode rows of up to 262144 keys take the
// bitmap path below (one pass over the scores after the histogram); other
// rows take the general radix path:
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
#include "block_ops.cuh"
#include "select_row.cuh"

namespace lidx {
namespace {

constexpr int kThreads = 512;            // general kernel (block mode)
constexpr int kPer = 16;                 // consecutive positions per thread in one compaction chunk

template <int NT>
struct GenShared {
    uint32_t hist[2048];
    uint32_t warp_sums[NT / 32];
    uint32_t sel_bin;
    uint32_t sel_above;
};

// exclusive prefix sum of v over the CTA; *total receives the CTA sum
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, GenShared<NT>& sh, uint32_t* total) {
    constexpr int NW = NT / 32;
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
        uint32_t s = lane < NW ? sh.warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < NW) sh.warp_sums[lane] = s;
    }
    __syncthreads();
    const uint32_t before = wid > 0 ? sh.warp_sums[wid - 1] : 0u;
    *total = sh.warp_sums[NW - 1];
    __syncthreads();
    return before + x - v;
}

// One radix round over keys matching (prefix, mask): returns via shared memory
// the bin (of `bits` bits at `shift`) that holds the `need`-th largest key and
// the number of matching keys in higher bins.
template <int NT>
__device__ __forceinline__ void radix_round(const float* s, int n, uint32_t prefix,
                                            uint32_t mask, int shift, int bits, uint32_t need,
                                            GenShared<NT>& sh) {
    const int nbins = 1 << bits;
    for (int i = threadIdx.x; i < nbins; i += NT) sh.hist[i] = 0u;
    __syncthreads();
    // Scores crowd into few bins, so equal bins are combined across the warp
    // first (one shared-memory atomic per distinct bin per warp instruction);
    // warps without a matching key skip the combine.
    const int lane = threadIdx.x & 31;
    auto count = [&](uint32_t key, bool in) {
        const bool hit = in && (key & mask) == prefix;
        if (__ballot_sync(0xffffffffu, hit) == 0u) return;
        const uint32_t bin = hit ? (key >> shift) & (nbins - 1) : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (hit && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
    };
    if ((reinterpret_cast<uintptr_t>(s) & 15u) == 0) {
        const int n4 = n >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(s);
        // kBatch independent 16-byte loads in flight per thread before any is used
        constexpr int kBatch = 8;
        const int step = NT * kBatch;
        const int lim = (n4 + step - 1) / step * step;   // whole warps stay converged
        for (int i0 = threadIdx.x; i0 < lim; i0 += step) {
            float4 v[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = i0 + b * NT;
                v[b] = i < n4 ? s4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const bool in = i0 + b * NT < n4;
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
        const int lim = (n + NT - 1) / NT * NT;
        for (int j = threadIdx.x; j < lim; j += NT) {
            const bool in = j < n;
            count(in ? order_key(s[j]) : 0u, in);
        }
    }
    __syncthreads();
    // thread t owns nbins/NT consecutive bins (or one, or none), walked from the top
    const int per = nbins / NT > 0 ? nbins / NT : 1;
    const bool owner = threadIdx.x * per < nbins;
    const int top = nbins - 1 - threadIdx.x * per;
    uint32_t local = 0;
    if (owner)
        for (int i = 0; i < per; ++i) local += sh.hist[top - i];
    uint32_t tot;
    uint32_t c = block_excl_scan(local, sh, &tot);
    if (owner) {
        for (int i = 0; i < per; ++i) {
            const uint32_t h = sh.hist[top - i];
            if (c < need && need <= c + h) {
                sh.sel_bin = (uint32_t)(top - i);
                sh.sel_above = c;
            }
            c += h;
        }
    }
    __syncthreads();
}

// The general selection of one row by a CTA of NT threads.
template <bool kBlocks, int NT>
__device__ __forceinline__ void select_row(const float* s, int n_vis, int top_k, int C,
                                           int32_t* out, int32_t* n_sel_row, GenShared<NT>& sh) {
    constexpr int kChunk = NT * kPer;
    // n = candidates (tokens or complete blocks), K = how many of them to take
    const int n = kBlocks ? n_vis / C : n_vis;
    const int K = kBlocks ? min(top_k / C, n) : min(top_k, n_vis);
    const int cap = kBlocks ? (top_k / C) * C + C - 1 : top_k;
    const int tail0 = kBlocks ? n * C : n_vis;  // first tail token (block mode)
    const int n_out = kBlocks ? K * C + (n_vis - tail0) : K;

    if (K == n) {
        // every candidate kept: the selection is all visible positions
        for (int i = threadIdx.x; i < n_vis; i += NT) out[i] = i;
    } else if (K > 0) {
        uint32_t prefix = 0u, mask = 0u, need = (uint32_t)K;
        const int shifts[3] = {21, 10, 0};
        const int bitsv[3] = {11, 11, 10};
#pragma unroll 1
        for (int round = 0; round < 3; ++round) {
            radix_round<NT>(s, n, prefix, mask, shifts[round], bitsv[round], need, sh);
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
            for (int i = threadIdx.x; i < n_vis - tail0; i += NT) out[K * C + i] = tail0 + i;
        }
    } else if (kBlocks) {
        // no whole block fits the budget: the tail alone
        for (int i = threadIdx.x; i < n_vis - tail0; i += NT) out[i] = tail0 + i;
    }
    for (int i = n_out + threadIdx.x; i < cap; i += NT) out[i] = -1;
    if (n_sel_row && threadIdx.x == 0) *n_sel_row = n_out;
}

template <bool kBlocks>
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* scores,
                                                        int64_t score_row_stride, Geom g, int top_k,
                                                        int C, int32_t* idx,
                                                        int64_t idx_row_stride,
                                                        int32_t* n_sel) {
    __shared__ GenShared<kThreads> sh;
    const int64_t r = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    select_row<kBlocks, kThreads>(scores + r * score_row_stride, row_n_vis(g, r), top_k, C,
                                  idx + r * idx_row_stride, n_sel ? n_sel + r : nullptr, sh);
}

// Block mode with at most blk::kRankMax complete blocks per row: one CTA per row (blk::block_rank_row).
__global__ void __launch_bounds__(blk::kRankThreads) topk_block_rank_kernel(const float* scores,
                                                                           int64_t score_row_stride, Geom g,
                                                                           int top_k, int C, int32_t* idx,
                                                                           int64_t idx_row_stride, int32_t* n_sel) {
    __shared__ blk::RankShared rs;
    const int64_t r = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    blk::block_rank_row<blk::kRankThreads>(scores + r * score_row_stride, row_n_vis(g, r), top_k, C, idx + r * idx_row_stride,
                        n_sel ? n_sel + r : nullptr, rs);
}

// ---------------------------------------------------------------------------
// Token-mode selection for rows of up to kMapMax candidates, touching the
// scores in one pass after the histogram:
//   1. histogram of the top 11 key bits -> the bin B1 holding the K-th
//      largest key and the count of keys in higher bins;
//   2. one pass over the row: every key in a bin above B1 is selected (a bit
//      in a shared-memory position bitmap), every key in bin B1 is a candidate
//      (key, position) appended to a shared-memory list;
//   3. two radix rounds (11 and 10 bits) over the candidates in shared memory
//      give the exact threshold key T and how many keys equal to T are taken;
//      candidates above T are marked selected, those equal to T in a second
//      bitmap;
//   4. a block-wide scan over the bitmap words writes the selected positions
//      in ascending order, taking the lowest-position keys equal to T.
// If the candidates overflow the list the row is handed back to the general
// kernel.
// ---------------------------------------------------------------------------
constexpr int kMapThreads = 1024;
constexpr int kMapWarps = kMapThreads / 32;
constexpr int kMapMax = 262144;                 // positions covered by the bitmaps
constexpr int kCandCap = 8192;
constexpr int kMapWords = kMapMax / 32;

struct MapShared {
    uint32_t hist[2048];
    uint32_t sel[kMapWords];
    uint32_t eq[kMapWords];
    uint32_t cand_key[kCandCap];
    int32_t cand_pos[kCandCap];
    uint32_t warp_a[kMapWarps];
    uint32_t warp_b[kMapWarps];
    uint32_t cand_n;
    uint32_t bin, above;
    int overflow;
    uint32_t total;
};

// exclusive prefix sums of (a, b) over the CTA
__device__ __forceinline__ void map_scan2(uint32_t a, uint32_t b, MapShared& sh, uint32_t* ea, uint32_t* eb,
                                          uint32_t* ta, uint32_t* tb) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = a, y = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t xa = __shfl_up_sync(0xffffffffu, x, o);
        const uint32_t yb = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) {
            x += xa;
            y += yb;
        }
    }
    if (lane == 31) {
        sh.warp_a[wid] = x;
        sh.warp_b[wid] = y;
    }
    __syncthreads();
    if (wid == 0) {
        uint32_t u = sh.warp_a[lane], v = sh.warp_b[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t ua = __shfl_up_sync(0xffffffffu, u, o);
            const uint32_t vb = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) {
                u += ua;
                v += vb;
            }
        }
        sh.warp_a[lane] = u;
        sh.warp_b[lane] = v;
    }
    __syncthreads();
    *ea = (wid > 0 ? sh.warp_a[wid - 1] : 0u) + x - a;
    *eb = (wid > 0 ? sh.warp_b[wid - 1] : 0u) + y - b;
    *ta = sh.warp_a[kMapWarps - 1];
    *tb = sh.warp_b[kMapWarps - 1];
    __syncthreads();
}

// bin (of `bits` bits at `shift`) holding the need-th largest of the counted
// keys, and the count in higher bins; the histogram is in sh.hist
__device__ __forceinline__ void map_find_bin(int nbins, uint32_t need, MapShared& sh) {
    const int per = nbins / kMapThreads > 0 ? nbins / kMapThreads : 1;
    const bool owner = threadIdx.x * per < nbins;
    const int top = nbins - 1 - threadIdx.x * per;
    uint32_t local = 0;
    if (owner)
        for (int i = 0; i < per; ++i) local += sh.hist[top - i];
    uint32_t c, dummy, ta, tb;
    map_scan2(local, 0u, sh, &c, &dummy, &ta, &tb);
    if (owner) {
        for (int i = 0; i < per; ++i) {
            const uint32_t h = sh.hist[top - i];
            if (c < need && need <= c + h) {
                sh.bin = (uint32_t)(top - i);
                sh.above = c;
            }
            c += h;
        }
    }
    __syncthreads();
}

// histogram of the candidate keys matching (prefix, mask) at (shift, bits)
__device__ __forceinline__ void map_cand_hist(MapShared& sh, uint32_t n_cand, uint32_t prefix, uint32_t mask,
                                              int shift, int bits) {
    const int nbins = 1 << bits;
    for (int i = threadIdx.x; i < nbins; i += kMapThreads) sh.hist[i] = 0u;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < n_cand; i += kMapThreads) {
        const uint32_t key = sh.cand_key[i];
        if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & (nbins - 1)], 1u);
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kMapThreads, 1) topk_map_kernel(const float* scores,
                                                                  int64_t score_row_stride, Geom g, int top_k,
                                                                  int32_t* idx, int64_t idx_row_stride,
                                                                  int32_t* n_sel, const uint32_t* hist) {
    extern __shared__ __align__(16) unsigned char map_raw[];
    MapShared& sh = *reinterpret_cast<MapShared*>(map_raw);
    pdl_trigger();
    pdl_wait();
    const int64_t r = blockIdx.x;
    const int n = row_n_vis(g, r);
    const int K = min(top_k, n);
    const float* s = scores + r * score_row_stride;
    int32_t* out = idx + r * idx_row_stride;
    const int lane = threadIdx.x & 31;

    GenShared<kMapThreads>& gsh = *reinterpret_cast<GenShared<kMapThreads>*>(map_raw);
    if (K == n || n > kMapMax) {
        // dense rows and rows longer than the bitmaps take the general path
        select_row<false, kMapThreads>(s, n, top_k, 1, out, n_sel ? n_sel + r : nullptr, gsh);
        return;
    }
    const int nwords = (n + 31) >> 5;
    for (int i = threadIdx.x; i < nwords; i += kMapThreads) {
        sh.sel[i] = 0u;
        sh.eq[i] = 0u;
    }
    // the fused path brings the row's histogram from the scorer (pass 1 is then skipped, unless the
    // histogram is not exact: its total must be the row's key count)
    uint32_t hpart = 0;
    for (int i = threadIdx.x; i < 2048; i += kMapThreads) {
        const uint32_t v = hist ? hist[r * 2048 + i] : 0u;
        sh.hist[i] = v;
        hpart += v;
    }
    if (threadIdx.x == 0) {
        sh.cand_n = 0u;
        sh.overflow = 0;
        sh.total = 0u;
    }
    __syncthreads();
    if (hist) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) hpart += __shfl_xor_sync(0xffffffffu, hpart, o);
        if (lane == 0 && hpart) atomicAdd(&sh.total, hpart);
        __syncthreads();
    }
    const bool have_hist = hist && sh.total == (uint32_t)n;
    if (hist && !have_hist) {
        for (int i = threadIdx.x; i < 2048; i += kMapThreads) sh.hist[i] = 0u;
        __syncthreads();
    }

    const bool vec = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
    const int n4 = vec ? n >> 2 : 0;
    const float4* s4 = reinterpret_cast<const float4*>(s);
    constexpr int kBatch = 4;
    const int step = kMapThreads * kBatch;
    const int lim = (n4 + step - 1) / step * step;

    // 1. histogram of the top 11 bits (equal bins combined across the warp)
    auto hcount = [&](uint32_t key, bool in) {
        const uint32_t bin = in ? key >> 21 : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
    };
    for (int i0 = threadIdx.x; !have_hist && i0 < lim; i0 += step) {
        float4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * kMapThreads;
            v[b] = i < n4 ? s4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const bool in = i0 + b * kMapThreads < n4;
            hcount(order_key(v[b].x), in);
            hcount(order_key(v[b].y), in);
            hcount(order_key(v[b].z), in);
            hcount(order_key(v[b].w), in);
        }
    }
    for (int j0 = (n4 << 2); !have_hist && j0 < n; j0 += kMapThreads) {   // the unaligned rest, whole warps
        const int j = j0 + threadIdx.x;
        const bool in = j < n;
        hcount(in ? order_key(s[j]) : 0u, in);
    }
    __syncthreads();
    map_find_bin(2048, (uint32_t)K, sh);
    const uint32_t B1 = sh.bin;
    uint32_t need = (uint32_t)K - sh.above;

    // 2. mark keys above bin B1, collect the candidates of bin B1
    auto mark = [&](uint32_t key, int p, bool in) {
        const uint32_t bin = key >> 21;
        if (in && bin > B1) atomicOr(&sh.sel[p >> 5], 1u << (p & 31));
        const bool cand = in && bin == B1;
        const uint32_t m = __ballot_sync(0xffffffffu, cand);
        if (m) {
            uint32_t base = 0;
            if (lane == __ffs(m) - 1) base = atomicAdd(&sh.cand_n, (uint32_t)__popc(m));
            base = __shfl_sync(0xffffffffu, base, __ffs(m) - 1);
            if (cand) {
                const uint32_t slot = base + __popc(m & ((1u << lane) - 1u));
                if (slot < (uint32_t)kCandCap) {
                    sh.cand_key[slot] = key;
                    sh.cand_pos[slot] = p;
                }
            }
        }
    };
    for (int i0 = threadIdx.x; i0 < lim; i0 += step) {
        float4 v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * kMapThreads;
            v[b] = i < n4 ? s4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = i0 + b * kMapThreads;
            const bool in = i < n4;
            mark(order_key(v[b].x), 4 * i, in);
            mark(order_key(v[b].y), 4 * i + 1, in);
            mark(order_key(v[b].z), 4 * i + 2, in);
            mark(order_key(v[b].w), 4 * i + 3, in);
        }
    }
    for (int j0 = (n4 << 2); j0 < n; j0 += kMapThreads) {
        const int j = j0 + threadIdx.x;
        const bool in = j < n;
        mark(in ? order_key(s[j]) : 0u, j, in);
    }
    __syncthreads();
    const uint32_t n_cand = sh.cand_n;
    if (n_cand > (uint32_t)kCandCap) {
        // too many keys in the threshold bin (e.g. mass ties): the general path
        select_row<false, kMapThreads>(s, n, top_k, 1, out, n_sel ? n_sel + r : nullptr, gsh);
        return;
    }

    // 3. exact threshold among the candidates
    uint32_t prefix = B1 << 21, mask = 0xffe00000u;
    map_cand_hist(sh, n_cand, prefix, mask, 10, 11);
    map_find_bin(2048, need, sh);
    prefix |= sh.bin << 10;
    mask |= 0x7ffu << 10;
    need -= sh.above;
    map_cand_hist(sh, n_cand, prefix, mask, 0, 10);
    map_find_bin(1024, need, sh);
    need -= sh.above;
    const uint32_t T = prefix | sh.bin;
    for (uint32_t i = threadIdx.x; i < n_cand; i += kMapThreads) {
        const uint32_t key = sh.cand_key[i];
        const int p = sh.cand_pos[i];
        if (key > T) atomicOr(&sh.sel[p >> 5], 1u << (p & 31));
        else if (key == T) atomicOr(&sh.eq[p >> 5], 1u << (p & 31));
    }
    __syncthreads();

    // 4. ordered write-out: thread t owns consecutive bitmap words
    const int wpt = (nwords + kMapThreads - 1) / kMapThreads;
    const int w0 = threadIdx.x * wpt;
    uint32_t cs = 0, ce = 0;
    for (int w = w0; w < min(w0 + wpt, nwords); ++w) {
        cs += __popc(sh.sel[w]);
        ce += __popc(sh.eq[w]);
    }
    uint32_t bs, be, ts, te;
    map_scan2(cs, ce, sh, &bs, &be, &ts, &te);
    uint32_t off = bs + min(be, need);
    uint32_t eq_rank = be;
    for (int w = w0; w < min(w0 + wpt, nwords); ++w) {
        uint32_t a = sh.sel[w], e = sh.eq[w];
        uint32_t any = a | e;
        while (any) {
            const int bit = __ffs(any) - 1;
            any &= any - 1;
            const uint32_t m = 1u << bit;
            bool take = (a & m) != 0;
            if (!take) {
                take = eq_rank < need;
                ++eq_rank;
            }
            if (take) out[off++] = w * 32 + bit;
        }
    }
    for (int i = K + threadIdx.x; i < top_k; i += kMapThreads) out[i] = -1;
    if (threadIdx.x == 0 && n_sel) n_sel[r] = K;
}

// ---------------------------------------------------------------------------
// Multi-CTA selection for few long rows (decode), with a caller workspace:
//   A. one CTA per row histograms a sample of the row (64 blocks of 128
//      scores spread over it) and picks a lower bound L on the order key
//      with about twice K keys expected at or above it;
//   B. (row, chunk) CTAs collect every key >= L of their chunk (key and
//      position) in shared memory and append them to the row's candidate
//      list with one global reservation per CTA;
//   C. one CTA per row takes the exact top K of the candidates (three radix
//      rounds over the full keys in shared memory), marks them in a position
//      bitmap and writes them in ascending order, ties at the threshold going
//      to the lowest positions.
// The result is exactly that of the one-CTA kernels: the sample only decides
// how much is filtered.  If the bound let fewer than K keys or more than the
// list holds through, kernel C does the row with the general path.
// ---------------------------------------------------------------------------
constexpr int kMcThreads = 256;
constexpr int kMcChunk = 8192;              // scores per (row, chunk) CTA
constexpr int kMcCandCap = kCandCap;        // candidates kept per row
constexpr int kMcLocal = 1024;              // candidates a chunk CTA buffers before flushing
constexpr int kSampleBlocks = 64, kSampleLen = 128;

struct McLayout {
    uint32_t* bound;    // [rows]: lower bound L on the order key
    uint32_t* cnt;      // [rows]: candidates appended
    uint64_t* cand;     // [rows][kMcCandCap]: key << 32 | position
};

__host__ __device__ inline size_t mc_bytes(int64_t rows) {
    return (size_t)rows * ((size_t)kMcCandCap * 8 + 8) + 256;
}

__host__ __device__ inline McLayout mc_layout(void* ws, int64_t rows) {
    McLayout L;
    char* p = static_cast<char*>(ws);
    L.cand = reinterpret_cast<uint64_t*>(p);
    p += (size_t)rows * kMcCandCap * 8;
    L.bound = reinterpret_cast<uint32_t*>(p);
    p += (size_t)rows * 4;
    L.cnt = reinterpret_cast<uint32_t*>(p);
    return L;
}

// threshold bin of row r from its histogram: bin holding the K-th largest key
__device__ __forceinline__ void mc_find_bin(const uint32_t* h, uint32_t K, uint32_t* bin_out,
                                            uint32_t* above_out, uint32_t* scratch) {
    // thread t owns bins [2047 - 8t - 7, 2047 - 8t], walked from the top
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int top = 2047 - threadIdx.x * 8;
    uint32_t local = 0;
    for (int i = 0; i < 8; ++i) local += h[top - i];
    uint32_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[wid] = x;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < wid; ++w) before += scratch[w];
    uint32_t c = before + x - local;
    for (int i = 0; i < 8; ++i) {
        const uint32_t hh = h[top - i];
        if (c < K && K <= c + hh) {
            *bin_out = (uint32_t)(top - i);
            *above_out = c;
        }
        c += hh;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kMcThreads) topk_mc_bound_kernel(const float* scores,
                                                                   int64_t score_row_stride, Geom g, int top_k,
                                                                   McLayout L) {
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t scratch[kMcThreads / 32];
    __shared__ uint32_t sb[2];
    pdl_trigger();
    pdl_wait();
    const int64_t r = blockIdx.x;
    const int n = row_n_vis(g, r);
    const int K = min(top_k, n);
    if (threadIdx.x == 0) L.cnt[r] = 0u;
    if (K == n) return;
    for (int i = threadIdx.x; i < 2048; i += kMcThreads) hist[i] = 0u;
    __syncthreads();
    const float* s = scores + r * score_row_stride;
    // sample: kSampleBlocks blocks of kSampleLen consecutive scores, evenly spread;
    // each thread loads all of its sample keys at once (one memory round trip) and
    // keeps them for the refinement pass
    constexpr int kPerThread = kSampleBlocks * kSampleLen / kMcThreads;   // 32
    const int64_t span = n - kSampleLen;
    uint32_t keys[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int i = threadIdx.x + k * kMcThreads;
        const int blk = i / kSampleLen, off = i % kSampleLen;
        int p = (int)(span * blk / (kSampleBlocks - 1)) + off;
        p = p < 0 ? 0 : (p >= n ? n - 1 : p);   // rows shorter than one sample block
        keys[k] = order_key(s[p]);
    }
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) atomicAdd(&hist[keys[k] >> 21], 1u);
    __syncthreads();
    // expected keys per sample above the threshold: K * samples / n; aim for twice that
    const int64_t est = ((int64_t)2 * K * kSampleBlocks * kSampleLen + n - 1) / n + 1;
    const uint32_t want = (uint32_t)(est < kSampleBlocks * kSampleLen ? est : kSampleBlocks * kSampleLen);
    mc_find_bin(hist, want, &sb[0], &sb[1], scratch);
    // refine inside that bin with the next 11 bits, so L cuts close to the wanted count
    const uint32_t b1 = sb[0], need2 = want - sb[1];
    for (int i = threadIdx.x; i < 2048; i += kMcThreads) hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPerThread; ++k)
        if ((keys[k] >> 21) == b1) atomicAdd(&hist[(keys[k] >> 10) & 2047u], 1u);
    __syncthreads();
    mc_find_bin(hist, need2, &sb[0], &sb[1], scratch);
    if (threadIdx.x == 0) L.bound[r] = (b1 << 21) | (sb[0] << 10);
}

// append every position j in [c0, c1) of row r whose order key is >= lo to the row's candidate
// list (key << 32 | position): warp-aggregated slots in a shared buffer, one global reservation
// per CTA for the buffer, straight to the list when the buffer is full
__device__ __forceinline__ void mc_filter_range(const float* s, int c0, int c1, uint32_t lo,
                                                const McLayout& L, int64_t r, uint64_t* buf, uint32_t& nbuf,
                                                uint32_t& base) {
    if (threadIdx.x == 0) nbuf = 0u;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    uint32_t* cnt = L.cnt + r;
    uint64_t* cand = L.cand + r * (int64_t)kMcCandCap;
    for (int j0 = c0; j0 < c1; j0 += kMcThreads * 8) {
        float v[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int j = j0 + b * kMcThreads + threadIdx.x;
            v[b] = j < c1 ? s[j] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int j = j0 + b * kMcThreads + threadIdx.x;
            const uint32_t key = order_key(v[b]);
            const bool hit = j < c1 && key >= lo;
            const uint32_t m = __ballot_sync(0xffffffffu, hit);
            if (m) {
                uint32_t at = 0;
                if (lane == __ffs(m) - 1) at = atomicAdd(&nbuf, (uint32_t)__popc(m));
                at = __shfl_sync(0xffffffffu, at, __ffs(m) - 1) + __popc(m & ((1u << lane) - 1u));
                if (hit) {
                    const uint64_t kp = ((uint64_t)key << 32) | (uint32_t)j;
                    if (at < (uint32_t)kMcLocal) {
                        buf[at] = kp;
                    } else {   // local buffer full: straight to the row's list
                        const uint32_t slot = atomicAdd(cnt, 1u);
                        if (slot < (uint32_t)kMcCandCap) cand[slot] = kp;
                    }
                }
            }
        }
    }
    __syncthreads();
    const uint32_t nb = min(nbuf, (uint32_t)kMcLocal);
    if (threadIdx.x == 0) base = nb ? atomicAdd(cnt, nb) : 0u;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < nb; i += kMcThreads)
        if (base + i < (uint32_t)kMcCandCap) cand[base + i] = buf[i];
}

__global__ void __launch_bounds__(kMcThreads) topk_mc_filter_kernel(const float* scores,
                                                                    int64_t score_row_stride, Geom g, int top_k,
                                                                    McLayout L) {
    __shared__ uint64_t buf[kMcLocal];
    __shared__ uint32_t nbuf, base;
    pdl_trigger();
    pdl_wait();
    const int64_t r = blockIdx.y;
    const int n = row_n_vis(g, r);
    const int K = min(top_k, n);
    const int c0 = blockIdx.x * kMcChunk;
    if (K == n || c0 >= n) return;
    mc_filter_range(scores + r * score_row_stride, c0, min(n, c0 + kMcChunk), L.bound[r], L, r, buf, nbuf, base);
}

// Fused path: the scorer counted each row's order keys by their top 11 bits; each filter CTA derives
// from that exact histogram the bin b* holding the K-th largest key, with the count above it
// (L.bound[r] = b* << 21 | above, recorded by the row's first CTA for the finish kernel).  Every key in a higher bin is selected and only the keys of b*
// remain to be ranked, so the filter keeps the keys with bin >= b* (above + hist[b*] of them) and
// the finish kernel resolves b*.  A bound of ~0 (the histogram was not exact: its launch could not
// count, see the scorer) makes every key a candidate; the list overflows and the finish takes the
// general path.
// the bound of row r from its histogram (as topk_hist_bound computes it) to every thread of a
// kMcThreads CTA: thread t owns bins [2047 - 8t - 7, 2047 - 8t]
__device__ __forceinline__ uint32_t hist_bound(const uint32_t* hrow, int n, int K, uint32_t* scratch, uint32_t* sb) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const uint4* h4 = reinterpret_cast<const uint4*>(hrow + 2040 - 8 * threadIdx.x);
    const uint4 lo4 = h4[0], hi4 = h4[1];
    const uint32_t bins[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};   // from the top
    uint32_t local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) local += bins[i];
    uint32_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[wid] = x;
    if (threadIdx.x == 0) *sb = 0xffffffffu;
    __syncthreads();
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kMcThreads / 32; ++w) {
        before += w < wid ? scratch[w] : 0u;
        total += scratch[w];
    }
    uint32_t c = before + x - local;
    if (total == (uint32_t)n) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (c < (uint32_t)K && (uint32_t)K <= c + bins[i]) *sb = ((uint32_t)(2047 - 8 * threadIdx.x - i) << 21) | c;
            c += bins[i];
        }
    }
    __syncthreads();
    return *sb;
}

// (at most 40 registers: six CTAs per SM, so a batch's 1024 chunk CTAs take fewer waves)
__global__ void __launch_bounds__(kMcThreads, 6) topk_hist_filter_kernel(const float* scores,
                                                                      int64_t score_row_stride,
                                                                      const uint32_t* hist, Geom g, int top_k,
                                                                      McLayout L, int chunk) {
    __shared__ uint64_t buf[kMcLocal];
    __shared__ uint32_t nbuf, base;
    __shared__ uint32_t scratch[kMcThreads / 32], sbound;
    pdl_trigger();
    pdl_wait();
    const int64_t r = blockIdx.y;
    const int n = row_n_vis(g, r);
    const int K = min(top_k, n);
    const int c0 = blockIdx.x * chunk;
    if (K == n || c0 >= n) return;
    const float* s = scores + r * score_row_stride;
    const int c1 = min(n, c0 + chunk);
    const bool aligned = ((reinterpret_cast<uintptr_t>(s) | (uint32_t)c0) & 15u) == 0;
    // the first pass's 16-byte loads are issued before the row's bound is derived from its histogram
    // (every CTA of the row derives it; the first records it for the finish kernel)
    constexpr int kV = 4;                     // float4s per thread per pass
    float4 v[kV];
    if (aligned) {
#pragma unroll
        for (int b = 0; b < kV; ++b) {
            const int j = c0 + (b * kMcThreads + threadIdx.x) * 4;
            v[b] = j + 3 < c1 ? *reinterpret_cast<const float4*>(s + j)
                              : make_float4(j < c1 ? s[j] : 0.f, j + 1 < c1 ? s[j + 1] : 0.f,
                                            j + 2 < c1 ? s[j + 2] : 0.f, 0.f);
        }
    }
    if (threadIdx.x == 0) nbuf = 0u;
    const uint32_t b = hist_bound(hist + r * 2048, n, K, scratch, &sbound);   // (synchronises)
    if (blockIdx.x == 0 && threadIdx.x == 0) L.bound[r] = b;
    const uint32_t lo = b == 0xffffffffu ? 0u : (b & 0xffe00000u);
    if (!aligned) {
        mc_filter_range(s, c0, c1, lo, L, r, buf, nbuf, base);
        return;
    }
    // 16-byte loads: thread t takes the float4s t, t + 256, ... of the chunk, all issued at once; each
    // thread marks its hits in a bit mask, one warp scan places them, one shared atomic per warp
    const int lane = threadIdx.x & 31;
    uint32_t* cnt = L.cnt + r;
    uint64_t* cand = L.cand + r * (int64_t)kMcCandCap;
    for (int j0 = c0; j0 < c1; j0 += kMcThreads * 4 * kV) {
        if (j0 > c0) {
#pragma unroll
            for (int b = 0; b < kV; ++b) {
                const int j = j0 + (b * kMcThreads + threadIdx.x) * 4;
                v[b] = j + 3 < c1 ? *reinterpret_cast<const float4*>(s + j)
                                  : make_float4(j < c1 ? s[j] : 0.f, j + 1 < c1 ? s[j + 1] : 0.f,
                                                j + 2 < c1 ? s[j + 2] : 0.f, 0.f);
            }
        }
        uint32_t keys[4 * kV];
        uint32_t hits = 0;
#pragma unroll
        for (int b = 0; b < kV; ++b) {
            const float e[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = j0 + (b * kMcThreads + threadIdx.x) * 4 + q;
                keys[4 * b + q] = order_key(e[q]);
                hits |= (uint32_t)(j < c1 && keys[4 * b + q] >= lo) << (4 * b + q);
            }
        }
        const uint32_t nh = __popc(hits);
        uint32_t incl = nh;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t wtot = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t wbase = 0;
        if (lane == 31 && wtot) wbase = atomicAdd(&nbuf, wtot);
        wbase = __shfl_sync(0xffffffffu, wbase, 31);
        uint32_t at = wbase + incl - nh;
        while (hits) {
            const int q = __ffs(hits) - 1;
            hits &= hits - 1;
            const int j = j0 + ((q >> 2) * kMcThreads + threadIdx.x) * 4 + (q & 3);
            const uint64_t kp = ((uint64_t)keys[q] << 32) | (uint32_t)j;
            if (at < (uint32_t)kMcLocal) {
                buf[at] = kp;
            } else {
                const uint32_t slot = atomicAdd(cnt, 1u);
                if (slot < (uint32_t)kMcCandCap) cand[slot] = kp;
            }
            ++at;
        }
    }
    __syncthreads();
    const uint32_t nb = min(nbuf, (uint32_t)kMcLocal);
    if (threadIdx.x == 0) base = nb ? atomicAdd(cnt, nb) : 0u;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < nb; i += kMcThreads)
        if (base + i < (uint32_t)kMcCandCap) cand[base + i] = buf[i];
}

__global__ void __launch_bounds__(kMapThreads, 1) topk_mc_finish_kernel(const float* scores,
                                                                       int64_t score_row_stride, Geom g, int top_k,
                                                                       McLayout L, int32_t* idx,
                                                                       int64_t idx_row_stride,
                                                                       int32_t* n_sel, int known_bin) {
    extern __shared__ __align__(16) unsigned char map_raw[];
    MapShared& sh = *reinterpret_cast<MapShared*>(map_raw);
    GenShared<kMapThreads>& gsh = *reinterpret_cast<GenShared<kMapThreads>*>(map_raw);
    pdl_trigger();
    pdl_wait();
    const int64_t r = blockIdx.x;
    const int n = row_n_vis(g, r);
    const int K = min(top_k, n);
    const float* s = scores + r * score_row_stride;
    int32_t* out = idx + r * idx_row_stride;
    const uint32_t n_cand = L.cnt[r];
    if (K == n || n > kMapMax || n_cand > (uint32_t)kCandCap || n_cand < (uint32_t)K) {
        select_row<false, kMapThreads>(s, n, top_k, 1, out, n_sel ? n_sel + r : nullptr, gsh);
        return;
    }
    // exact top K among the candidates: three radix rounds over the full keys; on the fused path
    // the first round's bin and the count above it are known from the row's histogram
    uint32_t need = (uint32_t)K, prefix = 0u, mask = 0u;
    const int shifts[3] = {21, 10, 0};
    const int bitsv[3] = {11, 11, 10};
    int round0 = 0;
    if (known_bin) {
        const uint32_t b = L.bound[r];
        if (b != 0xffffffffu) {
            prefix = b & 0xffe00000u;
            mask = 0xffe00000u;
            need -= b & 0x1fffffu;
            round0 = 1;
        }
    }
    const int nwords = (n + 31) >> 5;
    for (int i = threadIdx.x; i < nwords; i += kMapThreads) {
        sh.sel[i] = 0u;
        sh.eq[i] = 0u;
    }
    // with the first bin known, the next round's histogram is counted while the candidates load
    if (round0 == 1)
        for (int i = threadIdx.x; i < 2048; i += kMapThreads) sh.hist[i] = 0u;
    __syncthreads();
    const uint64_t* cand = L.cand + r * (int64_t)kMcCandCap;
    for (uint32_t i = threadIdx.x; i < n_cand; i += kMapThreads) {
        const uint64_t kp = cand[i];
        const uint32_t key = (uint32_t)(kp >> 32);
        sh.cand_key[i] = key;
        sh.cand_pos[i] = (int32_t)(uint32_t)kp;
        if (round0 == 1 && (key & mask) == prefix) atomicAdd(&sh.hist[(key >> 10) & 2047u], 1u);
    }
    __syncthreads();
    if (round0 == 1) {
        map_find_bin(2048, need, sh);
        prefix |= sh.bin << 10;
        mask |= 2047u << 10;
        need -= sh.above;
        round0 = 2;
    }
#pragma unroll 1
    for (int round = round0; round < 3; ++round) {
        if (round == 2 && sh.hist[sh.bin] <= 64u) {
            // the last round sees only the keys sharing T's top 22 bits (the previous round's bin
            // count, at most 64 here): T is the need-th largest of them, found by ranking them
            // directly - the same T and count above it as the 1024-bin histogram gives
            uint32_t* small = sh.hist;
            __syncthreads();   // (every thread has read the bin count)
            if (threadIdx.x == 0) sh.cand_n = 0u;
            __syncthreads();
            for (uint32_t i = threadIdx.x; i < n_cand; i += kMapThreads) {
                const uint32_t key = sh.cand_key[i];
                if ((key & mask) == prefix) {
                    const uint32_t slot = atomicAdd(&sh.cand_n, 1u);
                    if (slot < 64u) small[slot] = key;
                }
            }
            __syncthreads();
            const uint32_t m = min(sh.cand_n, 64u);
            if (threadIdx.x < m) {
                const uint32_t key = small[threadIdx.x];
                uint32_t gt = 0, ge = 0;
                for (uint32_t j = 0; j < m; ++j) {
                    gt += small[j] > key ? 1u : 0u;
                    ge += small[j] >= key ? 1u : 0u;
                }
                if (gt < need && need <= ge) {   // (keys equal to T all write the same values)
                    sh.bin = key & 1023u;
                    sh.above = gt;
                }
            }
            __syncthreads();
            prefix |= sh.bin;
            mask = 0xffffffffu;
            need -= sh.above;
            break;
        }
        map_cand_hist(sh, n_cand, prefix, mask, shifts[round], bitsv[round]);
        map_find_bin(1 << bitsv[round], need, sh);
        prefix |= sh.bin << shifts[round];
        mask |= ((1u << bitsv[round]) - 1u) << shifts[round];
        need -= sh.above;
    }
    const uint32_t T = prefix;
    for (uint32_t i = threadIdx.x; i < n_cand; i += kMapThreads) {
        const uint32_t key = sh.cand_key[i];
        const int p = sh.cand_pos[i];
        if (key > T) atomicOr(&sh.sel[p >> 5], 1u << (p & 31));
        else if (key == T) atomicOr(&sh.eq[p >> 5], 1u << (p & 31));
    }
    __syncthreads();
    const int wpt = (nwords + kMapThreads - 1) / kMapThreads;
    const int w0 = threadIdx.x * wpt;
    uint32_t cs = 0, ce = 0;
    for (int w = w0; w < min(w0 + wpt, nwords); ++w) {
        cs += __popc(sh.sel[w]);
        ce += __popc(sh.eq[w]);
    }
    uint32_t bs, be, ts, te;
    map_scan2(cs, ce, sh, &bs, &be, &ts, &te);
    uint32_t off = bs + min(be, need);
    uint32_t eq_rank = be;
    for (int w = w0; w < min(w0 + wpt, nwords); ++w) {
        const uint32_t a = sh.sel[w];
        uint32_t any = a | sh.eq[w];
        while (any) {
            const int bit = __ffs(any) - 1;
            any &= any - 1;
            bool take = (a >> bit) & 1u;
            if (!take) {
                take = eq_rank < need;
                ++eq_rank;
            }
            if (take) out[off++] = w * 32 + bit;
        }
    }
    for (int i = K + threadIdx.x; i < top_k; i += kMapThreads) out[i] = -1;
    if (threadIdx.x == 0 && n_sel) n_sel[r] = K;
}

// Many rows of at most sel::kMaxKeys scores (a causal prefill): one CTA of kRowThreads per row, the
// row's order keys in shared memory (two CTAs per SM), three radix rounds and an ordered write-out
// from per-group selection bits (select_row.cuh).
constexpr int kRowThreads = 384;

__global__ void __launch_bounds__(kRowThreads) topk_rows_kernel(const float* scores, int64_t score_row_stride,
                                                               Geom g, int top_k, int32_t* idx,
                                                               int64_t idx_row_stride, int32_t* n_sel) {
    extern __shared__ __align__(16) uint8_t rows_smem[];
    pdl_trigger();
    pdl_wait();
    const int64_t r = blockIdx.x;
    sel::select_row<kRowThreads>(scores + r * score_row_stride, row_n_vis(g, r), top_k, nullptr,
                                 idx + r * idx_row_stride, n_sel ? n_sel + r : nullptr, rows_smem);
}

}  // namespace

cudaError_t launch_topk(const float* scores, int64_t score_row_stride, const Geom& g, int top_k,
                        int block_size, int32_t* idx, int64_t idx_row_stride, int32_t* n_sel, void* ws,
                        size_t ws_bytes, cudaStream_t st) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0) return cudaSuccess;
    if (block_size > 1) {
        if (g.max_n_kv / block_size <= blk::kRankMax)
            return launch_pdl(topk_block_rank_kernel, dim3((unsigned)n_rows), dim3(blk::kRankThreads), 0, st, scores,
                              score_row_stride, g, top_k, block_size, idx, idx_row_stride, n_sel);
        return launch_pdl(topk_kernel<true>, dim3((unsigned)n_rows), dim3(kThreads), 0, st, scores, score_row_stride,
                          g, top_k, block_size, idx, idx_row_stride, n_sel);
    } else if (ws && ws_bytes >= mc_bytes(n_rows) && n_rows < 2 * sm_count() && g.max_n_kv >= 4 * kMcChunk) {
        // few long rows: spread the passes over the rows' chunks
        const McLayout L = mc_layout(ws, n_rows);
        const int chunks = (g.max_n_kv + kMcChunk - 1) / kMcChunk;
        cudaError_t e = launch_pdl(topk_mc_bound_kernel, dim3((unsigned)n_rows), dim3(kMcThreads), 0, st, scores,
                                   score_row_stride, g, top_k, L);
        if (e != cudaSuccess) return e;
        if (chunks > 0) {
            e = launch_pdl(topk_mc_filter_kernel, dim3((unsigned)chunks, (unsigned)n_rows), dim3(kMcThreads), 0, st,
                           scores, score_row_stride, g, top_k, L);
            if (e != cudaSuccess) return e;
        }
        const size_t sm = sizeof(MapShared);
        cudaFuncSetAttribute(topk_mc_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        return launch_pdl(topk_mc_finish_kernel, dim3((unsigned)n_rows), dim3(kMapThreads), sm, st, scores,
                          score_row_stride, g, top_k, L, idx, idx_row_stride, n_sel, 0);
    } else if (g.max_n_kv <= sel::kMaxKeys && n_rows >= 2 * sm_count()) {
        // many short rows: a lighter CTA per row, two per SM
        cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sel::kBytes);
        return launch_pdl(topk_rows_kernel, dim3((unsigned)n_rows), dim3(kRowThreads), (size_t)sel::kBytes, st,
                          scores, score_row_stride, g, top_k, idx, idx_row_stride, n_sel);
    } else {
        const size_t sm = sizeof(MapShared);
        cudaFuncSetAttribute(topk_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        return launch_pdl(topk_map_kernel, dim3((unsigned)n_rows), dim3(kMapThreads), sm, st, scores,
                          score_row_stride, g, top_k, idx, idx_row_stride, n_sel,
                          static_cast<const uint32_t*>(nullptr));
    }
    return cudaGetLastError();
}

// the fused workspace: [rows][2048] histogram counts, then the candidate lists, bounds and
// candidate counters of the multi-CTA path (mc_layout)
size_t topk_fused_workspace_bytes(int64_t n_rows) {
    if (n_rows <= 0) return 0;
    return (size_t)n_rows * 2048 * sizeof(uint32_t) + mc_bytes(n_rows);
}

static McLayout fused_mc(void* ws, int64_t n_rows) {
    return mc_layout(static_cast<char*>(ws) + (size_t)n_rows * 2048 * sizeof(uint32_t), n_rows);
}

FusedArrays topk_fused_arrays(void* ws, int64_t n_rows) {
    FusedArrays a;
    a.hist = static_cast<uint32_t*>(ws);
    a.cnt = fused_mc(ws, n_rows).cnt;
    return a;
}

// Rows up to kFusedMapMax keys: one CTA per row (topk_map_kernel seeded with the row's histogram:
// one pass over the scores, which the scorer left in L2, marks the keys above the threshold bin
// and collects that bin's keys, ranked in shared memory).  Longer rows: the filter over all SMs
// (each CTA derives the row's bound from the histogram first), then the finish (one SM streaming a 131072-key row is slower than the
// two extra launches).
constexpr int kFusedMapMax = 16384;

cudaError_t launch_topk_fused(const float* scores, int64_t score_row_stride, const Geom& g, int top_k, int32_t* idx,
                              int64_t idx_row_stride, int32_t* n_sel, void* ws, cudaStream_t st) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0) return cudaSuccess;
    const size_t sm = sizeof(MapShared);
    if (g.max_n_kv <= kFusedMapMax) {
        cudaFuncSetAttribute(topk_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        return launch_pdl(topk_map_kernel, dim3((unsigned)n_rows), dim3(kMapThreads), sm, st, scores,
                          score_row_stride, g, top_k, idx, idx_row_stride, n_sel, static_cast<const uint32_t*>(ws));
    }
    const McLayout L = fused_mc(ws, n_rows);
    // filter chunks of 8192 scores (two passes of four 16-byte loads per thread), longer when a
    // batch would need more than 2048 CTAs
    int64_t chunk = 8192;
    while ((g.max_n_kv + chunk - 1) / chunk * n_rows > 2048 && chunk < (1 << 20)) chunk *= 2;
    const int64_t chunks = (g.max_n_kv + chunk - 1) / chunk;
    cudaError_t e = launch_pdl(topk_hist_filter_kernel, dim3((unsigned)chunks, (unsigned)n_rows), dim3(kMcThreads),
                               0, st, scores, score_row_stride, static_cast<const uint32_t*>(ws), g, top_k, L,
                               (int)chunk);
    if (e != cudaSuccess) return e;
    cudaFuncSetAttribute(topk_mc_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    return launch_pdl(topk_mc_finish_kernel, dim3((unsigned)n_rows), dim3(kMapThreads), sm, st, scores,
                      score_row_stride, g, top_k, L, idx, idx_row_stride, n_sel, 1);
}

size_t topk_workspace_bytes(int64_t n_rows, int top_k) {
    if (n_rows <= 0 || top_k <= 0) return 0;
    int sms = sm_count();
    if (sms < 2) sms = 152;
    return n_rows < 2 * sms ? mc_bytes(n_rows) : 0;
}

}  // namespace lidx
