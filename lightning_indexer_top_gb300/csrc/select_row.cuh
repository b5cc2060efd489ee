// Top-k of one row of scores by one CTA, in shared memory (the decode step's selection and the
// selection of many rows of at most kMaxKeys scores): the same positions idx_topk selects - the
// top_k largest scores in ascending position order, the lowest positions first among equal scores
// (-0 == +0), -1 padding - from three radix rounds over the order keys' bits (11, 11, 10), the first
// from a histogram of the top 11 bits when one is given, and selection bits per 32-key group.
#pragma once
#include "lidx_internal.cuh"

namespace lidx {
namespace sel {

constexpr int kMaxKeys = 16384;                       // keys a row may have
constexpr int kKeysOff = 0;                           // order keys [kMaxKeys]
constexpr int kHistOff = kKeysOff + kMaxKeys * 4;     // histograms of the three rounds [2048 + 2048 + 1024]
constexpr int kGroups = kMaxKeys / 32;                // 32-key groups of a row
constexpr int kBitsOff = kHistOff + 5120 * 4;         // per group, the selected and the equal keys' bits
constexpr int kScratchOff = kBitsOff + 2 * kGroups * 4;   // scan and bin-search slots [6][32]
constexpr int kBytes = kScratchOff + 6 * 32 * 4;      // shared memory of one row's selection

// exclusive prefix of v over the CTA (kT threads) and the total.  `slot` (2 x kWarps words)
// must not be used by another scan or bin search before the next CTA barrier after this one.
template <int kT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* slot, uint32_t* total) {
    constexpr int kW = kT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    __syncwarp();   // shuffles of a reconverged warp (a diverged one pays for every shuffle)
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) slot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t u = lane < kW ? slot[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += y;
        }
        if (lane < kW) slot[kW + lane] = u;
    }
    __syncthreads();
    *total = slot[2 * kW - 1];
    return (wid > 0 ? slot[kW + wid - 1] : 0u) + x - v;
}

// bin of a histogram (NB bins) holding the need-th largest counted key, the count in higher bins,
// and the histogram's total, to every thread (bin and count unspecified when need > total).
// Thread t < NB/8 sums the 8 bins NB-8(t+1) .. NB-8t-1 (higher bins to lower threads); warp scans
// and the warps' totals give each thread the count in its bins and all higher ones, and the one
// thread whose bins hold the need-th key walks them.  `slot` (kWarps + 3 words) as for block_scan.
template <int NB, int kT>
__device__ __forceinline__ void find_bin(const uint32_t* hist, uint32_t need, uint32_t* slot, uint32_t* bin,
                                         uint32_t* above, uint32_t* total) {
    constexpr int nt = NB / 8, nw = nt / 32, kW = kT / 32;
    static_assert(nt % 32 == 0 && nt <= kT && nw <= kW, "whole warps, 8 bins per thread");
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t h[8], c = 0, x = 0;
    if (threadIdx.x < nt) {
        const uint4* h4 = reinterpret_cast<const uint4*>(hist + NB - 8 * (threadIdx.x + 1));
        const uint4 a0 = h4[0], a1 = h4[1];
        h[0] = a0.x; h[1] = a0.y; h[2] = a0.z; h[3] = a0.w;
        h[4] = a1.x; h[5] = a1.y; h[6] = a1.z; h[7] = a1.w;
        c = ((h[0] + h[1]) + (h[2] + h[3])) + ((h[4] + h[5]) + (h[6] + h[7]));
        __syncwarp();
        x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) slot[wid] = x;
    }
    __syncthreads();
    if (threadIdx.x < nt) {
        uint32_t off = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < nw; ++w) {
            const uint32_t t = slot[w];
            off += w < wid ? t : 0u;
            tot += t;
        }
        x += off;   // keys in this thread's bins and all higher bins
        if (x - c < need && x >= need) {
            uint32_t cc = x - c;
            int b = NB - 8 * (int)threadIdx.x - 8;
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (cc + h[i] >= need) {
                    b = NB - 8 * (int)threadIdx.x - 8 + i;
                    break;
                }
                cc += h[i];
            }
            slot[kW] = (uint32_t)b;
            slot[kW + 1] = cc;
        }
        if (threadIdx.x == 0) slot[kW + 2] = tot;
    }
    __syncthreads();
    *bin = slot[kW];
    *above = slot[kW + 1];
    *total = slot[kW + 2];
}

// The top_k positions of a row of n <= kMaxKeys scores (complete in global memory) in ascending order,
// the lowest positions first among equal scores (-0 == +0), -1 padding up to top_k; n_sel[r].
// ghist: the row's histogram of the order keys' top 11 bits (NULL: counted here).
// Three radix rounds (11, 11, 10 bits) find the top_k-th order key T: the first from the
// histogram (its bin found while the row's scores are in flight), the others counting only the
// keys in the previous round's bin.  Position i of the row is handled by thread i mod kT, so
// a warp holds the 32 keys of one group in each batch entry, one ballot gives the group's
// selection bits, and the output is written from those bits.
template <int kT>
__device__ void select_row(const float* s, int n, int top_k, const uint32_t* ghist, int32_t* out, int32_t* n_sel_r,
                           uint8_t* smem) {
    constexpr int kW = kT / 32;
    static_assert(2 * kT >= kGroups, "two 32-key groups per thread cover a row");
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kKeysOff);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kHistOff);
    uint32_t* hist2 = hist + 2048;
    uint32_t* hist3 = hist + 4096;
    uint32_t* selw = reinterpret_cast<uint32_t*>(smem + kBitsOff);
    uint32_t* eqw = selw + kGroups;
    uint32_t* scratch = reinterpret_cast<uint32_t*>(smem + kScratchOff);   // 6 slots of 32 words
    const int K = min(top_k, n);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (K == n) {
        for (int i = threadIdx.x; i < n; i += kT) out[i] = i;
    } else {
        constexpr int kB = 24;                          // positions per thread and batch
        constexpr int kStride = kB * kT;          // 9216 positions (288 groups) per batch
        constexpr int kHB = (2048 + kT - 1) / kT;
        // the histogram and the first batch of scores in flight together
        uint32_t hv[kHB];
#pragma unroll
        for (int u = 0; u < kHB; ++u) {
            const int i = threadIdx.x + u * kT;
            hv[u] = (ghist && i < 2048) ? __ldcg(ghist + i) : 0u;
        }
        float v[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int i = threadIdx.x + u * kT;
            v[u] = i < n ? __ldcg(s + i) : 0.f;
        }
        for (int i = threadIdx.x; i < 3072; i += kT) hist2[i] = 0u;   // rounds 2 and 3
#pragma unroll
        for (int u = 0; u < kHB; ++u) {
            const int i = threadIdx.x + u * kT;
            if (i < 2048) hist[i] = hv[u];
        }
        __syncthreads();
        // round 1 from the scorer's histogram when it counts exactly this row's keys
        uint32_t need = (uint32_t)K, bin, above, total;
        find_bin<2048, kT>(hist, need, scratch + 32, &bin, &above, &total);
        const bool have = total == (uint32_t)n;
        // order keys to shared memory; the first round's bin counted for round 2
        for (int b0 = 0; b0 < n; b0 += kStride) {
            if (b0 > 0) {
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int i = b0 + threadIdx.x + u * kT;
                    v[u] = i < n ? __ldcg(s + i) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = b0 + threadIdx.x + u * kT;
                const uint32_t key = order_key(v[u]);
                if (i < n) keys[i] = key;
                if (have && i < n && (key >> 21) == bin) atomicAdd(&hist2[(key >> 10) & 2047u], 1u);
            }
        }
        __syncthreads();
        if (!have) {
            // the scorer's counts are incomplete: count here
            for (int i = threadIdx.x; i < 2048; i += kT) hist[i] = 0u;
            __syncthreads();
            for (int i = threadIdx.x; i < n; i += kT) atomicAdd(&hist[keys[i] >> 21], 1u);
            __syncthreads();
            find_bin<2048, kT>(hist, need, scratch + 32, &bin, &above, &total);
            for (int i = threadIdx.x; i < n; i += kT) {
                const uint32_t key = keys[i];
                if ((key >> 21) == bin) atomicAdd(&hist2[(key >> 10) & 2047u], 1u);
            }
            __syncthreads();
        }
        need -= above;
        const uint32_t p1 = bin;                        // top 11 bits of T
        find_bin<2048, kT>(hist2, need, scratch + 64, &bin, &above, &total);
        need -= above;
        const uint32_t p2 = (p1 << 11) | bin;           // top 22 bits of T
        for (int b0 = 0; b0 < n; b0 += kStride) {
            uint32_t kk[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = b0 + threadIdx.x + u * kT;
                kk[u] = i < n ? keys[i] : 0u;
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const bool ok = b0 + (int)threadIdx.x + u * kT < n;
                if (ok && (kk[u] >> 10) == p2) atomicAdd(&hist3[kk[u] & 1023u], 1u);
            }
        }
        __syncthreads();
        find_bin<1024, kT>(hist3, need, scratch + 96, &bin, &above, &total);
        need -= above;                                  // keys equal to T to take (the lowest positions)
        const uint32_t T = (p2 << 10) | bin;
        const bool all_eq = need == hist3[bin];         // (uniform) every key equal to T is taken
        // selection bits of each 32-key group: entry u of warp w in the batch at b0 is group
        // b0/32 + w + 12u; lane u of the warp keeps that group's bits and stores them
        for (int b0 = 0; b0 < n; b0 += kStride) {
            uint32_t kk[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = b0 + threadIdx.x + u * kT;
                kk[u] = i < n ? keys[i] : 0u;
            }
            __syncwarp();
            uint32_t my_sel = 0u, my_eq = 0u;
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const bool ok = b0 + (int)threadIdx.x + u * kT < n;
                const uint32_t gt = __ballot_sync(0xffffffffu, ok && kk[u] > T);
                const uint32_t eq = __ballot_sync(0xffffffffu, ok && kk[u] == T);
                my_sel = lane == u ? (all_eq ? (gt | eq) : gt) : my_sel;
                my_eq = lane == u ? eq : my_eq;
            }
            const int grp = (b0 >> 5) + wid + lane * (kT / 32);
            if (lane < kB && grp < kGroups) {
                selw[grp] = my_sel;
                eqw[grp] = my_eq;
            }
        }
        const int groups = (n + 31) >> 5;
        const int ga = 2 * threadIdx.x, gb = ga + 1;    // this thread's two groups, in position order
        __syncthreads();
        if (!all_eq) {
            // ties at T: only the lowest `need` positions among the keys equal to T
            const uint32_t ea = ga < groups ? eqw[ga] : 0u, eb = gb < groups ? eqw[gb] : 0u;
            uint32_t tot;
            const uint32_t before = block_scan<kT>((uint32_t)(__popc(ea) + __popc(eb)), scratch + 128, &tot);
            uint32_t left = before >= need ? 0u : need - before;
            uint32_t ta = 0u, tb = 0u;
            for (uint32_t w = ea; w && left; w &= w - 1u, --left) ta |= w & (0u - w);
            for (uint32_t w = eb; w && left; w &= w - 1u, --left) tb |= w & (0u - w);
            if (ga < groups) selw[ga] |= ta;
            if (gb < groups) selw[gb] |= tb;
            __syncthreads();
        }
        // ordered write-out: each thread the set bits of its two groups
        const uint32_t sa = ga < groups ? selw[ga] : 0u, sb = gb < groups ? selw[gb] : 0u;
        uint32_t tot;
        uint32_t pos = block_scan<kT>((uint32_t)(__popc(sa) + __popc(sb)), scratch + 160, &tot);
        for (uint32_t w = sa; w; w &= w - 1u) out[pos++] = ga * 32 + (__ffs(w) - 1);
        for (uint32_t w = sb; w; w &= w - 1u) out[pos++] = gb * 32 + (__ffs(w) - 1);
    }
    for (int i = K + threadIdx.x; i < top_k; i += kT) out[i] = -1;
    if (threadIdx.x == 0 && n_sel_r) *n_sel_r = K;
    __syncthreads();
}

}  // namespace sel
}  // namespace lidx
