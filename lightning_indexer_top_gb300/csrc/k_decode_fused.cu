// The fused decode step for few short rows: lightning-indexer scores, top-k
// selection and sparse MLA attention in ONE persistent launch (the pages' fused
// indexer + top-k op, "Route DSA indexer selection through ggml_indexer_topk",
// feeding the gathered decode attention, "Gather OpenPangu DSA decode reads",
// ik_llama_opt commit log).  Decode rows (one query per sequence) with few
// keys leave every separate kernel latency-bound; here one grid of 2-CTA
// clusters, all resident at once (a cooperative launch), runs four phases:
//   1. scores: CTA b takes the 128-key tiles b, b+G, b+2G, ... of all rows
//      (G CTAs) and computes s[r, j] = sum_h w[r, h] max(0, q[r, h] . k_j)
//      exactly as idx_score does on the tensor cores: the tile (16-byte
//      cp.async copies into the 128-byte swizzle, through the page table when
//      there is one) and the row's q converted to the key type are the A and B
//      operands of 8 tcgen05.mma (M=128 keys, N=64 heads, K=16 each) into
//      TMEM, and four epilogue warps (thread = key) apply ReLU, the weights and
//      the head sum in the same order, so the scores are bit for bit those of
//      idx_score.  All of a CTA's tiles (four at most at a time) are loaded at
//      once, and two TMEM accumulators let a tile's MMAs run under the
//      previous tile's epilogue.  The epilogue also counts every score into
//      its row's 2048-bin histogram of the order key's top 11 bits (equal bins
//      of a warp folded into one atomic add; the histograms, in the workspace,
//      are zeroed by all CTAs at the start behind a counter).
//   2. selection: each row is selected by a CTA of its own (one without an
//      attention unit when there are enough) once a per-row counter shows
//      all its tiles scored: order keys in shared memory; the histogram gives the
//      bin of the top_k-th key, two more radix rounds (11 and 10 bits) over
//      that bin fix the top_k-th key T and how many keys equal to T are taken,
//      and two block scans write the positions in ascending order, the lowest
//      positions first among keys equal to T - the selection idx_topk makes.
//      It then raises the row's ready flag.
//   3. attention: cluster c runs unit c = (row, key split) of the MLA
//      attention (the code of sparse_attn_decode's 2-CTA unit) once its row's
//      flag is up; its Q went into TMEM at the start, while phase 1 ran.
//   4. merge: after a grid barrier every CTA merges the key splits of a share
//      of the (row, 4-column) items, thread = head (the combine kernel's
//      layout and arithmetic, an item's loads of all splits issued together).
// Flags and counters live in one of 256 slots of a device array (round-robin
// per launch); the last CTA to finish returns its slot to zero.  Every wait is
// bounded: a timeout records IDX_ERR_TIMEOUT and the CTA goes on (its inputs
// are then unspecified but every access stays in bounds), so the grid always
// completes.
#include <atomic>
#include <cstring>
#include <type_traits>

#include "attn_mla_tc.cuh"
#include "select_row.cuh"

namespace lidx {

constexpr int kFusedSlots = 256;
constexpr int kFusedMaxRows = 32;                   // one lane of warp 0 per row at the start
static_assert(kFusedMaxRows <= 32, "rows are counted by the lanes of one warp");
constexpr int kFusedWords = 2 * kFusedMaxRows + 3;   // row tile counters, row flags, grid barrier, finished CTAs,
                                                     // CTAs that have zeroed their histogram slice
__device__ unsigned int g_fused_sync[kFusedSlots][kFusedWords];

namespace {
using namespace sm100;

constexpr int kFK = 128;                          // keys per score tile
constexpr int kFH = 64;                           // indexer heads
constexpr int kFD = 128;                          // indexer head dim
constexpr int kFKHalf = kFK * 128;                // one 64-column block of a key tile (16 KB)
constexpr int kFQHalf = kFH * 128;                // one 64-column block of q (8 KB)
constexpr int kFStage = 2 * kFKHalf + 2 * kFQHalf;   // 48 KB
constexpr int kFStages = 4;                       // score tiles in flight per CTA
constexpr int kFMaxSplits = 8;                    // key splits the merge handles
constexpr int kFWOff = kFStages * kFStage;        // weights of the stages [kFStages][64]
// score accumulators (two, used in turn): rank 0 in its S columns (Q at 0..287; S is used only in
// phase 3), rank 1 in its O columns (written only in phase 3)
constexpr uint32_t kFAccCol0 = 384;
constexpr uint32_t kFAccCol1 = 0;
static_assert(sel::kBytes <= kFWOff, "the selection's shared memory inside the score stages");

// after the attention unit's control block
struct FCtl {
    uint64_t mma[2];               // phase 1: MMAs into accumulator a completed
    uint64_t kfull[kFStages];      // phase 1: stage's key tile landed (tensor-map loads)
    uint64_t accfree[2];           // phase 1: the epilogue warps have read accumulator a
    int tdone[kFStages];           // phase 1: epilogue warps done with the stage's tile
    int n_pend;                    // rows this CTA completed (to select)
    int pend[kFusedMaxRows];
    int pre[kFusedMaxRows + 1];    // score tiles of the rows before row r
    int nvis[kFusedMaxRows];       // visible keys of row r
    int flag_ok;
};
constexpr size_t kFSmemBytes = kSmemBytes + 8 + sizeof(FCtl);
static_assert(kFSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename TK, typename TQ>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) decode_fused_kernel(
    const TQ* __restrict__ qi, const float* __restrict__ w, const TK* __restrict__ kc, int64_t k_row_stride,
    int64_t k_rows, Geom g, int top_k, float* scores, int64_t score_row_stride, int32_t* idx, int64_t idx_row_stride,
    int32_t* n_sel, const __nv_bfloat16* __restrict__ lat, int64_t lat_row_stride, int64_t kv_rows,
    const __nv_bfloat16* __restrict__ qa, float scale_log2, int splits, int kps, void* out, int out_dtype,
    float* part_o, float* part_ml, uint32_t* ghist, int slot, const __grid_constant__ CUtensorMap kmap,
    int use_tma) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const MlaSmem sm = mla_smem(smem);
    Ctl& c = *sm.c;
    FCtl& f = *reinterpret_cast<FCtl*>((reinterpret_cast<uintptr_t>(sm.c + 1) + 7) & ~uintptr_t(7));
    unsigned int* sync = g_fused_sync[slot];
    unsigned int* row_cnt = sync;
    unsigned int* row_flag = sync + kFusedMaxRows;
    unsigned int* gbar = sync + 2 * kFusedMaxRows;
    unsigned int* fin = gbar + 1;
    unsigned int* zeroed = gbar + 2;

    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = g.B;                        // one query row per sequence
    const int64_t cid = blockIdx.x >> 1;
    const int64_t n_units = (int64_t)n_rows * splits;

    if (warp == 0) {
        // lane r: row r's visible keys and score tiles (all rows' loads in flight at once), a warp
        // scan for the tiles before each row
        const int r = lane;   // n_rows <= 32
        int nv = 0, tiles = 0;
        if (r < n_rows) {
            nv = row_n_vis(g, r);
            tiles = (nv + kFK - 1) / kFK;
        }
        int incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (r < n_rows) {
            f.nvis[r] = nv;
            f.pre[r] = incl - tiles;
        }
        if (lane == 31) f.pre[n_rows] = incl;
        // row r is selected, once all its tiles are scored, by a CTA of its own: one of the
        // clusters without an attention unit when there are enough of them
        const int64_t sel_cta = 2 * (int64_t)n_rows * splits + n_rows <= (int64_t)gridDim.x
                                    ? 2 * (int64_t)n_rows * splits + r
                                    : (int64_t)r * gridDim.x / n_rows;
        const bool mine = r < n_rows && sel_cta == (int64_t)blockIdx.x;
        const unsigned int m = __ballot_sync(0xffffffffu, mine);
        if (mine) f.pend[__popc(m & ((1u << lane) - 1u))] = r;
        if (lane == 0) {
            f.n_pend = __popc(m);
            mla_init(c);
            mbar_init(&f.mma[0], 1);
            mbar_init(&f.mma[1], 1);
            for (int i = 0; i < kFStages; ++i) mbar_init(&f.kfull[i], 1);
            mbar_init(&f.accfree[0], 4);
            mbar_init(&f.accfree[1], 4);
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // this CTA's slice of the rows' histograms (16-byte stores), then a count on `zeroed`
    {
        const int64_t n4 = (int64_t)n_rows * 512;
        const int64_t per = (n4 + gridDim.x - 1) / gridDim.x;
        const int64_t a0 = (int64_t)blockIdx.x * per, e = min(n4, a0 + per);
        uint4* h4 = reinterpret_cast<uint4*>(ghist);
        for (int64_t i = a0 + threadIdx.x; i < e; i += kThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(zeroed, 1u);
    }
    const uint32_t tmem = c.tmem_base;

    // ------------------------------------------------------------------ 1. scores
    const int total = f.pre[n_rows];
    const int G = (int)gridDim.x;
    const int my_n = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / G + 1 : 0;
    const uint32_t acc_col0 = rank == 0 ? kFAccCol0 : kFAccCol1;
    // row and tile of this CTA's i-th tile; `r` carries the row of an earlier call (tiles are
    // visited in increasing order, so the search only moves forward)
    auto tile_row = [&](int i, int& r, int& t) {
        const int gt = (int)blockIdx.x + i * G;
        while (r + 1 < n_rows && f.pre[r + 1] <= gt) ++r;
        t = gt - f.pre[r];
    };
    const uint32_t idesc = idesc_f16_f32(kFK, kFH, std::is_same<TK, __nv_bfloat16>::value ? 1 : 0);
    // the epilogue warps add to the histograms only once every CTA has zeroed its slice (checked
    // before a warp's first add, so the wait overlaps the first tiles' loads)
    int hist_state = 0;   // 0 not yet checked, 1 zeroed everywhere, -1 gave up waiting
    int r_ld = 0, r_q = 0, r_ep = 0, r_pub = 0;   // running rows of the loops over this CTA's tiles
    for (int i0 = 0; i0 < my_n; i0 += kFStages) {
        const int nb = min(kFStages, my_n - i0);
        // every tile of the batch: the key rows of a contiguous cache by two tensor-map boxes of
        // 64 columns x 128 rows (zero-filled past the allocation), of a paged one by 16-byte copies...
        if (use_tma) {
            if (threadIdx.x == 0) {
                for (int bt = 0; bt < nb; ++bt) {
                    int t;
                    tile_row(i0 + bt, r_ld, t);
                    const int r = r_ld;
                    const int64_t krow = seq_row0(g, r) + (int64_t)t * kFK;
                    if (krow < 0 || krow + min(f.nvis[r] - t * kFK, kFK) > k_rows)
                        flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                    uint8_t* dst = smem + bt * kFStage;
                    mbar_arrive_expect_tx(&f.kfull[bt], (uint32_t)(2 * kFKHalf));
                    tma_load_2d(dst, &kmap, &f.kfull[bt], 0, (int32_t)krow);
                    tma_load_2d(dst + kFKHalf, &kmap, &f.kfull[bt], 64, (int32_t)krow);
                }
            }
        } else for (int bt = 0; bt < nb; ++bt) {
            int t;
            tile_row(i0 + bt, r_ld, t);
            const int r = r_ld;
            const int nv = f.nvis[r];
            const uint32_t base = smem_u32(smem + bt * kFStage);
            const int64_t row0 = g.page_table ? 0 : seq_row0(g, r);   // read once per tile
            for (int e = threadIdx.x; e < kFK * 16; e += kThreads) {
                const int key = e >> 4, cc = e & 15;
                const int j = t * kFK + key;
                const int jj = j < nv ? j : 0;
                const int64_t row = g.page_table ? key_row(g, r, jj) : row0 + jj;
                const bool ok = row >= 0 && row < k_rows;
                if (!ok && j < nv && cc == 0) flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                const TK* src = kc + (ok ? row * k_row_stride : 0) + cc * 8;
                cp_async16_zfill(base + (cc >> 3) * kFKHalf + key * 128 + (((cc & 7) ^ (key & 7)) << 4), src,
                                 ok ? 16u : 0u);
            }
        }
        cp_async_commit();
        // ... and each tile's q row converted to the key type (the B operand, swizzled) with its
        // weights; all of the batch's q loads are issued before the first conversion
        {
            constexpr int kPer = (kFH * 16 + kThreads - 1) / kThreads;   // 16-byte q pieces per thread and tile
            constexpr int kRaw = sizeof(TQ) == 2 ? 1 : 2;
            uint4 raw[kFStages][kPer][kRaw];
#pragma unroll
            for (int bt = 0; bt < kFStages; ++bt) {
                if (bt >= nb) break;
                int t;
                tile_row(i0 + bt, r_q, t);
                const int r = r_q;
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int ch = threadIdx.x + k * kThreads;
                    if (ch < kFH * 16) {
                        const uint4* src = reinterpret_cast<const uint4*>(qi + ((int64_t)r * kFH + (ch >> 4)) * kFD +
                                                                          (ch & 15) * 8);
#pragma unroll
                        for (int x = 0; x < kRaw; ++x) raw[bt][k][x] = src[x];
                    }
                }
                float* ws = reinterpret_cast<float*>(smem + kFWOff) + bt * kFH;
                if (threadIdx.x < kFH) ws[threadIdx.x] = w[(int64_t)r * kFH + threadIdx.x];
            }
            bool overflow = false;
#pragma unroll
            for (int bt = 0; bt < kFStages; ++bt) {
                if (bt >= nb) break;
                uint8_t* qdst = smem + bt * kFStage + 2 * kFKHalf;
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int ch = threadIdx.x + k * kThreads;
                    if (ch >= kFH * 16) continue;
                    const int h = ch >> 4, cc = ch & 15;
                    TK vals[8];
                    if constexpr (sizeof(TQ) == 2) {
                        const TQ* e = reinterpret_cast<const TQ*>(&raw[bt][k][0]);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const float x = to_f32(e[jj]);
                            vals[jj] = from_f32<TK>(x);
                            if constexpr (std::is_same<TK, __half>::value) overflow |= fabsf(x) >= 65520.f;
                        }
                    } else {
                        const float* e = reinterpret_cast<const float*>(&raw[bt][k][0]);
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) vals[jj] = from_f32<TK>(e[jj]);
                    }
                    *reinterpret_cast<uint4*>(qdst + (cc >> 3) * kFQHalf + h * 128 + (((cc & 7) ^ (h & 7)) << 4)) =
                        *reinterpret_cast<const uint4*>(vals);
                }
            }
            if (overflow) flag(g.status, IDX_ERR_INEXACT);
        }
        cp_async_wait_group<0>();
        fence_proxy_async_smem();   // this thread's copies and q stores before the MMAs read them
        if (threadIdx.x < kFStages) f.tdone[threadIdx.x] = 0;
        __syncthreads();
        // Roles within the batch, with no CTA barrier per tile: warp 1 issues tile bt's MMAs into
        // accumulator k & 1 (k = i0 + bt) once its keys have landed and the epilogue of tile k-2
        // has read that accumulator; warps 4..7 run the epilogues; warp 2 publishes each finished
        // tile to its row's counter (the selector starts when a row's last tile is counted).
        if (warp == 1) {
            if (lane == 0) {
                for (int bt = 0; bt < nb; ++bt) {
                    const int k = i0 + bt;
                    if (use_tma && !mbar_wait(&f.kfull[bt], (uint32_t)((i0 / kFStages) & 1)))
                        flag(g.status, IDX_ERR_TIMEOUT);
                    if (k >= 2 && !mbar_wait(&f.accfree[k & 1], (uint32_t)(((k - 2) >> 1) & 1)))
                        flag(g.status, IDX_ERR_TIMEOUT);
                    const uint32_t a0 = smem_u32(smem + bt * kFStage), b0 = a0 + 2 * kFKHalf;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kFD / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t ad = desc_sw128_kmajor(a0 + (kk >> 2) * kFKHalf + off, 1024);
                        const uint64_t bd = desc_sw128_kmajor(b0 + (kk >> 2) * kFQHalf + off, 1024);
                        mma_f16_ss(tmem + acc_col0 + (k & 1) * kFH, ad, bd, idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&f.mma[k & 1]);
                }
            }
            __syncwarp();
        } else if (warp >= 4 && warp < 8) {
            for (int bt = 0; bt < nb; ++bt) {
                const int k = i0 + bt;
                int t;
                tile_row(k, r_ep, t);
                const int r = r_ep;
                // epilogue (thread = key = TMEM lane): sum_h w_h relu(D_h) in idx_score's order
                const int quad = warp & 3;
                const int j = t * kFK + quad * 32 + lane;
                const int nv = f.nvis[r];
                const bool ok = warp_wait(&f.mma[k & 1], (uint32_t)((k >> 1) & 1));
                float v0[32], v1[32];
                if (ok) {
                    tc_fence_after();
                    const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + acc_col0 + (k & 1) * kFH;
                    tmem_ld_32x32b_x32(ta, v0);
                    tmem_ld_32x32b_x32(ta + 32, v1);
                    tmem_ld_wait();
                } else if (lane == 0) {
                    flag(g.status, IDX_ERR_TIMEOUT);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&f.accfree[k & 1]);   // the accumulator may be reused
                if (ok) {
                    const float* wv = reinterpret_cast<const float*>(smem + kFWOff) + bt * kFH;
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int h = 0; h < 32; h += 2) {
                        s0 = fmaf(wv[h], fmaxf(v0[h], 0.f), s0);
                        s1 = fmaf(wv[h + 1], fmaxf(v0[h + 1], 0.f), s1);
                        s2 = fmaf(wv[32 + h], fmaxf(v1[h], 0.f), s2);
                        s3 = fmaf(wv[33 + h], fmaxf(v1[h + 1], 0.f), s3);
                    }
                    float sc = (s0 + s1) + (s2 + s3);
                    sc += 0.0f;   // -0 + +0 = +0
                    if (j < nv) scores[(int64_t)r * score_row_stride + j] = sc;
                    if (hist_state == 0) {
                        int ready = 1;
                        if (lane == 0) ready = wait_counter(zeroed, gridDim.x) ? 1 : 0;
                        hist_state = __shfl_sync(0xffffffffu, ready, 0) ? 1 : -1;
                        if (hist_state < 0 && lane == 0) flag(g.status, IDX_ERR_TIMEOUT);
                    }
                    if (hist_state > 0 && j < nv) atomicAdd(&ghist[(int64_t)r * 2048 + (order_key(sc) >> 21)], 1u);
                }
                __syncwarp();
                if (lane == 0) {   // the warp's scores and counts before its count of the tile
                    __threadfence_block();
                    atomicAdd(&f.tdone[bt], 1);
                }
            }
        } else if (warp == 2) {
            if (lane == 0) {
                for (int bt = 0; bt < nb; ++bt) {
                    int t;
                    tile_row(i0 + bt, r_pub, t);
                    const int r = r_pub;
                    const long long c0 = clock64();
                    while (*reinterpret_cast<volatile int*>(&f.tdone[bt]) < 4) {
                        if (clock64() - c0 > kWaitCycles) {
                            flag(g.status, IDX_ERR_TIMEOUT);
                            break;
                        }
                    }
                    __threadfence();   // the epilogue warps' scores and counts, then the count
                    atomicAdd(&row_cnt[r], 1u);
                }
            }
            __syncwarp();
        }
        tc_fence_before();
        __syncthreads();   // the batch's stages and both accumulators free
        tc_fence_after();
    }
    // (a row whose counts are incomplete - a CTA that gave up waiting for the zeroing - has a
    // histogram total below its key count, and its select counts the keys itself)

    // ------------------------------------------------------------------ 2. selections
    for (int k = 0; k < f.n_pend; ++k) {
        const int r = f.pend[k];
        if (threadIdx.x == 0 && !wait_counter(&row_cnt[r], (unsigned)(f.pre[r + 1] - f.pre[r])))
            flag(g.status, IDX_ERR_TIMEOUT);
        __syncthreads();
        __threadfence();   // the other CTAs' scores and counts of row r (their counts were seen above)
        sel::select_row<kThreads>(scores + (int64_t)r * score_row_stride, f.nvis[r], top_k,
                                  ghist + (int64_t)r * 2048, idx + (int64_t)r * idx_row_stride, n_sel + r, smem);
        if (threadIdx.x == 0) {
            __threadfence();
            atomicExch(&row_flag[r], 1u);
        }
    }

    // ------------------------------------------------------------------ 3. attention
    if (cid < n_units) {
        const int r = (int)(cid / splits);
        // rank 0 puts the unit's Q into TMEM while thread 0 waits for the row's selection
        if (mla_q_warp(rank)) mla_load_q(c, sm.xtiles, tmem, qa, r);
        if (threadIdx.x == 0) f.flag_ok = wait_counter(&row_flag[r], 1u) ? 1 : 0;
        __syncthreads();
        if (!f.flag_ok && threadIdx.x == 0) flag(g.status, IDX_ERR_TIMEOUT);
        __threadfence();
        const Unit u = make_unit(cid, g, n_sel, idx_row_stride, kv_rows, splits, kps);
        if (!mla_q_warp(rank)) mla_stage_rows(sm, rank, u, g, idx, idx_row_stride, kv_rows);
        tc_fence_before();
        cluster_sync();   // both CTAs' indices staged
        tc_fence_after();
        mla_run(sm, tmem, rank, u, cid, lat, lat_row_stride, g, scale_log2, splits, out, out_dtype, part_o, part_ml);
    }

    // ------------------------------------------------------------------ 4. merge of key splits
    if (splits > 1) {
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(gbar, 1u);
            if (!wait_counter(gbar, gridDim.x)) flag(g.status, IDX_ERR_TIMEOUT);
            __threadfence();
        }
        __syncthreads();
        // work item (row, 4 columns), thread = head (the combine kernel's layout and arithmetic); a
        // thread group takes two items at a time, all of their loads issued together
        const int grp = threadIdx.x >> 7, h = threadIdx.x & 127;
        const int64_t items = (int64_t)n_rows * (kDv / 4);
        const int64_t gs = (int64_t)gridDim.x * (kThreads / 128);   // thread groups in the grid
        for (int64_t p0 = (int64_t)blockIdx.x * (kThreads / 128) + grp; p0 < items; p0 += 2 * gs) {
            float ml_m[2][kFMaxSplits], ml_l[2][kFMaxSplits];
            float4 o[2][kFMaxSplits];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int64_t p = p0 + k * gs;
                const int64_t r = p / (kDv / 4);
                const int c4 = (int)(p % (kDv / 4));
#pragma unroll
                for (int s = 0; s < kFMaxSplits; ++s) {
                    ml_m[k][s] = 0.f;
                    ml_l[k][s] = 0.f;
                    o[k][s] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (p < items && s < splits) {
                        const int64_t un = r * splits + s;
                        ml_m[k][s] = __ldcg(part_ml + (un * kHq + h) * 2);
                        ml_l[k][s] = __ldcg(part_ml + (un * kHq + h) * 2 + 1);
                        o[k][s] = __ldcg(reinterpret_cast<const float4*>(part_o + un * (int64_t)kDv * kHq) +
                                         (int64_t)c4 * kHq + h);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int64_t p = p0 + k * gs;
                if (p >= items) continue;
                const int64_t r = p / (kDv / 4);
                const int c0 = (int)(p % (kDv / 4)) * 4;
                float M = -3.0e38f;
                bool any = false;
#pragma unroll
                for (int s = 0; s < kFMaxSplits; ++s) {
                    if (s < splits && ml_l[k][s] > 0.f) {
                        M = fmaxf(M, ml_m[k][s]);
                        any = true;
                    }
                }
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                float den = 0.f;
                if (any) {
#pragma unroll
                    for (int s = 0; s < kFMaxSplits; ++s) {
                        if (s >= splits || !(ml_l[k][s] > 0.f)) continue;
                        const float wgt = exp2f(ml_m[k][s] - M);
                        den += wgt * ml_l[k][s];
                        acc[0] += wgt * o[k][s].x;
                        acc[1] += wgt * o[k][s].y;
                        acc[2] += wgt * o[k][s].z;
                        acc[3] += wgt * o[k][s].w;
                    }
                }
                const float inv = den > 0.f ? 1.f / den : 0.f;
                const int64_t base = (r * kHq + h) * (int64_t)kDv + c0;
                if (out_dtype == IDX_BF16) {
                    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out) + base;
                    *reinterpret_cast<__nv_bfloat162*>(ob) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
                    *reinterpret_cast<__nv_bfloat162*>(ob + 2) = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
                } else {
                    *reinterpret_cast<float4*>(static_cast<float*>(out) + base) =
                        make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // no cross-CTA traffic may target a CTA that has left
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    // the last CTA to finish returns the slot to zero for a later launch
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(fin, 1u) == gridDim.x - 1) {
            for (int i = 0; i < kFusedWords; ++i) atomicExch(&sync[i], 0u);
            __threadfence();
        }
    }
}

int fused_clusters_cache[64] = {};

template <typename TK, typename TQ>
cudaError_t launch_fused_t(const void* qi, const float* w, const void* k, int64_t k_row_stride, int64_t k_rows,
                           const Geom& g, int top_k, float* scores, int64_t score_row_stride, int32_t* idx,
                           int64_t idx_row_stride, int32_t* n_sel, const void* lat, int64_t lat_row_stride,
                           int64_t kv_rows, const void* qa, float scale, int splits, int kps, void* out,
                           int out_dtype, float* part_o, float* part_ml, uint32_t* ghist, int clusters,
                           cudaStream_t st) {
    static std::atomic<unsigned> next_slot{0};
    const int slot = (int)(next_slot.fetch_add(1u) % kFusedSlots);
    auto kern = decode_fused_kernel<TK, TQ>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kFSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float scale_log2 = scale * 1.4426950408889634f;
    // contiguous caches: key tiles by tensor-map loads (rows addressable by a 32-bit coordinate)
    CUtensorMap kmap;
    memset(&kmap, 0, sizeof(kmap));
    const int use_tma = !g.page_table && k_rows < (int64_t)INT32_MAX &&
                        make_key_tmap(&kmap, k, std::is_same<TK, __nv_bfloat16>::value, k_row_stride, k_rows, kFK);
    return cudaLaunchKernelEx(&cfg, kern, static_cast<const TQ*>(qi), w, static_cast<const TK*>(k), k_row_stride,
                              k_rows, g, top_k, scores, score_row_stride, idx, idx_row_stride, n_sel,
                              static_cast<const __nv_bfloat16*>(lat), lat_row_stride, kv_rows,
                              static_cast<const __nv_bfloat16*>(qa), scale_log2, splits, kps, out, out_dtype, part_o,
                              part_ml, ghist, slot, kmap, use_tma);
}

}  // namespace

// clusters of the fused decode kernel that can be resident at once (0: not launchable)
int fused_decode_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (fused_clusters_cache[dev]) return fused_clusters_cache[dev] > 0 ? fused_clusters_cache[dev] : 0;
    auto kern = decode_fused_kernel<__half, __nv_bfloat16>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmemBytes);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kFSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    fused_clusters_cache[dev] = n > 0 ? n : -1;
    return n > 0 ? n : 0;
}

// the fused decode step's workspace: the attention's split partials, then the rows' score histograms
size_t fused_decode_workspace_bytes(int64_t n_rows, int64_t idx_row_stride) {
    return (mla_workspace_bytes(n_rows, idx_row_stride) + 15) / 16 * 16 + (size_t)n_rows * 2048 * sizeof(uint32_t);
}

// whether the fused decode kernel takes this batch: decode rows, few and short enough
bool fused_decode_fits(int64_t n_rows, int max_n_kv, int top_k, int64_t idx_row_stride) {
    if (n_rows < 1 || n_rows > kFusedMaxRows || max_n_kv > sel::kMaxKeys || idx_row_stride > kMaxKps) return false;
    const int clusters = fused_decode_clusters();
    const int splits = mla_splits(n_rows, idx_row_stride);
    return clusters > 0 && splits <= kFMaxSplits && n_rows * (int64_t)splits <= clusters && top_k >= 1;
}

cudaError_t launch_decode_fused(const void* qi, int qi_dtype, const float* w, const void* k, int k_dtype,
                                int64_t k_row_stride, int64_t k_rows, const Geom& g, int top_k, float* scores,
                                int64_t score_row_stride, int32_t* idx, int64_t idx_row_stride, int32_t* n_sel,
                                const void* lat, int64_t lat_row_stride, int64_t kv_rows, const void* qa, float scale,
                                void* out, int out_dtype, void* ws, size_t ws_bytes, cudaStream_t st) {
    const int64_t n_rows = g.B;
    const int clusters = fused_decode_clusters();
    if (clusters <= 0) return cudaErrorNotSupported;
    const int splits = mla_splits(n_rows, idx_row_stride);
    const int64_t kps = ((idx_row_stride + splits - 1) / splits + kKeys - 1) / kKeys * kKeys;
    float* part_o = nullptr;
    float* part_ml = nullptr;
    const size_t need = fused_decode_workspace_bytes(n_rows, idx_row_stride);
    if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u)) return cudaErrorInvalidValue;
    if (splits > 1) {
        part_o = static_cast<float*>(ws);
        part_ml = part_o + (size_t)n_rows * splits * kHq * kDv;
    }
    uint32_t* ghist = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) +
                                                  (mla_workspace_bytes(n_rows, idx_row_stride) + 15) / 16 * 16);
#define LIDX_FUSED(TK_, TQ_)                                                                                   \
    return launch_fused_t<TK_, TQ_>(qi, w, k, k_row_stride, k_rows, g, top_k, scores, score_row_stride, idx, \
                                    idx_row_stride, n_sel, lat, lat_row_stride, kv_rows, qa, scale, splits,     \
                                    (int)kps, out, out_dtype, part_o, part_ml, ghist, clusters, st)
    if (k_dtype == IDX_F16) {
        if (qi_dtype == IDX_F16) LIDX_FUSED(__half, __half);
        if (qi_dtype == IDX_BF16) LIDX_FUSED(__half, __nv_bfloat16);
    } else if (k_dtype == IDX_BF16) {
        if (qi_dtype == IDX_BF16) LIDX_FUSED(__nv_bfloat16, __nv_bfloat16);
    }
#undef LIDX_FUSED
    return cudaErrorNotSupported;
}

}  // namespace lidx
