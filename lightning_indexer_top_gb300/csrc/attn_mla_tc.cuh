// Device code of the sparse MLA attention unit, shared by the attention kernel
// and the fused decode kernel.
//
// Sparse MLA attention on the 5th-generation tensor cores: 128 query heads
// over the selected rows of a 576-wide bf16 latent cache, value = the first
// 512 columns of the same row ("Gather OpenPangu DSA decode reads" and
// "openpangu: MLA-latent KV cache", ik_llama_opt commit log):
//     l[h, j] = scale * q[h] . c_j,   o[h] = sum_j softmax_j(l)[h, j] * c_j[0:512]
// over j in the row's selected positions.
//
// The output accumulator O [128 heads x 512] f32 fills all 512 TMEM columns,
// so one work unit (query row, key split) runs on a CLUSTER OF TWO CTAs:
//   rank 0: Q [128 x 576] bf16 lives in TMEM (288 columns) as the MMA A
//           operand; key tiles of 64 selected rows x 576 are gathered with
//           16-byte cp.async copies (128-byte swizzle) into a 3-stage ring;
//           S = Q K^T (M=128 heads, N=64 keys, K=576) goes to one of two TMEM
//           buffers; four softmax warps (thread = head) turn S into
//           P = 2^(S*scale*log2e - m) as bf16 and write P, the per-head
//           rescale factor, row sum and max straight into rank 1's packet
//           slot with st.async stores that complete the slot's barrier there.
//   rank 1: O lives in TMEM (512 columns); value tiles (the same rows, first
//           512 columns) are gathered into its own 2-stage ring; O += P V with
//           P as a K-major and V as an MN-major shared-memory operand (M=128,
//           N=256 x 2, K=16 x 4).  Four correction warps rescale their heads'
//           O rows when rank 0 raised a row maximum by more than 2^8 (rare
//           after the first tiles, so P stays <= 2^8 otherwise) and finally
//           write O / l, or the unnormalised partial (O, m, l) of a key split.
// Each CTA first turns its slice of the index list into cache rows and a
// validity bitmask in shared memory (rank 0 meanwhile puts Q into TMEM);
// padding and invalid indices gather a valid row and get p = 0.  Key splits
// (few query rows) are merged by a small combine kernel.  Both kernels take
// part in the decode launch chain (pdl_trigger / pdl_wait): everything up to
// the Q load runs while the previous kernel drains.  Every wait is bounded; a
// timeout records IDX_ERR_TIMEOUT and the cluster winds down.
#pragma once

#include "lidx_internal.cuh"
#include "sm100_ptx.cuh"

namespace lidx {
namespace {
using namespace sm100;

constexpr int kHq = 128;
constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kKeys = 64;                               // keys per tile
constexpr int kDkBlocks = kDk / 64;                     // 9 column blocks of 128 bytes
constexpr int kDvBlocks = kDv / 64;                     // 8
constexpr int kBlockBytes = kKeys * 128;                // one column block of a tile
constexpr int kKTileBytes = kDkBlocks * kBlockBytes;    // 73728
constexpr int kVTileBytes = kDvBlocks * kBlockBytes;    // 65536
constexpr int kStagesK = 3;                             // rank 0: key tiles in flight
constexpr int kStagesV = 2;                             // rank 1: value tiles in flight
constexpr int kPBytes = kHq * kKeys * 2;                // P tile, bf16, 128-byte swizzle K-major
constexpr int kPktBytes = kPBytes + 3 * kHq * 4;        // P tile + alpha, l, m per head
constexpr int kPktStride = 18432;                       // P tile + tail, 1024-aligned
constexpr int kMaxKps = 2048;                           // selected keys per split, at most
// Shared memory, per rank (the two CTAs share one launch size):
//   rank 0: [0, 3 x 72 KB) key-tile ring
//   rank 1: [0, 2 x 64 KB) value-tile ring, then the two P packet slots that
//           rank 0 writes directly
//   both:   from kTailOff the staged cache rows, the validity bits, barriers
constexpr int kPktOff = kStagesV * kVTileBytes;
constexpr int kTailOff = kStagesK * kKTileBytes;
static_assert(kPktOff + 2 * kPktStride <= kTailOff, "rank 1 layout");
#ifndef LIDX_MLA_WARPS
#define LIDX_MLA_WARPS 12
#endif
// Random 1152-byte row gathers by cp.async are bound by the copies each warp
// keeps in flight: one SM reaches ~22 GB/s with 4 issuing warps, ~33 GB/s with
// 8 and ~40 GB/s with 16 (about HBM speed over all SMs), so every warp without
// another role gathers.
constexpr int kThreads = 32 * LIDX_MLA_WARPS;
// Warp roles: 1 issues the MMAs, 2..5 (one per TMEM lane quarter) run the softmax (rank 0) or the
// O correction (rank 1), 0 and 6.. gather, except warp 9, which shares warp 1's scheduler: a busy
// third warp there slows the MMA issue (the tensor pipe then idles between instructions).
constexpr int kProducerWarps = LIDX_MLA_WARPS - 6;      // warps 0, 6..8, 10..
static_assert(kProducerWarps >= 1 && LIDX_MLA_WARPS >= 10 && LIDX_MLA_WARPS % 4 == 0,
              "warp roles; whole TMEM lane quarters");
constexpr int kTmemCols = 512;
constexpr int kSCol0 = 320;                             // rank 0: S buffers at 320 and 384 (Q at 0..287)
constexpr float kRescaleLog2 = 8.f;

struct PktTail {
    float alpha[kHq];
    float l[kHq];
    float m[kHq];
};
static_assert(kPBytes + sizeof(PktTail) <= kPktStride, "packet layout");

struct Ctl {
    uint64_t xfull[kStagesK];  // gathered tile landed (every producer lane arrives)
    uint64_t xempty[kStagesK]; // tile consumed by the MMAs
    uint64_t sfull[2];         // rank 0: S accumulator written
    uint64_t sempty[2];        // rank 0: S read by the softmax warps
    uint64_t qready;           // rank 0: Q stored in TMEM (its shared-memory staging free again)
    uint64_t qbulk;            // rank 0: Q's rows landed in shared memory
    uint64_t pfree[2];         // rank 0: rank 1's packet slot j consumed by its MMAs
    uint64_t pfull[2];         // rank 1: packet j landed (rank 0 posts its byte count, its stores complete it)
    uint64_t cdone[2];         // rank 1: O corrected for packet j
    uint64_t pvdone[2];        // rank 1: PV MMAs that read packet j completed
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kTailOff + kMaxKps * 4 + kMaxKps / 8 + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ void abort_cta(Ctl& c, int* status) {
    *(volatile int*)&c.abort = 1;
    flag(status, IDX_ERR_TIMEOUT);
}

__device__ __forceinline__ bool aborted(Ctl& c) { return *(volatile int*)&c.abort != 0; }

// the whole warp sees the same answer
__device__ __forceinline__ bool warp_aborted(Ctl& c) { return __any_sync(0xffffffffu, aborted(c)); }

struct Unit {
    int64_t r;        // query row
    int k0, k1;       // selected-key range [k0, k1) of this split
    int n_tiles;
    int b;            // the row's sequence
    int n_kv;         // keys of the sequence
    int64_t fallback; // an in-bounds cache row for padding keys
};

__device__ __forceinline__ Unit make_unit(int64_t unit, const Geom& g, const int32_t* n_sel, int64_t idx_row_stride,
                                          int64_t kv_rows, int splits, int kps) {
    Unit u;
    u.r = unit / splits;
    const int s = (int)(unit % splits);
    int ns = n_sel[u.r];
    if (ns < 0 || ns > idx_row_stride) ns = ns < 0 ? 0 : (int)idx_row_stride;
    u.k0 = s * kps;
    u.k1 = min(ns, u.k0 + kps);
    u.n_tiles = u.k1 > u.k0 ? (u.k1 - u.k0 + kKeys - 1) / kKeys : 0;
    const int b = (int)(u.r / g.T);
    u.n_kv = seq_n_kv(g, b);
    u.b = b;
    int64_t fb = g.page_table ? 0 : seq_row0(g, b);
    if (fb < 0) fb = 0;
    if (fb >= kv_rows) fb = kv_rows - 1;
    u.fallback = fb;
    return u;
}

// Producer warps (kProducerWarps of them, index p): gather each tile's 64 rows
// (the first kChunks*16 bytes of each row) with 16-byte cp.async copies into
// the 128-byte swizzled layout the MMA descriptors read: column block
// db = chunk/8 at db*8192, row at row*128, the 16-byte chunk at
// ((chunk%8) ^ (row%8))*16.  A warp instruction copies 512 contiguous bytes.
// Each producer lane hands its copies of tile t to xfull with a no-increment
// cp.async arrival, so a tile is announced the moment its bytes have landed
// and the producers go straight on to the next free stage.  The consumer
// orders the landed bytes before its MMAs with a proxy fence.
template <int kChunks, int kNStages, int kStageBytes>
__device__ __forceinline__ void gather_tiles(Ctl& c, uint8_t* xtiles, const __nv_bfloat16* lat,
                                             int64_t lat_row_stride, const Unit& u, const int32_t* rows_s,
                                             int p, int* status) {
    const int lane = threadIdx.x & 31;
    const char* base = reinterpret_cast<const char*>(lat);
    const int64_t row_bytes = lat_row_stride * 2;
    for (int t = 0; t < u.n_tiles; ++t) {
        const int stage = t % kNStages;
        const uint32_t ph = (uint32_t)((t / kNStages) & 1);
        if (warp_aborted(c) || !warp_wait(&c.xempty[stage], ph ^ 1)) {
            abort_cta(c, status);
            break;
        }
        const uint32_t dst0 = smem_u32(xtiles + (size_t)stage * kStageBytes);
        const int32_t* rr = rows_s + t * kKeys;
        // warp p copies rows p, p + kProducerWarps, ...; lane l the 16-byte chunks l, l + 32, l + 64 of
        // each (a warp instruction covers 512 contiguous bytes of a row; the swizzle XORs bits 4-6)
#pragma unroll 2
        for (int row = p; row < kKeys; row += kProducerWarps) {
            const char* src = base + (int64_t)rr[row] * row_bytes;
            const uint32_t rb = dst0 + row * 128, x = (uint32_t)(row & 7) << 4;
#pragma unroll
            for (int k = 0; k < (kChunks + 31) / 32; ++k) {
                const int cc = lane + 32 * k;
                if (cc < kChunks) cp_async16(rb + ((uint32_t)((cc >> 3) * kBlockBytes + ((cc & 7) << 4)) ^ x), src + cc * 16);
            }
        }
        cp_async_mbar_arrive_noinc(&c.xfull[stage]);
    }
    // no copy may still be writing when the CTA winds down
    cp_async_wait_all();
}

// this CTA's pieces of the unit's shared memory (the base 1024-byte aligned)
struct MlaSmem {
    uint8_t* xtiles;      // K tiles (rank 0) / V tiles (rank 1)
    uint8_t* pkts;        // rank 1: P packets (rank 0 writes them)
    int32_t* rows_s;      // cache row of each selected key
    uint32_t* vmask;      // bit = key index is valid
    Ctl* c;
};

__device__ __forceinline__ MlaSmem mla_smem(uint8_t* smem) {
    MlaSmem s;
    s.xtiles = smem;
    s.pkts = smem + kPktOff;
    s.rows_s = reinterpret_cast<int32_t*>(smem + kTailOff);
    s.vmask = reinterpret_cast<uint32_t*>(s.rows_s + kMaxKps);
    s.c = reinterpret_cast<Ctl*>(s.vmask + kMaxKps / 32);
    return s;
}

// one thread: the unit's barriers
__device__ __forceinline__ void mla_init(Ctl& c) {
    for (int i = 0; i < kStagesK; ++i) {
        mbar_init(&c.xfull[i], 32 * kProducerWarps);
        mbar_init(&c.xempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
        mbar_init(&c.sfull[i], 1);
        mbar_init(&c.sempty[i], 4);
        mbar_init(&c.pfree[i], 1);
        mbar_init(&c.pfull[i], 1);
        mbar_init(&c.cdone[i], 4);
        mbar_init(&c.pvdone[i], 1);
    }
    mbar_init(&c.qready, 4);
    mbar_init(&c.qbulk, 1);
    mbar_init(&c.done, 1);
    c.abort = 0;
    fence_mbar_init();
}

// rank 0, warps 2..5 (thread = head): Q of query row qrow into TMEM columns 0..287 (the QK^T MMA's A
// operand), then an arrival on qready.  Each thread bulk-copies its head's row (1152 contiguous bytes)
// into the key ring, not yet in use, at a pitch of kQPitch bytes (rows 4 banks apart, so a warp's
// 16-byte reads of its 32 rows do not collide), and moves it to TMEM a column block at a time.  The
// key producers start only after qready (the staging area is their first stages).
constexpr int kQPitch = kDk * 2 + 16;
static_assert(kHq * kQPitch <= kStagesK * kKTileBytes, "Q staging inside the key ring");
__device__ __forceinline__ void mla_load_q(Ctl& c, uint8_t* xtiles, uint32_t tmem, const __nv_bfloat16* __restrict__ q,
                                           int64_t qrow) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int h = quad * 32 + lane;
    uint8_t* row = xtiles + h * kQPitch;
    if (warp == 2 && lane == 0) mbar_arrive_expect_tx(&c.qbulk, kHq * kDk * 2);
    bulk_load(row, q + (qrow * kHq + h) * (int64_t)kDk, kDk * 2, &c.qbulk);
    const bool ok = warp_wait(&c.qbulk, 0);
    const uint4* src = reinterpret_cast<const uint4*>(row);
#pragma unroll
    for (int cb = 0; cb < kDkBlocks; ++cb) {
        uint32_t regs[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 x = ok ? src[cb * 8 + i] : make_uint4(0u, 0u, 0u, 0u);
            regs[4 * i] = x.x;
            regs[4 * i + 1] = x.y;
            regs[4 * i + 2] = x.z;
            regs[4 * i + 3] = x.w;
        }
        tmem_st_32x32b_x32(tmem + lane_off + cb * 32, regs);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.qready);
}

__device__ __forceinline__ bool mla_q_warp(uint32_t rank) {
    const int warp = threadIdx.x >> 5;
    return rank == 0 && warp >= 2 && warp <= 5;
}

// every warp but the Q loaders: the unit's selected keys -> cache rows + validity bits in shared
// memory (32 keys per warp step, the index loads of a warp issued together)
__device__ __forceinline__ void mla_stage_rows(const MlaSmem& sm, uint32_t rank, const Unit& u, const Geom& g,
                                           const int32_t* idx, int64_t idx_row_stride, int64_t kv_rows) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* rows_s = sm.rows_s;
    uint32_t* vmask = sm.vmask;
    const int n_st = rank == 0 ? kThreads / 32 - 4 : kThreads / 32;
    const int si = rank == 0 && warp > 5 ? warp - 4 : warp;
    const int n_words = u.n_tiles * (kKeys / 32);
    const int64_t row0 = g.page_table ? 0 : seq_row0(g, u.b);   // contiguous caches: read once
    constexpr int kBatch = 8;
    for (int w0 = si; w0 < n_words; w0 += kBatch * n_st) {
        int pos[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int j = u.k0 + (w0 + k * n_st) * 32 + lane;
            pos[k] = (w0 + k * n_st < n_words && j < u.k1) ? idx[u.r * idx_row_stride + j] : -1;
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int wd = w0 + k * n_st;
            if (wd >= n_words) break;
            const int j = u.k0 + wd * 32 + lane;
            bool valid = false;
            int64_t row = u.fallback;
            if (j < u.k1) {
                const int64_t rr = (pos[k] >= 0 && pos[k] < u.n_kv)
                                       ? (g.page_table ? key_row(g, u.b, pos[k]) : row0 + pos[k]) : -1;
                if (rr >= 0 && rr < kv_rows) {
                    valid = true;
                    row = rr;
                } else if (rank == 0) {
                    flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                }
            }
            rows_s[wd * 32 + lane] = (int32_t)row;
            const uint32_t bits = __ballot_sync(0xffffffffu, valid);
            if (lane == 0) vmask[wd] = bits;
        }
    }
}

// the unit after its Q load and index staging (both CTAs past a cluster_sync): gathers,
// QK^T, softmax, PV and the output (or the split's partial result)
__device__ __forceinline__ void mla_run(const MlaSmem& sm, uint32_t tmem, uint32_t rank, const Unit& u, int64_t unit,
                                        const __nv_bfloat16* __restrict__ lat, int64_t lat_row_stride, const Geom& g,
                                        float scale_log2, int splits, void* __restrict__ out, int out_dtype,
                                        float* __restrict__ part_o, float* __restrict__ part_ml) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    uint8_t* xtiles = sm.xtiles;
    uint8_t* pkts = sm.pkts;
    const int32_t* rows_s = sm.rows_s;
    const uint32_t* vmask = sm.vmask;
    Ctl& c = *sm.c;
    const int producer = warp == 0 ? 0 : (warp >= 6 && warp != 9 ? warp - (warp > 9 ? 6 : 5) : -1);   // index or -1
    if (rank == 0) {
        if (producer >= 0) {
            // Q's staging area is the ring's first stages: gather once Q is in TMEM
            if (u.n_tiles > 0 && !warp_wait(&c.qready, 0)) abort_cta(c, g.status);
            gather_tiles<kDkBlocks * 8, kStagesK, kKTileBytes>(c, xtiles, lat, lat_row_stride, u, rows_s, producer,
                                                               g.status);
        } else if (warp == 1) {
            if (lane == 0) {
                // ---------------------------------------------------- S = Q K^T issuer
                const uint32_t idesc = idesc_f16_f32_major(kHq, kKeys, 1, 0, 0);
                bool ok = u.n_tiles == 0 || mbar_wait(&c.qready, 0);
                if (!ok) abort_cta(c, g.status);
                tc_fence_after();
                for (int t = 0; ok && t < u.n_tiles; ++t) {
                    const int stage = t % kStagesK, sb = t & 1;
                    if (aborted(c)) break;
                    if (!mbar_wait(&c.xfull[stage], (uint32_t)((t / kStagesK) & 1)) ||
                        !mbar_wait(&c.sempty[sb], (uint32_t)((t >> 1) & 1) ^ 1)) {
                        abort_cta(c, g.status);
                        break;
                    }
                    fence_proxy_async_smem();   // cp.async bytes (generic proxy) before the MMA reads them
                    tc_fence_after();
                    const uint32_t kb = smem_u32(xtiles + (size_t)stage * kKTileBytes);
                    const uint32_t d = tmem + kSCol0 + sb * kKeys;
#pragma unroll 4
                    for (int ks = 0; ks < kDk / 16; ++ks) {
                        const uint64_t bd = desc_sw128_kmajor(kb + (ks >> 2) * kBlockBytes + (ks & 3) * 32, 1024);
                        mma_f16_ts(d, tmem + ks * 8, bd, idesc, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&c.xempty[stage]);
                    mma_commit(&c.sfull[sb]);
                }
                mma_commit(&c.done);
                mbar_wait(&c.done, 0);
            }
            __syncwarp();
        } else if (warp >= 2 && warp <= 5) {
            // ---------------------------------------------------------- softmax (thread = head); P goes
            // straight into rank 1's packet slot by asynchronous stores that complete its barrier
            const int h = quad * 32 + lane;
            float m_used = 0.f, lsum = 0.f;
            bool has_m = false;
            for (int t = 0; t < u.n_tiles; ++t) {
                const int sb = t & 1, j = t & 1;
                const uint32_t ph = (uint32_t)((t >> 1) & 1);
                const uint32_t ma = vmask[2 * t], mb = vmask[2 * t + 1];
                if (warp_aborted(c) || !warp_wait(&c.sfull[sb], ph)) {
                    abort_cta(c, g.status);
                    break;
                }
                tc_fence_after();
                float s0[32], s1[32];
                tmem_ld_32x32b_x32(tmem + lane_off + kSCol0 + sb * kKeys, s0);
                tmem_ld_32x32b_x32(tmem + lane_off + kSCol0 + sb * kKeys + 32, s1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.sempty[sb]);

                // the tile's largest scaled logit: for a full tile and a positive scale, the scaled
                // largest logit (the same value: rounding a product by a positive factor is monotone)
                const bool full = (ma & mb) == 0xffffffffu;
                float mt = -3.0e38f;
                if (full && scale_log2 > 0.f) {
                    float a0 = fmaxf(s0[0], s0[1]), a1 = fmaxf(s0[2], s0[3]);
                    float a2 = fmaxf(s1[0], s1[1]), a3 = fmaxf(s1[2], s1[3]);
#pragma unroll
                    for (int i = 4; i < 32; i += 4) {
                        a0 = fmaxf(a0, fmaxf(s0[i], s0[i + 1]));
                        a1 = fmaxf(a1, fmaxf(s0[i + 2], s0[i + 3]));
                        a2 = fmaxf(a2, fmaxf(s1[i], s1[i + 1]));
                        a3 = fmaxf(a3, fmaxf(s1[i + 2], s1[i + 3]));
                    }
                    mt = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * scale_log2;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if ((ma >> i) & 1u) mt = fmaxf(mt, s0[i] * scale_log2);
                        if ((mb >> i) & 1u) mt = fmaxf(mt, s1[i] * scale_log2);
                    }
                }
                float alpha = 1.f;
                if ((ma | mb) != 0u) {
                    if (!has_m) {
                        m_used = mt;
                        has_m = true;
                    } else if (mt > m_used + kRescaleLog2) {
                        alpha = ex2_approx(m_used - mt);
                        lsum *= alpha;
                        m_used = mt;
                    }
                }
                // p = 2^(s * scale_log2 - m) with one rounding of the exponent's argument (FMA)
                uint32_t pk[32];
                float psum = 0.f;
                const float nm = -m_used;
                const uint32_t ka = full ? 0xffffffffu : ma, kb = full ? 0xffffffffu : mb;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float e0 = ex2_approx(fmaf(s0[2 * i], scale_log2, nm));
                    const float e1 = ex2_approx(fmaf(s0[2 * i + 1], scale_log2, nm));
                    const float e2 = ex2_approx(fmaf(s1[2 * i], scale_log2, nm));
                    const float e3 = ex2_approx(fmaf(s1[2 * i + 1], scale_log2, nm));
                    const float p0 = ((ka >> (2 * i)) & 1u) ? e0 : 0.f;
                    const float p1 = ((ka >> (2 * i + 1)) & 1u) ? e1 : 0.f;
                    const float p2 = ((kb >> (2 * i)) & 1u) ? e2 : 0.f;
                    const float p3 = ((kb >> (2 * i + 1)) & 1u) ? e3 : 0.f;
                    psum += (p0 + p1) + (p2 + p3);
                    const __nv_bfloat162 a = __floats2bfloat162_rn(p0, p1);
                    const __nv_bfloat162 bb = __floats2bfloat162_rn(p2, p3);
                    pk[i] = *reinterpret_cast<const uint32_t*>(&a);
                    pk[16 + i] = *reinterpret_cast<const uint32_t*>(&bb);
                }
                lsum += psum;

                // rank 1's slot j is free once its MMAs of tile t-2 have completed
                if (!warp_wait(&c.pfree[j], ph ^ 1)) {
                    abort_cta(c, g.status);
                    break;
                }
                const uint32_t slot = mapa(pkts + j * kPktStride, 1);
                const uint32_t rbar = mapa(&c.pfull[j], 1);
                if (h == 0) mbar_arrive_expect_tx_remote(rbar, kPktBytes);
                const uint32_t rowp = slot + (uint32_t)((h >> 3) * 1024 + (h & 7) * 128);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_async_v4(rowp + ((ch ^ (h & 7)) << 4),
                                make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]), rbar);
                const uint32_t tail = slot + kPBytes + (uint32_t)h * 4;
                st_async_f32(tail + offsetof(PktTail, alpha), alpha, rbar);
                st_async_f32(tail + offsetof(PktTail, l), lsum, rbar);
                st_async_f32(tail + offsetof(PktTail, m), m_used, rbar);
            }
            // rank 1's last arrivals on pfree land before this CTA may leave
            const int n = min(u.n_tiles, 2);
            for (int t = u.n_tiles - n; t < u.n_tiles; ++t)
                if (!warp_aborted(c)) warp_wait(&c.pfree[t & 1], (uint32_t)((t >> 1) & 1));
        }
    } else {
        if (producer >= 0) {
            gather_tiles<kDvBlocks * 8, kStagesV, kVTileBytes>(c, xtiles, lat, lat_row_stride, u, rows_s, producer,
                                                               g.status);
        } else if (warp == 1) {
            if (lane == 0) {
                const uint32_t idesc = idesc_f16_f32_major(kHq, 256, 1, 0, 1);
                for (int t = 0; t < u.n_tiles; ++t) {
                    const int stage = t % kStagesV, j = t & 1;
                    const uint32_t ph = (uint32_t)((t >> 1) & 1);
                    if (aborted(c)) break;
                    if (!mbar_wait(&c.xfull[stage], (uint32_t)((t / kStagesV) & 1)) || !mbar_wait(&c.cdone[j], ph)) {
                        abort_cta(c, g.status);
                        break;
                    }
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t pb = smem_u32(pkts + j * kPktStride);
                    const uint32_t vb = smem_u32(xtiles + (size_t)stage * kVTileBytes);
#pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks) {
                        const uint64_t ad = desc_sw128_kmajor(pb + ks * 32, 1024);
#pragma unroll
                        for (int nh = 0; nh < 2; ++nh) {
                            const uint64_t bd = desc_sw128_mnmajor(vb + nh * 4 * kBlockBytes + ks * 2 * 1024,
                                                                   kBlockBytes, 1024);
                            mma_f16_ss(tmem + nh * 256, ad, bd, idesc, (t > 0 || ks > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(&c.xempty[stage]);
                    mma_commit(&c.pvdone[j]);
                    mma_commit_multicast(&c.pfree[j], (uint16_t)0x1);
                }
                mma_commit(&c.done);
                mbar_wait(&c.done, 0);
            }
            __syncwarp();
        } else if (warp >= 2 && warp <= 5) {
            // ---------------------------------------------------------- O correction (thread = head)
            const int h = quad * 32 + lane;
            for (int t = 0; t < u.n_tiles; ++t) {
                const int j = t & 1;
                const uint32_t ph = (uint32_t)((t >> 1) & 1);
                if (warp_aborted(c) || !warp_wait_cluster(&c.pfull[j], ph)) {
                    abort_cta(c, g.status);
                    break;
                }
                const PktTail& tail = *reinterpret_cast<const PktTail*>(pkts + j * kPktStride + kPBytes);
                const float a = tail.alpha[h];
                if (t > 0 && __any_sync(0xffffffffu, a != 1.f)) {
                    const int tp = t - 1;
                    if (!warp_wait(&c.pvdone[tp & 1], (uint32_t)((tp >> 1) & 1))) {
                        abort_cta(c, g.status);
                        break;
                    }
                    tc_fence_after();
                    for (int cb = 0; cb < kDv / 32; ++cb) {
                        float v[32];
                        tmem_ld_32x32b_x32(tmem + lane_off + cb * 32, v);
                        tmem_ld_wait();
                        uint32_t w[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * a);
                        tmem_st_32x32b_x32(tmem + lane_off + cb * 32, w);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.cdone[j]);
            }
        }
        // ------------------------------------------------------------------ output: every warp, three
        // per TMEM lane quarter (thread = head), warp w taking the quarter's column blocks w/4, w/4 + 3, ...
        const int h = quad * 32 + lane;
        const int part = warp >> 2;
        float lsum = 0.f, mrow = 0.f;
        const bool have = u.n_tiles > 0 && !warp_aborted(c);
        if (have) {
            // every PV MMA of the unit completed: `done` completes once per unit, so a warp that
            // arrives here early (a producer) cannot mistake an older phase for it, as it could
            // with the per-packet barriers
            const int tl = u.n_tiles - 1;
            if (!warp_wait(&c.done, 0u)) {
                abort_cta(c, g.status);
            } else {
                tc_fence_after();
                const PktTail& tail = *reinterpret_cast<const PktTail*>(pkts + (tl & 1) * kPktStride + kPBytes);
                lsum = tail.l[h];
                mrow = tail.m[h];
            }
        }
        const bool read_o = have && !warp_aborted(c);
        if (splits == 1) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const int64_t base = (u.r * kHq + h) * (int64_t)kDv;
            for (int cb = part; cb < kDv / 32; cb += kThreads / 128) {
                float v[32];
                if (read_o) {
                    tmem_ld_32x32b_x32(tmem + lane_off + cb * 32, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
                if (out_dtype == IDX_BF16) {
                    // the warp's 32 heads x 32 columns pass through shared memory (the value-tile ring is
                    // idle once every PV MMA completed; rows of 80 bytes, conflict-free 16-byte stores), so
                    // that each store instruction writes eight heads' 64-byte row segments whole instead
                    // of 32 scattered 16-byte pieces
                    uint8_t* tw = xtiles + warp * (32 * 80);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 pk;
                        __nv_bfloat162 a0 = __floats2bfloat162_rn(v[8 * q4] * inv, v[8 * q4 + 1] * inv);
                        __nv_bfloat162 a1 = __floats2bfloat162_rn(v[8 * q4 + 2] * inv, v[8 * q4 + 3] * inv);
                        __nv_bfloat162 a2 = __floats2bfloat162_rn(v[8 * q4 + 4] * inv, v[8 * q4 + 5] * inv);
                        __nv_bfloat162 a3 = __floats2bfloat162_rn(v[8 * q4 + 6] * inv, v[8 * q4 + 7] * inv);
                        pk.x = *reinterpret_cast<uint32_t*>(&a0);
                        pk.y = *reinterpret_cast<uint32_t*>(&a1);
                        pk.z = *reinterpret_cast<uint32_t*>(&a2);
                        pk.w = *reinterpret_cast<uint32_t*>(&a3);
                        *reinterpret_cast<uint4*>(tw + lane * 80 + q4 * 16) = pk;
                    }
                    __syncwarp();
                    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out) + (u.r * kHq + quad * 32) * (int64_t)kDv + cb * 32;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int rr = 8 * j + (lane >> 2), ch = lane & 3;
                        *reinterpret_cast<uint4*>(ob + (int64_t)rr * kDv + ch * 8) =
                            *reinterpret_cast<const uint4*>(tw + rr * 80 + ch * 16);
                    }
                    __syncwarp();
                } else {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + base + cb * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        dst[q4] = make_float4(v[4 * q4] * inv, v[4 * q4 + 1] * inv, v[4 * q4 + 2] * inv,
                                              v[4 * q4 + 3] * inv);
                }
            }
        } else {
            // partial O as [unit][column / 4][head][4]: for each 4 columns the warp's 32 heads are
            // 512 contiguous bytes (one 16-byte store per head, coalesced across the warp)
            float4* po = reinterpret_cast<float4*>(part_o + unit * (int64_t)kDv * kHq) + h;
            for (int cb = part; cb < kDv / 32; cb += kThreads / 128) {
                float v[32];
                if (read_o) {
                    tmem_ld_32x32b_x32(tmem + lane_off + cb * 32, v);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    po[(int64_t)(cb * 8 + q4) * kHq] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
            }
            if (part == 0) {
                part_ml[(unit * kHq + h) * 2] = mrow;
                part_ml[(unit * kHq + h) * 2 + 1] = read_o ? lsum : 0.f;
            }
        }
    }
}

}  // namespace
}  // namespace lidx
