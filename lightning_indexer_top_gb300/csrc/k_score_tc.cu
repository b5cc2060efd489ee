// Lightning-indexer scores of decode query rows on the 5th-generation tensor
// cores (H = 64 indexer heads, d = 128, 16-bit key cache):
//     s[r, j] = sum_h w[r, h] * max(0, q[r, h, :] . k[j, :])
// (ik_llama_opt commit log, "openpangu: DSA lightning indexer + SWA schedule";
// ReLU per head before the head sum, llama.cpp commit c88c916636, QSA commit
// message).  The pages' fused indexer ("Route DSA indexer selection through
// ggml_indexer_topk", same log) avoids a per-head score tensor; here the
// per-head dot products live only in TMEM.
//
// Why tensor cores for decode: a 256-byte F16 key row costs 64*128 MACs, 64
// flop/byte; streaming keys at HBM speed needs ~430 TFLOP/s, several times
// what the CUDA cores deliver.  Per tile of 128 keys one MMA chain
//     D[128 keys x 64 heads] = K_tile[128 x 128] . Q^T[128 x 64]
// (M = 128, N = 64, K = 128 as 8 steps of 16) puts one key per TMEM lane, so
// the epilogue thread that owns a lane applies ReLU, weights and sums its 64
// head columns with no cross-thread reduction.
//
// Persistent CTAs (one per SM) with dynamic scheduling.  The work is split into
// chunks of up to 8 key tiles of one query row; CTAs take chunks in order from
// a device counter, so SMs that stream faster take more chunks (on GB300 some
// SMs sustain ~15% less bandwidth than others, and an even static split ends
// on the slowest).  Chunks are numbered row by row through a prefix of the
// rows' chunk counts that the CTA builds in shared memory; above kMaxPrefixRows
// rows a chunk is a whole row.  Warp roles:
//   warp 0      producer (one lane): takes a chunk, publishes its descriptor
//               (row, first tile, end tile) in a small ring, and issues the TMA
//               loads of its key tiles (two 64-column boxes, 128-byte swizzle)
//               into a 5-stage ring.
//   warp 1      TMEM owner and MMA issuer (one lane): 8 tcgen05.mma per tile
//               into one of 4 TMEM accumulators of 64 columns.
//   warps 2-5   epilogue: tcgen05.ld of the tile's [128 x 64] accumulator, one
//               key per thread, then sum_h w_h*relu(d_h) and a coalesced store.
//   warp 6      q stager: converts each chunk's query row q to the key dtype
//               with 16-byte loads and writes it, swizzled, into one of two q
//               buffers (the MMA's B operand), a chunk ahead of the MMAs.
// With a histogram buffer (the fused score + top-k), the epilogue also counts
// every score of a row into a 2048-bin histogram of its order key's top 11
// bits: each warp folds equal bins (match_any) into a shared-memory histogram
// of the chunk (two counts of 16 bits per word, two buffers used in turn), and
// when all four epilogue warps have finished the chunk (an mbarrier), each
// flushes its quarter of the nonzero bins to the row's global histogram with
// atomic adds and clears them.  The launch zeroes the histograms itself: each
// CTA clears a slice in its prologue and counts itself on the slot's third
// counter, and the epilogue adds nothing before every CTA has (a grid barrier,
// safe because the persistent CTAs, one per SM, are all resident once the
// previous kernel has drained; the wait is bounded, and a timeout leaves the
// histogram incomplete, which the select detects and bypasses).
// Every wait is bounded; a timeout records IDX_ERR_TIMEOUT and the CTA winds
// down (drains its TMA loads and MMAs, frees TMEM) instead of hanging.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "lidx_internal.cuh"
#include "sm100_ptx.cuh"

namespace lidx {

// chunk counters of the decode scorer: [next chunk, CTAs finished, CTAs whose
// histogram slice is zeroed] per slot; a launch uses one slot (round-robin on
// the host) and its last CTA zeroes it
constexpr int kSchedSlots = 1024;
__device__ unsigned int g_score_sched[kSchedSlots][3];

namespace {
using namespace sm100;

// the fused select's inputs the decode scorer produces (all NULL: plain scoring)
struct HistOut {
    uint32_t* hist;       // [rows][2048] counts of the order keys' top 11 bits
    uint32_t* cnt;        // [rows] candidate counters of the select, zeroed here
};

constexpr int kTileKeys = 128;
constexpr int kH = 64;
constexpr int kD = 128;
#ifndef LIDX_SCORE_STAGES
#define LIDX_SCORE_STAGES 5
#endif
#ifndef LIDX_SCORE_CHUNK
#define LIDX_SCORE_CHUNK 8
#endif
constexpr int kStages = LIDX_SCORE_STAGES;
constexpr int kAcc = 4;
constexpr int kTmemCols = kAcc * kH;                 // 256
constexpr int kTmemColsQ8 = 512;                     // int8 keys: + the widened A tiles (64 columns each) at 256
constexpr int kTileBytes = kTileKeys * kD * 2;       // 32 KB
constexpr int kHalfBytes = kTileBytes / 2;           // one 64-column box
constexpr int kQBytes = kH * kD * 2;                 // 16 KB
constexpr int kQHalfBytes = kQBytes / 2;
constexpr int kThreads = 224;                        // 16-bit keys: 7 warps
constexpr int kThreadsQ8 = 352;                      // int8 keys: + 4 converter warps
#ifndef LIDX_Q8_RAW_STAGES
#define LIDX_Q8_RAW_STAGES 8
#endif
#ifndef LIDX_Q8_CONV_STAGES
#define LIDX_Q8_CONV_STAGES 2
#endif
constexpr int kRawStages = LIDX_Q8_RAW_STAGES;       // int8 keys: TMA ring of 16 KB code tiles
constexpr int kConvStages = LIDX_Q8_CONV_STAGES;     // int8 keys: widened tiles for the MMA (in TMEM)
constexpr int kRawPitchInline = kD + 16;             // int8 rows with their scale inline: 128 codes + f32 + pad
constexpr int kRawTileBytes = kTileKeys * kRawPitchInline;   // 18 KB stage (16 KB used without inline scales)
constexpr int kSRing = 8;                            // int8 keys, inline scales: tiles of scales in flight
constexpr int kChunkTiles = LIDX_SCORE_CHUNK;        // key tiles (32 KB each) per chunk, at most
constexpr int kRing = 4;                             // chunk descriptors in flight
#ifndef LIDX_SCORE_QBUFS
#define LIDX_SCORE_QBUFS 3
#endif
constexpr int kQBufs = LIDX_SCORE_QBUFS;             // staged q rows (one per chunk) in flight
constexpr int kMaxPrefixRows = 1024;
constexpr int kHistWords = 1024;                     // 2048 bins, two 16-bit counts per word

struct Chunk {
    int64_t row;      // query row, -1 = no more chunks
    int t0, t1;       // key tiles [t0, t1) of the row
};

struct Ctl {
    uint64_t full[8];          // TMA tile landed (16-bit keys: the MMA's tiles; int8: code tiles)
    uint64_t empty[8];
    uint64_t afull[kConvStages];   // int8 keys: widened tile written
    uint64_t aempty[kConvStages];  // int8 keys: widened tile read by the MMAs
    uint64_t sfull[kSRing];        // int8 keys, inline scales: a tile's scales staged by the converters
    uint64_t sempty[kSRing];       // ... and read by the epilogue
    uint64_t tfull[kAcc];
    uint64_t tempty[kAcc];
    uint64_t qfull[kQBufs];
    uint64_t qempty[kQBufs];
    uint64_t cfull[kRing];
    uint64_t cempty[kRing];
    uint64_t done;
    uint64_t hdone[2];             // fused top-k: the 4 epilogue warps finished adding a chunk's counts
    Chunk chunk[kRing];
    uint32_t tmem_base;
    int abort;
    int n_chunks;
};

static_assert(kStages <= 8 && kRawStages <= 8, "barrier arrays");
constexpr int kChunkReaders = 1 + 4 + 1;             // MMA lane, 4 epilogue warps, q stager (+4 converters)
template <bool Q8>
constexpr size_t smem_bytes() {
    return 1024 + (Q8 ? (size_t)kRawStages * kRawTileBytes : (size_t)kStages * kTileBytes) +
           kQBufs * kQBytes + sizeof(Ctl) + (2 * kMaxPrefixRows + 1) * sizeof(int) +
           (Q8 ? kSRing * kTileKeys * sizeof(float) : 2 * kHistWords * sizeof(uint32_t));
}
constexpr size_t kSmemBytes = smem_bytes<false>();
static_assert(smem_bytes<true>() <= 232448 && smem_bytes<false>() <= 232448, "shared memory");

template <typename T> constexpr bool kIsBF16 = false;
template <> constexpr bool kIsBF16<__nv_bfloat16> = true;

__device__ __forceinline__ int row_tiles(int n_keys) { return (n_keys + kTileKeys - 1) / kTileKeys; }
__device__ __forceinline__ int row_chunks(int n_keys, int ct) {
    return (row_tiles(n_keys) + ct - 1) / ct;
}

// one query row's q [64 heads x 128] -> key dtype TK in the MMA's B layout
// (two 64-column halves, rows of 128 bytes, 16-byte chunks swizzled by row),
// 16-byte loads and stores, the warp's 32 lanes over the 1024 chunks
// (all loads of a batch are issued before the first conversion: two round
// trips per row for 16-bit q, four for f32)
// Returns true if a value overflowed the key type (a bf16 q element of magnitude >= 65520 staged
// as f16 becomes +-inf); below f16's normal range values keep their f16 rounding (an error of at
// most 2^-25 per element).
template <typename TK, typename TQ>
__device__ __forceinline__ bool stage_q_row(const TQ* __restrict__ qrow, uint8_t* qdst, int lane) {
    bool overflow = false;
    constexpr int kPerLane = kH * kD / 8 / 32;                   // 32 chunks of 8 elements
    constexpr int kBatch = sizeof(TQ) == 2 ? 16 : 8;
#pragma unroll
    for (int b0 = 0; b0 < kPerLane; b0 += kBatch) {
        uint4 raw[kBatch * sizeof(TQ) / 2];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int ch = (b0 + i) * 32 + lane;
            const uint4* src = reinterpret_cast<const uint4*>(qrow + ch * 8);
            if constexpr (sizeof(TQ) == 2) {
                raw[i] = src[0];
            } else {
                raw[2 * i] = src[0];
                raw[2 * i + 1] = src[1];
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int ch = (b0 + i) * 32 + lane;
            const int h = ch >> 4, cc = ch & 15;
            const int half = cc >> 3, c8 = cc & 7;
            TK vals[8];
            if constexpr (sizeof(TQ) == 2) {
                const TQ* e = reinterpret_cast<const TQ*>(&raw[i]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float x = to_f32(e[j]);
                    vals[j] = from_f32<TK>(x);
                    if constexpr (std::is_same<TK, __half>::value) overflow |= fabsf(x) >= 65520.f;
                }
            } else {
                const float* e = reinterpret_cast<const float*>(&raw[2 * i]);
#pragma unroll
                for (int j = 0; j < 8; ++j) vals[j] = from_f32<TK>(e[j]);
            }
            uint8_t* dst = qdst + half * kQHalfBytes + h * 128 + ((c8 ^ (h & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(vals);
        }
    }
    return overflow;
}

// chunk number `ch` -> (row, tiles); prefix mode: pre[i] = chunks of the rows
// before row i, nvis[i] = visible keys of row i (both in shared memory)
__device__ __forceinline__ Chunk chunk_of(const Geom& g, const int* pre, const int* nvis, int64_t n_rows,
                                          bool prefix, int ch, int n_chunks, int ct) {
    Chunk d;
    d.row = -1;
    d.t0 = d.t1 = 0;
    if (ch >= n_chunks) return d;
    if (prefix) {
        int lo = 0, hi = (int)n_rows;   // last row with pre[row] <= ch
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= ch) lo = mid;
            else hi = mid;
        }
        d.row = lo;
        const int nt = row_tiles(nvis[lo]);
        d.t0 = (ch - pre[lo]) * ct;
        d.t1 = min(nt, d.t0 + ct);
    } else {
        d.row = ch;
        d.t0 = 0;
        d.t1 = row_tiles(row_n_vis(g, ch));
    }
    return d;
}

__device__ __forceinline__ void abort_cta(Ctl& c, const Geom& g) {
    *(volatile int*)&c.abort = 1;
    flag(g.status, IDX_ERR_TIMEOUT);
}

// the whole warp sees the same answer
__device__ __forceinline__ bool warp_aborted(Ctl& c) { return __any_sync(0xffffffffu, *(volatile int*)&c.abort != 0); }

// a consumer's next chunk descriptor (the whole warp waits; lane 0 releases the slot)
__device__ __forceinline__ bool warp_next_chunk(Ctl& c, int k, Chunk& d) {
    const int slot = k % kRing;
    if (!warp_wait(&c.cfull[slot], (uint32_t)((k / kRing) & 1))) return false;
    d = c.chunk[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&c.cempty[slot]);
    return true;
}

// int8 codes of key row t of a 128-key tile -> f16, written into TMEM lane t as
// the MMA's A operand (column c holds elements 2c and 2c+1).  Thread t of the
// four converter warps owns TMEM lane t.  The TMA lands the code rows in the
// 128-byte swizzle (chunk i of row t at (i ^ (t % 8)) * 16), so the 8 threads
// of a shared-memory phase hit 8 different bank groups.
// The widening is exact and stays on the integer/half ALUs: a code b becomes
// the unsigned byte u = b + 128 (xor 0x80), the f16 with bit pattern 0x6400 | u
// is 1024 + u, and subtracting 1152 leaves b (every step exact in f16).
// With inline scales the rows are 144 bytes apart (no swizzle), which already
// spreads 8 consecutive rows over 8 bank groups.
__device__ __forceinline__ void widen_row_tmem(const uint8_t* __restrict__ raw, uint32_t taddr, int t,
                                               bool inline_scale) {
    // row t's 128 codes (eight 16-byte chunks; in the 128-byte swizzle of the TMA box unless the
    // rows carry their scale inline, whose 144-byte pitch already spreads the lanes over the banks)
    const uint8_t* src = raw + t * (inline_scale ? kRawPitchInline : 128);
    const int sw = inline_scale ? 0 : (t & 7);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    uint4 row[8];                                          // all loads first: one latency per tile
#pragma unroll
    for (int i = 0; i < 8; ++i) row[i] = *reinterpret_cast<const uint4*>(src + ((i ^ sw) << 4));
    uint32_t out[64];                                      // column c = elements 2c, 2c+1
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t in[4] = {row[i].x, row[i].y, row[i].z, row[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t u = in[j] ^ 0x80808080u;
            const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);   // {0x64|u0, 0x64|u1}
            const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);   // {0x64|u2, 0x64|u3}
            const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), bias);
            const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), bias);
            out[8 * i + 2 * j] = *reinterpret_cast<const uint32_t*>(&a);
            out[8 * i + 2 * j + 1] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    tmem_st_32x32b_x32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(out));
    tmem_st_32x32b_x32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(out + 32));
    tmem_st_wait();
}

template <typename TK, bool kQ8>
__global__ void __launch_bounds__(kQ8 ? kThreadsQ8 : kThreads, 1) score_tc_decode_kernel(
    const __grid_constant__ CUtensorMap kmap, const void* __restrict__ q, int q_dtype,
    const float* __restrict__ w, Geom g, float* __restrict__ scores, int64_t score_row_stride, int sched_slot,
    const float* __restrict__ k_scale, int64_t k_rows, HistOut ho, int chunk_tiles) {
    uint32_t* hist = ho.hist;
    constexpr int kNT = kQ8 ? kThreadsQ8 : kThreads;
    constexpr int kTmaStages = kQ8 ? kRawStages : kStages;   // the producer's ring
    constexpr int kTmaStride = kQ8 ? kRawTileBytes : kTileBytes;
    // int8 keys without a scale array carry each row's scale in bytes 128..131 of the row
    const bool inline_scale = kQ8 && k_scale == nullptr;
    const int kTmaBytes = kQ8 ? kTileKeys * (inline_scale ? kRawPitchInline : 128) : kTileBytes;
    constexpr int kAStages = kQ8 ? kConvStages : kStages;    // the MMA's A tiles
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tma_tiles = smem;                               // kTmaStages x kTmaBytes, 1024-aligned
    uint8_t* tiles = smem;                                   // 16-bit keys: kStages x 32 KB
    uint8_t* qbuf = kQ8 ? smem + (size_t)kRawStages * kRawTileBytes
                        : tiles + (size_t)kStages * kTileBytes;   // kQBufs x 16 KB, 1024-aligned
    Ctl& c = *reinterpret_cast<Ctl*>(qbuf + kQBufs * kQBytes);
    int* pre = reinterpret_cast<int*>(&c + 1);               // [n_rows + 1] in prefix mode
    int* nvis = pre + kMaxPrefixRows + 1;                    // [n_rows] in prefix mode
    float* escale = reinterpret_cast<float*>(nvis + kMaxPrefixRows);   // int8 keys: [4 warps][8 tiles][32],
                                                                       // or with inline scales [kSRing][128]
    uint32_t* shist = reinterpret_cast<uint32_t*>(nvis + kMaxPrefixRows);   // 16-bit keys: 2 x kHistWords

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_rows = (int64_t)g.B * g.T;
    const bool prefix = n_rows <= kMaxPrefixRows;
    pdl_trigger();
    pdl_wait();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTmaStages; ++i) {
            mbar_init(&c.full[i], 1);
            mbar_init(&c.empty[i], kQ8 ? 4 : 1);     // int8: freed by the 4 converter warps
        }
        for (int i = 0; i < kConvStages; ++i) {
            mbar_init(&c.afull[i], 4);
            mbar_init(&c.aempty[i], 1);
        }
        for (int i = 0; i < kSRing; ++i) {
            mbar_init(&c.sfull[i], 4);
            mbar_init(&c.sempty[i], 4);
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&c.tfull[i], 1);
            mbar_init(&c.tempty[i], 4);
        }
        for (int i = 0; i < kQBufs; ++i) {
            mbar_init(&c.qfull[i], 1);
            mbar_init(&c.qempty[i], 1);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&c.cfull[i], 1);
            mbar_init(&c.cempty[i], kChunkReaders + (kQ8 ? 4 : 0));
        }
        mbar_init(&c.done, 1);
        mbar_init(&c.hdone[0], 4);
        mbar_init(&c.hdone[1], 4);
        c.abort = 0;
        fence_mbar_init();
    }
    // chunks per row, then their prefix (all threads read the rows' bounds in parallel)
    if (prefix) {
        for (int64_t r = threadIdx.x; r < n_rows; r += kNT) {
            const int nv = row_n_vis(g, r);
            nvis[r] = nv;
            pre[r + 1] = row_chunks(nv, chunk_tiles);
        }
        __syncthreads();
        if (warp == 0) {
            int carry = 0;
            for (int base = 0; base < (int)n_rows; base += 32) {
                const int i = base + lane;
                int v = i < n_rows ? pre[i + 1] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                if (i < n_rows) pre[i + 1] = carry + v;
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
            if (lane == 0) {
                pre[0] = 0;
                c.n_chunks = carry;
            }
        }
    } else if (threadIdx.x == 0) {
        c.n_chunks = (int)n_rows;
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&kmap);
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, kQ8 ? kTmemColsQ8 : kTmemCols);
        tmem_relinquish();
    }
    if (!kQ8 && hist)
        for (int i = threadIdx.x; i < 2 * kHistWords; i += kNT) shist[i] = 0u;
    if (hist) {
        // this CTA's slice of the histograms (rows x 2048 counts, 16-byte stores), and the
        // select's per-row counters
        const int64_t n4 = n_rows * 512;
        const int64_t per = (n4 + gridDim.x - 1) / gridDim.x;
        const int64_t a = (int64_t)blockIdx.x * per, e = min(n4, a + per);
        uint4* h4 = reinterpret_cast<uint4*>(hist);
        for (int64_t i = a + threadIdx.x; i < e; i += kNT) h4[i] = make_uint4(0u, 0u, 0u, 0u);
        if (blockIdx.x == 0)
            for (int64_t i = threadIdx.x; i < n_rows; i += kNT) ho.cnt[i] = 0u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (hist && threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&g_score_sched[sched_slot][2], 1u);
    }
    const uint32_t tmem = c.tmem_base;
    const int n_chunks = c.n_chunks;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Lane 0 claims chunks, waits for free stages and issues the TMA loads.
        // For paged caches the whole warp first resolves the chunk's key rows
        // through the page table, one 64-key half per lane, so lane 0's per-tile
        // work stays as short as in the contiguous case.
        int stage = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        // key tiles are read once: tag them evict-first in L2, so that the scores this launch
        // writes (which the fused select reads back) are not pushed out by the stream of keys
        const uint64_t kpol = l2_evict_first_policy();
        // the next chunk is claimed one chunk ahead, so the counter's round
        // trip overlaps the current chunk's loads
        int ch = 0;
        if (lane == 0) ch = (int)atomicAdd(&g_score_sched[sched_slot][0], 1u);
        for (int k = 0;; ++k) {
            const int slot = k % kRing;
            int go = 1;
            if (lane == 0) {
                if (*(volatile int*)&c.abort || !mbar_wait(&c.cempty[slot], (uint32_t)(((k / kRing) & 1) ^ 1))) {
                    abort_cta(c, g);
                    go = 0;
                } else {
                    const Chunk d = chunk_of(g, pre, nvis, n_rows, prefix, ch, n_chunks, chunk_tiles);
                    c.chunk[slot] = d;
                    mbar_arrive(&c.cfull[slot]);
                    if (d.row < 0)
                        go = 0;
                    else
                        ch = (int)atomicAdd(&g_score_sched[sched_slot][0], 1u);
                }
            }
            __syncwarp();
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            const Chunk d = c.chunk[slot];
            const int b_seq = (int)(d.row / g.T);
            const int nk = prefix ? nvis[d.row] : row_n_vis(g, d.row);
            int ok = 1;
            if (!g.page_table) {
                if (lane == 0) {
                    const int64_t krow0 = seq_row0(g, b_seq);
                    for (int t = d.t0; t < d.t1; ++t) {
                        if (!mbar_wait(&c.empty[stage], phase ^ 1)) {
                            abort_cta(c, g);
                            ok = 0;
                            break;
                        }
                        uint8_t* dst = tma_tiles + (size_t)stage * kTmaStride;
                        const int64_t krow = krow0 + (int64_t)t * kTileKeys;
                        // rows past the visible keys may lie past the cache (TMA fills them with 0)
                        const int valid = min(kTileKeys, nk - t * kTileKeys);
                        if (krow < 0 || krow + valid > k_rows) flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                        mbar_arrive_expect_tx(&c.full[stage], kTmaBytes);
                        if constexpr (kQ8) {
                            tma_load_2d_hint(dst, &kmap, &c.full[stage], 0, (int32_t)krow, kpol);
                        } else {
                            tma_load_2d_hint(dst, &kmap, &c.full[stage], 0, (int32_t)krow, kpol);
                            tma_load_2d_hint(dst + kHalfBytes, &kmap, &c.full[stage], 64, (int32_t)krow, kpol);
                        }
                        ++issued;
                        if (++stage == kTmaStages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
            } else {
                // paged cache: two 64-key halves per tile, each inside one page
                // (page_size % 64 == 0); a half past the visible keys is not
                // loaded (its keys are never stored).  16 tiles = 32 halves per pass.
                for (int tg = d.t0; ok && tg < d.t1; tg += 16) {
                    const int tn = min(16, d.t1 - tg);
                    const int jj = tg * kTileKeys + 64 * lane;
                    int64_t kr = 0;
                    if (lane < 2 * tn && jj < nk) {
                        const int pg = jj / g.page_size;
                        kr = (int64_t)g.page_table[(int64_t)b_seq * g.page_table_stride + pg] * g.page_size +
                             (jj - pg * g.page_size);
                        if (kr < 0 || kr + min(64, nk - jj) > k_rows) flag(g.status, IDX_ERR_DEVICE_BOUNDS);
                    }
                    for (int i = 0; i < tn; ++i) {
                        const int64_t kr0 = __shfl_sync(0xffffffffu, kr, 2 * i);
                        const int64_t kr1 = __shfl_sync(0xffffffffu, kr, 2 * i + 1);
                        if (lane == 0) {
                            if (!mbar_wait(&c.empty[stage], phase ^ 1)) {
                                abort_cta(c, g);
                                ok = 0;
                            } else {
                                uint8_t* dst = tma_tiles + (size_t)stage * kTmaStride;
                                const int j0 = (tg + i) * kTileKeys;
                                const int halves = j0 + 64 < nk ? 2 : 1;
                                mbar_arrive_expect_tx(&c.full[stage], (uint32_t)(halves * (kTmaBytes / 2)));
                                for (int hh = 0; hh < halves; ++hh) {
                                    const int32_t kr_h = (int32_t)(hh ? kr1 : kr0);
                                    if constexpr (kQ8) {
                                        tma_load_2d_hint(dst + hh * (kTmaBytes / 2), &kmap, &c.full[stage], 0, kr_h, kpol);
                                    } else {
                                        tma_load_2d_hint(dst + hh * (kHalfBytes / 2), &kmap, &c.full[stage], 0, kr_h, kpol);
                                        tma_load_2d_hint(dst + kHalfBytes + hh * (kHalfBytes / 2), &kmap,
                                                         &c.full[stage], 64, kr_h, kpol);
                                    }
                                }
                                ++issued;
                                if (++stage == kTmaStages) {
                                    stage = 0;
                                    phase ^= 1;
                                }
                            }
                        }
                        if (!__shfl_sync(0xffffffffu, ok, 0)) {
                            ok = 0;
                            break;
                        }
                    }
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        }
        // never leave the CTA with TMA writes in flight
        if (lane == 0) {
            const int64_t n = issued < kTmaStages ? issued : kTmaStages;
            for (int64_t i = issued - n; i < issued; ++i)
                mbar_wait(&c.full[i % kTmaStages], (uint32_t)((i / kTmaStages) & 1));
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kTileKeys, kH, kIsBF16<TK> ? 1 : 0);
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            int64_t qseq = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k % kRing;
                if (*(volatile int*)&c.abort || !mbar_wait(&c.cfull[slot], (uint32_t)((k / kRing) & 1))) {
                    abort_cta(c, g);
                    break;
                }
                const Chunk d = c.chunk[slot];
                mbar_arrive(&c.cempty[slot]);
                if (d.row < 0) break;
                if (d.t1 <= d.t0) continue;
                const int qb = (int)(qseq % kQBufs);
                if (!mbar_wait(&c.qfull[qb], (uint32_t)((qseq / kQBufs) & 1))) {
                    abort_cta(c, g);
                    break;
                }
                const uint32_t b0 = smem_u32(qbuf + qb * kQBytes);
                uint64_t* a_full = kQ8 ? c.afull : c.full;
                uint64_t* a_empty = kQ8 ? c.aempty : c.empty;
                for (int t = d.t0; t < d.t1; ++t) {
                    if (!mbar_wait(&c.tempty[acc], aphase ^ 1) || !mbar_wait(&a_full[stage], phase)) {
                        abort_cta(c, g);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + acc * kH;
                    if constexpr (kQ8) {
                        // A = the widened key tile in TMEM (lane = key, two f16 per column)
                        const uint32_t at = tmem + kAcc * kH + stage * (kD / 2);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint32_t off = (kk & 3) * 32;
                            const uint64_t bd = desc_sw128_kmajor(b0 + (kk >> 2) * kQHalfBytes + off, 1024);
                            mma_f16_ts(dt, at + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
                        }
                    } else {
                        const uint32_t a0 = smem_u32(tiles + (size_t)stage * kTileBytes);
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint32_t off = (kk & 3) * 32;   // K offset inside the 128-byte row
                            const uint64_t ad = desc_sw128_kmajor(a0 + (kk >> 2) * kHalfBytes + off, 1024);
                            const uint64_t bd = desc_sw128_kmajor(b0 + (kk >> 2) * kQHalfBytes + off, 1024);
                            mma_f16_ss(dt, ad, bd, idesc, kk > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&a_empty[stage]);
                    mma_commit(&c.tfull[acc]);
                    if (++stage == kAStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++acc == kAcc) {
                        acc = 0;
                        aphase ^= 1;
                    }
                }
                mma_commit(&c.qempty[qb]);
                ++qseq;
            }
            // every MMA issued by this thread has completed before TMEM is freed
            mma_commit(&c.done);
            mbar_wait(&c.done, 0);
        }
        __syncwarp();
    } else if (warp == 6) {
        // ------------------------------------------------------------ q stager
        int64_t qseq = 0;
        for (int k = 0;; ++k) {
            Chunk d;
            if (warp_aborted(c) || !warp_next_chunk(c, k, d)) {
                abort_cta(c, g);
                break;
            }
            if (d.row < 0) break;
            if (d.t1 <= d.t0) continue;
            const int qb = (int)(qseq % kQBufs);
            if (!warp_wait(&c.qempty[qb], (uint32_t)(((qseq / kQBufs) & 1) ^ 1))) {
                abort_cta(c, g);
                break;
            }
            uint8_t* qdst = qbuf + qb * kQBytes;
            const int64_t off = d.row * (int64_t)kH * kD;
            bool ovf;
            if (q_dtype == IDX_F32) ovf = stage_q_row<TK>(static_cast<const float*>(q) + off, qdst, lane);
            else if (q_dtype == IDX_BF16) ovf = stage_q_row<TK>(static_cast<const __nv_bfloat16*>(q) + off, qdst, lane);
            else ovf = stage_q_row<TK>(static_cast<const __half*>(q) + off, qdst, lane);
            if (__any_sync(0xffffffffu, ovf) && lane == 0) flag(g.status, IDX_ERR_INEXACT);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.qfull[qb]);
            ++qseq;
        }
    } else if (kQ8 && warp >= 7) {
        // ------------------------------------------------------------ converters (int8 keys)
        // with inline scales they also hand each row's scale to the epilogue (ring of kSRing tiles)
        // key row of the tile = the TMEM lane this warp may write (lane quarter = warp % 4)
        const int t = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int rs = 0, as = 0, ss = 0;
        uint32_t rph = 0, aph = 0, sph = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Chunk d;
            if (warp_aborted(c) || !warp_next_chunk(c, k, d)) {
                abort_cta(c, g);
                break;
            }
            if (d.row < 0) break;
            for (int tt = d.t0; tt < d.t1; ++tt) {
                if (!warp_wait(&c.full[rs], rph) || !warp_wait(&c.aempty[as], aph ^ 1) ||
                    (inline_scale && !warp_wait(&c.sempty[ss], sph ^ 1))) {
                    abort_cta(c, g);
                    ok = false;
                    break;
                }
                static_assert(!kQ8 || std::is_same<TK, __half>::value, "int8 codes are widened to f16");
                const uint8_t* raw = tma_tiles + (size_t)rs * kRawTileBytes;
                widen_row_tmem(raw, tmem + lane_off + kAcc * kH + as * (kD / 2), t, inline_scale);
                if (inline_scale)
                    escale[ss * kTileKeys + t] = *reinterpret_cast<const float*>(raw + t * kRawPitchInline + kD);
                tc_fence_before();                  // the TMEM stores before the MMA reads them
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&c.empty[rs]);
                    mbar_arrive(&c.afull[as]);
                    if (inline_scale) mbar_arrive(&c.sfull[ss]);
                }
                if (inline_scale && ++ss == kSRing) {
                    ss = 0;
                    sph ^= 1;
                }
                if (++rs == kRawStages) {
                    rs = 0;
                    rph ^= 1;
                }
                if (++as == kConvStages) {
                    as = 0;
                    aph ^= 1;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;                 // TMEM lane quarter this warp may access
        float* esc = escale + (warp - 2) * 8 * 32;   // int8 keys: this warp's prefetched key scales
        int ss = 0;                                // inline scales: ring slot of the next tile
        uint32_t sph = 0;
        int acc = 0;
        uint32_t aphase = 0;
        float wv[kH];
        bool ok = true;
        // fused top-k: no count is added before every CTA has zeroed its histogram slice
        bool use_hist = hist != nullptr;
        int64_t hchunk = 0;                        // non-empty chunks this epilogue has finished
        if (use_hist) {
            int ready = 1;
            if (lane == 0) ready = wait_counter(&g_score_sched[sched_slot][2], gridDim.x) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ready, 0)) {
                flag(g.status, IDX_ERR_TIMEOUT);
                use_hist = false;
            }
        }
        for (int k = 0; ok; ++k) {
            Chunk d;
            if (warp_aborted(c) || !warp_next_chunk(c, k, d)) {
                abort_cta(c, g);
                break;
            }
            if (d.row < 0) break;
            if (d.t1 <= d.t0) continue;
            const int n_keys = prefix ? nvis[d.row] : row_n_vis(g, d.row);
            const int b_seq = (int)(d.row / g.T);
            const int64_t krow0 = (kQ8 && !g.page_table) ? seq_row0(g, b_seq) : 0;
            const float4* wr = reinterpret_cast<const float4*>(w + d.row * kH);
#pragma unroll
            for (int h4 = 0; h4 < kH / 4; ++h4) {
                const float4 x = wr[h4];
                wv[4 * h4] = x.x;
                wv[4 * h4 + 1] = x.y;
                wv[4 * h4 + 2] = x.z;
                wv[4 * h4 + 3] = x.w;
            }
            const int hb = (int)(hchunk & 1);      // shared histogram buffer of this chunk
            // tiles in groups of 8: an int8 cache's per-key scales of a whole group are
            // loaded at once, the next group's while this one is processed, and parked in
            // this lane's own shared-memory slots
            float scn[8];
            auto load_scales = [&](int g0) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = (g0 + i) * kTileKeys + quad * 32 + lane;
                    float v = 0.f;
                    if (g0 + i < d.t1 && j < n_keys) {
                        const int64_t kr = g.page_table ? key_row(g, b_seq, j) : krow0 + j;
                        if (kr >= 0 && kr < k_rows) v = k_scale[kr];
                    }
                    scn[i] = v;
                }
            };
            if (kQ8 && !inline_scale) load_scales(d.t0);
            for (int g0 = d.t0; ok && g0 < d.t1; g0 += 8) {
                if (kQ8 && !inline_scale) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) esc[i * 32 + lane] = scn[i];
                    if (g0 + 8 < d.t1) load_scales(g0 + 8);
                }
#pragma unroll 1
                for (int i = 0; i < 8; ++i) {
                    const int t = g0 + i;
                    if (t >= d.t1) break;
                    const int j = t * kTileKeys + quad * 32 + lane;
                    // int8 keys: the key's scale multiplies every head's dot product before the ReLU
                    float sc = 1.f;
                    if constexpr (kQ8) {
                        if (!inline_scale) {
                            sc = esc[i * 32 + lane];
                        } else {
                            if (!warp_wait(&c.sfull[ss], sph)) {
                                abort_cta(c, g);
                                ok = false;
                                break;
                            }
                            sc = j < n_keys ? escale[ss * kTileKeys + quad * 32 + lane] : 0.f;
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&c.sempty[ss]);
                            if (++ss == kSRing) {
                                ss = 0;
                                sph ^= 1;
                            }
                        }
                    }
                    if (!warp_wait(&c.tfull[acc], aphase)) {
                        abort_cta(c, g);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float v0[32], v1[32];
                    const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + acc * kH;
                    tmem_ld_32x32b_x32(ta, v0);
                    tmem_ld_32x32b_x32(ta + 32, v1);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c.tempty[acc]);
                    // four partial sums (a shorter dependent chain); the sum order is fixed.
                    // int8 keys: sum_h w_h relu(sc*D_h) = sc * sum_h w_h max(D_h, 0) for sc >= 0
                    // and sc * sum_h w_h min(D_h, 0) for sc < 0, so the scale costs one multiply
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
                    if (!kQ8 || sc >= 0.f) {
#pragma unroll
                        for (int h = 0; h < 32; h += 2) {
                            s0 = fmaf(wv[h], fmaxf(v0[h], 0.f), s0);
                            s1 = fmaf(wv[h + 1], fmaxf(v0[h + 1], 0.f), s1);
                            s2 = fmaf(wv[32 + h], fmaxf(v1[h], 0.f), s2);
                            s3 = fmaf(wv[33 + h], fmaxf(v1[h + 1], 0.f), s3);
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < 32; h += 2) {
                            s0 = fmaf(wv[h], fminf(v0[h], 0.f), s0);
                            s1 = fmaf(wv[h + 1], fminf(v0[h + 1], 0.f), s1);
                            s2 = fmaf(wv[32 + h], fminf(v1[h], 0.f), s2);
                            s3 = fmaf(wv[33 + h], fminf(v1[h + 1], 0.f), s3);
                        }
                    }
                    float s = (s0 + s1) + (s2 + s3);
                    if constexpr (kQ8) s *= sc;
                    s += 0.0f;   // -0 + +0 = +0
                    if (j < n_keys) scores[d.row * score_row_stride + j] = s;
                    if constexpr (!kQ8) {
                        if (use_hist) {
                            // equal bins of the warp folded into one shared-memory add (16-bit halves)
                            const uint32_t bin = j < n_keys ? order_key(s) >> 21 : 0xffffffffu;
                            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
                            if (j < n_keys && lane == __ffs(peers) - 1)
                                atomicAdd(&shist[hb * kHistWords + (bin >> 1)], (uint32_t)__popc(peers) << ((bin & 1) * 16));
                        }
                    }
                    if (++acc == kAcc) {
                        acc = 0;
                        aphase ^= 1;
                    }
                }
            }
            if constexpr (!kQ8) {
                if (use_hist && ok) {
                    // all four epilogue warps have added this chunk's counts: this warp flushes
                    // its quarter of the buffer's nonzero bins and clears them
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c.hdone[hb]);
                    if (!warp_wait(&c.hdone[hb], (uint32_t)((hchunk >> 1) & 1))) {
                        abort_cta(c, g);
                        ok = false;
                    } else {
                        uint32_t* hw = shist + hb * kHistWords;
                        uint32_t* grow = hist + d.row * 2048;
                        for (int i = quad * (kHistWords / 4) + lane; i < (quad + 1) * (kHistWords / 4); i += 32) {
                            const uint32_t v = hw[i];
                            if (v) {
                                hw[i] = 0u;
                                if (v & 0xffffu) atomicAdd(&grow[2 * i], v & 0xffffu);
                                if (v >> 16) atomicAdd(&grow[2 * i + 1], v >> 16);
                            }
                        }
                    }
                }
                ++hchunk;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kQ8 ? kTmemColsQ8 : kTmemCols);
    // the last CTA to finish returns the slot's counters to zero for a later launch
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&g_score_sched[sched_slot][1], 1u) == gridDim.x - 1) {
            atomicExch(&g_score_sched[sched_slot][0], 0u);
            atomicExch(&g_score_sched[sched_slot][1], 0u);
            atomicExch(&g_score_sched[sched_slot][2], 0u);
            __threadfence();
        }
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Prefill (many query rows per sequence, causal): tiles of 128 query rows x
// 256 keys of one sequence, persistent CTAs taking tiles round-robin.  Per tile
// the key tile [256 x 128] is loaded once and stays in shared memory; for each
// of the 64 heads the head's query tile Q_h [128 x 128] is loaded by TMA (a 3-D
// tensor map over [rows, heads, d], so head h's rows are strided) and
//     D_h[128 queries x 256 keys] = Q_h . K^T     (M=128, N=256, K=128)
// goes to one of two 256-column TMEM buffers while eight epilogue warps (two per
// TMEM lane quarter, one per 128-key half) add w[q, h] * relu(D_h) into f32
// registers.  After the 64 heads the visible scores (key < n_vis of the row)
// are written.  Tiles whose keys all lie beyond every row's causal bound are
// skipped.
// ---------------------------------------------------------------------------
constexpr int kPQ = 128;                          // query rows per tile
constexpr int kPK = 256;                          // keys per tile
constexpr int kPStages = 3;                       // Q_h stages
constexpr int kPQBytes = kPQ * kD * 2;            // 32 KB
constexpr int kPKBytes = kPK * kD * 2;            // 64 KB
constexpr int kPWBytes = kPQ * kH * 4;            // 32 KB
#ifndef LIDX_PREFILL_EPI_WARPS
#define LIDX_PREFILL_EPI_WARPS 8
#endif
constexpr int kPEpiWarps = LIDX_PREFILL_EPI_WARPS;  // a multiple of 4: each TMEM lane quarter split by keys
constexpr int kPKW = kPK / (kPEpiWarps / 4);      // keys per epilogue warp
static_assert(kPEpiWarps % 4 == 0 && kPKW % 32 == 0, "epilogue split");
constexpr int kPThreads = 32 * (2 + kPEpiWarps);  // producer, MMA, epilogue
constexpr int kPMaxQTiles = 4096;                 // (sequence, query tile) pairs enumerated in shared memory
constexpr int kPTmemCols = 512;

struct PCtl {
    uint64_t qfull[kPStages];
    uint64_t qempty[kPStages];
    uint64_t kfull, kempty;
    uint64_t wfull, wempty;
    uint64_t dfull[2], dempty[2];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kPSmemBytes =
    1024 + kPKBytes + (size_t)kPStages * kPQBytes + kPWBytes + sizeof(PCtl) + (kPMaxQTiles + 1) * sizeof(int);

struct PTile {
    int b, qt, kt;      // sequence, query tile, key tile
};

// Live tiles (some key visible to some row of the tile) are numbered with the
// key tile fastest; pre[i] = live tiles of the (sequence, query tile) pairs
// before pair i of this launch.  Consecutive CTAs therefore take neighbouring
// key tiles of the same query tile, and the query rows they stream are shared
// in L2.
__device__ __forceinline__ PTile ptile_live(const int* pre, int n_pairs, int pair0, int q_tiles, int live) {
    int lo = 0, hi = n_pairs;  // last pair with pre[pair] <= live
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= live) lo = mid;
        else hi = mid;
    }
    PTile p;
    p.b = (pair0 + lo) / q_tiles;
    p.qt = (pair0 + lo) % q_tiles;
    p.kt = live - pre[lo];
    return p;
}

__device__ __forceinline__ bool pc_aborted(PCtl& c) { return __any_sync(0xffffffffu, *(volatile int*)&c.abort != 0); }
__device__ __forceinline__ void pc_abort(PCtl& c, const Geom& g) {
    *(volatile int*)&c.abort = 1;
    flag(g.status, IDX_ERR_TIMEOUT);
}

template <int kBF16>
__global__ void __launch_bounds__(kPThreads, 1) score_tc_prefill_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap wmap, Geom g, float* __restrict__ scores, int64_t score_row_stride,
    int q_tiles, int k_tiles, int pair0, int n_pairs) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ktile = smem;                                  // 2 x [256 rows x 128 B]
    uint8_t* qst = ktile + kPKBytes;                        // kPStages x 2 x [128 rows x 128 B]
    float* wt = reinterpret_cast<float*>(qst + (size_t)kPStages * kPQBytes);   // [128 rows][64 heads]
    PCtl& c = *reinterpret_cast<PCtl*>(reinterpret_cast<uint8_t*>(wt) + kPWBytes);
    int* pre = reinterpret_cast<int*>(&c + 1);              // [n_pairs + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // live key tiles of each (sequence, query tile) pair: the keys visible to the
    // pair's rows, rounded up to whole tiles (one warp per pair)
    for (int i = warp; i < n_pairs; i += kPThreads / 32) {
        const int b = (pair0 + i) / q_tiles, qt = (pair0 + i) % q_tiles;
        int nv = 0;
        for (int t = qt * kPQ + lane; t < min(g.T, qt * kPQ + kPQ); t += 32)
            nv = max(nv, row_n_vis(g, (int64_t)b * g.T + t));
#pragma unroll
        for (int o = 16; o; o >>= 1) nv = max(nv, __shfl_xor_sync(0xffffffffu, nv, o));
        if (lane == 0) pre[i + 1] = min(k_tiles, (nv + kPK - 1) / kPK);
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&c.qfull[i], 1);
            mbar_init(&c.qempty[i], 1);
        }
        mbar_init(&c.kfull, 1);
        mbar_init(&c.kempty, 1);
        mbar_init(&c.wfull, 1);
        mbar_init(&c.wempty, kPEpiWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&c.dfull[i], 1);
            mbar_init(&c.dempty[i], kPEpiWarps);
        }
        mbar_init(&c.done, 1);
        c.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&wmap);
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, kPTmemCols);
        tmem_relinquish();
    }
    __syncthreads();
    if (warp == 0) {
        // inclusive scan of the per-pair counts
        int carry = 0;
        for (int base = 0; base < n_pairs; base += 32) {
            const int i = base + lane;
            int v = i < n_pairs ? pre[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (i < n_pairs) pre[i + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) pre[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    const int n_live = pre[n_pairs];

    if (warp == 0) {
        // ---------------------------------------------------------- producer (one lane)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, tph = 0;
            for (int64_t live = blockIdx.x; live < n_live; live += gridDim.x) {
                const PTile p = ptile_live(pre, n_pairs, pair0, q_tiles, (int)live);
                const int32_t row0 = (int32_t)((int64_t)p.b * g.T + p.qt * kPQ);
                if (!mbar_wait(&c.kempty, tph ^ 1) || !mbar_wait(&c.wempty, tph ^ 1)) {
                    pc_abort(c, g);
                    break;
                }
                if (!g.page_table) {
                    const int32_t key0 = (int32_t)(seq_row0(g, p.b) + (int64_t)p.kt * kPK);
                    mbar_arrive_expect_tx(&c.kfull, kPKBytes);
                    tma_load_2d(ktile, &kmap, &c.kfull, 0, key0);
                    tma_load_2d(ktile + kPKBytes / 2, &kmap, &c.kfull, 64, key0);
                } else {
                    // paged cache: 64-key quarters, each inside one page; quarters past the
                    // sequence's keys are not loaded
                    const int j0 = p.kt * kPK, nkv = seq_n_kv(g, p.b);
                    int nq = 0;
                    while (nq < 4 && j0 + 64 * nq < nkv) ++nq;
                    mbar_arrive_expect_tx(&c.kfull, (uint32_t)(nq * (kPKBytes / 4)));
                    for (int i = 0; i < nq; ++i) {
                        const int32_t kr = (int32_t)key_row(g, p.b, j0 + 64 * i);
                        tma_load_2d(ktile + i * (kPKBytes / 8), &kmap, &c.kfull, 0, kr);
                        tma_load_2d(ktile + kPKBytes / 2 + i * (kPKBytes / 8), &kmap, &c.kfull, 64, kr);
                    }
                }
                mbar_arrive_expect_tx(&c.wfull, kPWBytes);
                tma_load_2d(wt, &wmap, &c.wfull, 0, row0);
                for (int h = 0; h < kH; ++h) {
                    if (!mbar_wait(&c.qempty[stage], phase ^ 1)) {
                        pc_abort(c, g);
                        break;
                    }
                    uint8_t* dst = qst + (size_t)stage * kPQBytes;
                    mbar_arrive_expect_tx(&c.qfull[stage], kPQBytes);
                    tma_load_3d(dst, &qmap, &c.qfull[stage], 0, h, row0);
                    tma_load_3d(dst + kPQBytes / 2, &qmap, &c.qfull[stage], 64, h, row0);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (*(volatile int*)&c.abort) break;
                tph ^= 1;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer (one lane)
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kPQ, kPK, kBF16);
            int stage = 0, buf = 0;
            uint32_t phase = 0, bph = 0, tph = 0;
            for (int64_t live = blockIdx.x; live < n_live; live += gridDim.x) {
                const PTile p = ptile_live(pre, n_pairs, pair0, q_tiles, (int)live);
                if (!mbar_wait(&c.kfull, tph)) {
                    pc_abort(c, g);
                    break;
                }
                const uint32_t kb = smem_u32(ktile);
                bool ok = true;
                for (int h = 0; h < kH && ok; ++h) {
                    if (!mbar_wait(&c.qfull[stage], phase) || !mbar_wait(&c.dempty[buf], bph ^ 1)) {
                        pc_abort(c, g);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qb = smem_u32(qst + (size_t)stage * kPQBytes);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t ad = desc_sw128_kmajor(qb + (kk >> 2) * (kPQBytes / 2) + off, 1024);
                        const uint64_t bd = desc_sw128_kmajor(kb + (kk >> 2) * (kPKBytes / 2) + off, 1024);
                        mma_f16_ss(tmem + buf * kPK, ad, bd, idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&c.qempty[stage]);
                    mma_commit(&c.dfull[buf]);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++buf == 2) {
                        buf = 0;
                        bph ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&c.kempty);
                tph ^= 1;
            }
            mma_commit(&c.done);
            mbar_wait(&c.done, 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue: 8 warps, thread = query row
        const int ew = warp - 2;
        const int quad = warp & 3;                // TMEM lane quarter this warp may access
        const int part = ew >> 2;                 // which kPKW keys of the tile
        const int ql = quad * 32 + lane;          // query row within the tile
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int buf = 0;
        uint32_t bph = 0, tph = 0;
        for (int64_t live = blockIdx.x; live < n_live; live += gridDim.x) {
            const PTile p = ptile_live(pre, n_pairs, pair0, q_tiles, (int)live);
            if (pc_aborted(c) || !warp_wait(&c.wfull, tph)) {
                pc_abort(c, g);
                break;
            }
            float acc[kPKW];
#pragma unroll
            for (int j = 0; j < kPKW; ++j) acc[j] = 0.f;
            const float* wrow = wt + ql * kH;
            bool ok = true;
            for (int h = 0; h < kH; ++h) {
                const float wv = wrow[h];
                if (!warp_wait(&c.dfull[buf], bph)) {
                    pc_abort(c, g);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = tmem + lane_off + buf * kPK + part * kPKW;
#pragma unroll
                for (int cb = 0; cb < kPKW / 32; ++cb) {
                    float v[32];
                    tmem_ld_32x32b_x32(ta + cb * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[cb * 32 + i] = fmaf(wv, fmaxf(v[i], 0.f), acc[cb * 32 + i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.dempty[buf]);
                if (++buf == 2) {
                    buf = 0;
                    bph ^= 1;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.wempty);
            if (!ok) break;
            const int t = p.qt * kPQ + ql;
            if (t < g.T) {
                const int64_t r = (int64_t)p.b * g.T + t;
                const int nv = row_n_vis(g, r);
                const int j0 = p.kt * kPK + part * kPKW;
                float* dst = scores + r * score_row_stride + j0;
                const int nw = min(kPKW, nv - j0);
                if (nw == kPKW && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
                    for (int j = 0; j < kPKW; j += 4)
                        *reinterpret_cast<float4*>(dst + j) =
                            make_float4(acc[j] + 0.f, acc[j + 1] + 0.f, acc[j + 2] + 0.f, acc[j + 3] + 0.f);
                } else {
#pragma unroll
                    for (int j = 0; j < kPKW; ++j)
                        if (j < nw) dst[j] = acc[j] + 0.f;
                }
            }
            tph ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kPTmemCols);
}

cudaError_t launch_score_tc_prefill(const void* q, int q_dtype, const float* w, const void* k, int k_dtype,
                                    int64_t k_row_stride, int64_t k_rows, const Geom& g, float* scores,
                                    int64_t score_row_stride, cudaStream_t st) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0 || g.max_n_kv == 0) return cudaSuccess;
    if (n_rows > INT32_MAX || k_rows > INT32_MAX) return cudaErrorNotSupported;
    const bool bf16 = k_dtype == IDX_BF16;
    CUtensorMap qm, km, wm;
    if (g.page_table && g.page_size % 64 != 0) return cudaErrorNotSupported;
    if (!make_q3d_tmap(&qm, q, bf16, n_rows) ||
        !make_key_tmap(&km, k, bf16, k_row_stride, k_rows, g.page_table ? 64 : kPK) ||
        !make_w_tmap(&wm, w, n_rows))
        return cudaErrorNotSupported;
    const int q_tiles = (g.T + kPQ - 1) / kPQ;
    const int k_tiles = (g.max_n_kv + kPK - 1) / kPK;
    const int64_t pairs = (int64_t)g.B * q_tiles;
    auto kern = bf16 ? score_tc_prefill_kernel<1> : score_tc_prefill_kernel<0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmemBytes);
    if (e != cudaSuccess) return e;
    // one launch per chunk of (sequence, query tile) pairs: at most kPMaxQTiles,
    // and few enough that the chunk's tiles are numbered in 32 bits
    const int64_t chunk = std::min<int64_t>(kPMaxQTiles, std::max<int64_t>(1, INT32_MAX / k_tiles));
    for (int64_t p0 = 0; p0 < pairs; p0 += chunk) {
        const int np = (int)std::min<int64_t>(pairs - p0, chunk);
        const int64_t max_live = (int64_t)np * k_tiles;
        const int grid = (int)(max_live < sm_count() ? max_live : sm_count());
        kern<<<grid, kPThreads, kPSmemBytes, st>>>(qm, km, wm, g, scores, score_row_stride, q_tiles, k_tiles, (int)p0,
                                                   np);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    (void)q_dtype;
    return cudaSuccess;
}

namespace {
// grid of the decode scorer, the key tiles per chunk and the counter slot of this launch; false
// when the chunks would not number in 32 bits.  Chunks are kChunkTiles tiles, or fewer (down to 2)
// when a small batch would otherwise leave SMs idle: about four chunks per SM.
bool decode_launch_shape(const Geom& g, int& grid, int& ct, int& slot, int max_ct = kChunkTiles) {
    const int64_t n_rows = (int64_t)g.B * g.T;
    const int64_t tiles_per_row = (g.max_n_kv + kTileKeys - 1) / kTileKeys;
    ct = max_ct;
    if (n_rows <= kMaxPrefixRows) {
        while (ct > 2 && n_rows * ((tiles_per_row + ct - 1) / ct) < 4 * (int64_t)sm_count()) ct >>= 1;
    }
    const int64_t chunks_per_row = (tiles_per_row + ct - 1) / ct;
    const int64_t max_chunks = n_rows <= kMaxPrefixRows ? n_rows * chunks_per_row : n_rows;
    if (max_chunks >= INT32_MAX - 2 * (int64_t)sm_count()) return false;
    grid = (int)(max_chunks < sm_count() ? max_chunks : sm_count());
    // one counter slot per launch, round-robin (a slot is reused only after
    // kSchedSlots further launches; its previous launch has zeroed it by then
    // unless that many launches are in flight at once)
    static std::atomic<unsigned> next_slot{0};
    slot = (int)(next_slot.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
    return true;
}
}  // namespace

cudaError_t launch_score_tc_q8(const void* q, int q_dtype, const float* w, const int8_t* k8, int64_t k_row_stride,
                               const float* k_scale, int64_t k_rows, const Geom& g, float* scores,
                               int64_t score_row_stride, cudaStream_t st) {
    // the codes are widened to f16 exactly; q goes to f16 too (exact for f16 q, and for bf16
    // q inside f16's normal range, as on the F16-cache path)
    if (g.T != 1 || (q_dtype != IDX_BF16 && q_dtype != IDX_F16)) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(k8) & 15u) || (k_row_stride % 16) || k_rows < 1 || k_rows > INT32_MAX ||
        (reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u) ||
        (!k_scale && k_row_stride < kRawPitchInline))
        return cudaErrorNotSupported;
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0 || g.max_n_kv == 0) return cudaSuccess;
    CUtensorMap map;
    if (g.page_table && g.page_size % 64 != 0) return cudaErrorNotSupported;
    if (!make_key8_tmap(&map, k8, k_row_stride, k_rows, g.page_table ? 64 : kTileKeys, k_scale ? 128 : kRawPitchInline,
                        k_scale != nullptr))
        return cudaErrorNotSupported;
    int grid, ct, slot;
    // int8 keys: chunks of up to 32 tiles of 16 KB (the epilogue pays a row's weights and a group's
    // first scales once per chunk)
    if (!decode_launch_shape(g, grid, ct, slot, 4 * kChunkTiles)) return cudaErrorNotSupported;
    auto kern = score_tc_decode_kernel<__half, true>;
    constexpr size_t smem = smem_bytes<true>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kThreadsQ8), smem, st, map, q, q_dtype, w, g, scores, score_row_stride,
                      slot, k_scale, k_rows, HistOut{nullptr, nullptr}, ct);
}

cudaError_t launch_score_tc(const void* q, int q_dtype, const float* w, int H, int d, const void* k,
                            int k_dtype, int64_t k_row_stride, int64_t k_rows, const Geom& g, int block_size,
                            float* scores, int64_t score_row_stride, cudaStream_t st, uint32_t* hist,
                            uint32_t* cnt) {
    if (H != kH || d != kD || k_dtype == IDX_F32 || block_size > 1) return cudaErrorNotSupported;
    if (hist && g.T != 1) return cudaErrorNotSupported;   // the histogram epilogue is the decode scorer's
    if (g.T >= 64) {
        // many query rows per sequence: query tiles on the tensor cores (same-type operands)
        if (q_dtype != k_dtype || (reinterpret_cast<uintptr_t>(q) & 15u) || (k_row_stride % 8)) return cudaErrorNotSupported;
        return launch_score_tc_prefill(q, q_dtype, w, k, k_dtype, k_row_stride, k_rows, g, scores, score_row_stride,
                                       st);
    }
    if (g.T != 1) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(k) & 15u) || (k_row_stride % 8) || k_rows < 1 || k_rows > INT32_MAX ||
        (reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(q) & 15u))
        return cudaErrorNotSupported;
    const int64_t n_rows = (int64_t)g.B * g.T;
    if (n_rows == 0 || g.max_n_kv == 0) return cudaSuccess;
    CUtensorMap map;
    const bool bf16 = k_dtype == IDX_BF16;
    if (g.page_table && g.page_size % 64 != 0) return cudaErrorNotSupported;
    if (!make_key_tmap(&map, k, bf16, k_row_stride, k_rows, g.page_table ? 64 : kTileKeys)) return cudaErrorNotSupported;
    int grid, ct, slot;
    if (!decode_launch_shape(g, grid, ct, slot)) return cudaErrorNotSupported;
    auto kern = bf16 ? score_tc_decode_kernel<__nv_bfloat16, false> : score_tc_decode_kernel<__half, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, st, map, q, q_dtype, w, g, scores,
                      score_row_stride, slot, static_cast<const float*>(nullptr), k_rows,
                      HistOut{hist, cnt}, ct);
}

}  // namespace lidx
