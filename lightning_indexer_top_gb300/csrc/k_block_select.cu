// One launch for the indexer of a block-pooled decode step: the update of the
// pooled-key cache, the pooled-key scores and the block selection, i.e.
// idx_block_pool_update + idx_score over the pooled keys + idx_topk in block
// mode, with their results bit for bit (the three kernels and this one share
// the device code of block_ops.cuh).  Blocks are cuts of the position line of
// C tokens whose key is the mean of the block's raw keys; a query scores the
// complete blocks with the indexer's head-weighted ReLU sum and keeps the best
// floor(top_k/C) blocks plus the tail tokens (llama.cpp commit c88c916636, QSA
// commit message; DeepSeek-V3.2 lightning indexer, eq. 1).
//
// One cluster of CL CTAs (512 threads) per query row, CL the largest power of
// two up to 8 whose clusters are all resident at once.  CTA q of a row owns the row's blocks
// [q*per, (q+1)*per): it re-pools those at or after the sequence's first
// stale block (writing the pooled cache as the update does), scores its
// blocks (four threads per block key, two keys per thread) and writes each score both to the scores
// output and into rank 0's shared memory; after a cluster barrier rank 0 ranks
// the row's blocks and writes the selection.  Decode rows only (one query row
// per sequence: the pooled cache is per sequence, so rows of one sequence
// would pool the same blocks).
#include "block_ops.cuh"
#include "sm100_ptx.cuh"

namespace lidx {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxCl = 8;
constexpr int kPartFloats = 1024;             // pool partial sums: (128 / (d*size/16)) * d = 2048 / size

template <typename T, int HH>
__global__ void __launch_bounds__(kThreads, 1) block_score_topk_kernel(
    const void* q, int q_dtype, const float* __restrict__ w, int H, int d, const T* k, int64_t k_row_stride,
    int64_t k_rows, Geom g, int C, const int32_t* n_pooled, const int32_t* stale_pos, float* pooled,
    int64_t pool_seq_stride, bool vec, int top_k, float* scores, int64_t score_row_stride, int32_t* idx,
    int64_t idx_row_stride, int32_t* n_sel) {
    extern __shared__ __align__(16) float smem[];
    float* qs = smem;                  // [d][HH], heads >= H zero
    float* ws = qs + HH * d;           // [HH]
    float* part = ws + HH;             // pool partial sums
    float* sc = part + kPartFloats;    // the row's block scores (every CTA of the cluster)
    __shared__ blk::RankShared rs;
    __shared__ uint32_t cnts[kMaxCl];
    pdl_trigger();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");   // this CTA has started
    pdl_wait();
    const uint32_t cl = sm100::cluster_nctarank(), rank = sm100::cluster_ctarank();
    const int64_t r = blockIdx.x / cl;
    const int b = (int)r;   // one query row per sequence
    const int n_vis = row_n_vis(g, r);
    const int n_cb = n_vis / C;                     // blocks scored (visible to the row)
    const int n_cb_seq = seq_n_kv(g, b) / C;        // blocks pooled (the sequence's)
    const int nb = max(n_cb, n_cb_seq);
    const int per = (nb + (int)cl - 1) / (int)cl;   // a block is pooled and scored by the same CTA
    const int j0 = min(nb, (int)rank * per), j1 = min(nb, j0 + per);
    float* prow = pooled + (int64_t)b * pool_seq_stride * d;   // the sequence's pooled keys
    // 1. the changed pooled keys of this CTA's blocks
    const int beta0 = blk::pool_first_block(n_pooled, stale_pos, b, C, n_cb_seq);
    for (int beta = max(j0, beta0); beta < min(j1, n_cb_seq); ++beta)
        blk::pool_block(k, k_row_stride, k_rows, g, C, d, b, beta, part, prow + (int64_t)beta * d);
    // 2. the scores of this CTA's visible blocks (the pooled rows it wrote are visible to the CTA
    //    after pool_block's barriers)
    blk::load_q_split<HH>(q, q_dtype, w, H, d, r, qs, ws);
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // rank 0's shared memory is live
    uint32_t scq[kMaxCl];   // sc in each CTA of the cluster
#pragma unroll
    for (int q2 = 0; q2 < kMaxCl; ++q2) scq[q2] = q2 < (int)cl ? sm100::mapa(sc, (uint32_t)q2) : 0u;
    const int je = min(j1, n_cb);
    // two keys per thread (keys i and i + half of a pass of up to kThreads/2 keys): the q values a
    // thread reads serve both
    for (int jb = j0; jb < je; jb += kThreads / 2) {
        const int nk = min(kThreads / 2, je - jb), half = (nk + 1) >> 1;
        const int i = (int)(threadIdx.x >> 2), hg = threadIdx.x & 3;
        const int ja = jb + i, jc = jb + half + i;
        const bool va = i < half, vc = va && half + i < nk;
        float pa = 0.f, pc = 0.f;
        if (va)
            blk::score_split_part2<float, HH>(qs, ws, prow + (int64_t)ja * d, prow + (int64_t)(vc ? jc : ja) * d, d,
                                              hg, vec, pa, pc);
        pa = blk::score_split_sum(pa);
        pc = blk::score_split_sum(pc);
        if (hg == 0) {
            if (va) scores[r * score_row_stride + ja] = pa;
            if (vc) scores[r * score_row_stride + jc] = pc;
#pragma unroll
            for (int q2 = 0; q2 < kMaxCl; ++q2) {
                if (q2 >= (int)cl) break;
                if (va) sm100::st_cluster_f32(scq[q2] + 4u * (uint32_t)ja, pa);
                if (vc) sm100::st_cluster_f32(scq[q2] + 4u * (uint32_t)jc, pc);
            }
        }
    }
    // 3. every CTA holds all the row's block scores: it ranks its own blocks against all of them by
    //    the composite key (order key, then the complement of the block index: a larger composite is
    //    a better block, equal scores put the lower block first); block j is kept when fewer than K
    //    composites exceed its own (the same selection as blk::block_rank_row)
    sm100::cluster_sync();
    const int K = min(top_k / C, n_cb);
    for (int i = threadIdx.x; i < n_cb; i += kThreads)
        rs.comp[i] = ((uint64_t)order_key(sc[i]) << 32) | (uint32_t)(0xffffffffu - (uint32_t)i);
    for (int i = threadIdx.x; i < blk::kRankMax / 32; i += kThreads) rs.sel[i] = 0u;
    __syncthreads();
    for (int jb = j0; jb < je; jb += kThreads / 4) {   // four threads per block, each a quarter of the keys
        const int j = jb + (int)(threadIdx.x >> 2), pt = threadIdx.x & 3;
        uint32_t above = 0;
        if (j < je) {
            const uint64_t cj = rs.comp[j];
            for (int i = pt; i < n_cb; i += 4) above += rs.comp[i] > cj ? 1u : 0u;
        }
        above += __shfl_xor_sync(0xffffffffu, above, 1);
        above += __shfl_xor_sync(0xffffffffu, above, 2);
        if (j < je && pt == 0 && above < (uint32_t)K) atomicOr(&rs.sel[(j - j0) >> 5], 1u << ((j - j0) & 31));
    }
    __syncthreads();
    // this CTA's kept blocks in ascending order (a scan of the selection words), their count to every CTA
    const int nw = (max(je - j0, 0) + 31) >> 5;
    if (threadIdx.x < 32) {
        uint32_t carry = 0;
        for (int w0 = 0; w0 < nw; w0 += 32) {
            const int w = w0 + (int)threadIdx.x;
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
        if (threadIdx.x < cl) sm100::st_cluster_f32(sm100::mapa(&cnts[rank], threadIdx.x), __uint_as_float(carry));
    }
    __syncthreads();
    for (int j = j0 + (int)threadIdx.x; j < je; j += kThreads) {
        const uint32_t word = rs.sel[(j - j0) >> 5];
        if ((word >> ((j - j0) & 31)) & 1u)
            rs.blk[rs.pre[(j - j0) >> 5] + __popc(word & ((1u << ((j - j0) & 31)) - 1u))] = j;
    }
    sm100::cluster_sync();   // (every CTA's count is in every CTA)
    uint32_t base = 0, mine = cnts[rank];
    for (uint32_t q2 = 0; q2 < rank; ++q2) base += cnts[q2];
    int32_t* out = idx + r * idx_row_stride;
    for (int e = threadIdx.x; e < (int)mine * C; e += kThreads) {
        const int p = e / C, t = e - p * C;
        out[(int64_t)(base + p) * C + t] = rs.blk[p] * C + t;
    }
    if (rank == cl - 1) {
        // the tail tokens after the kept blocks, the padding, the count
        const int tail0 = n_cb * C, n_out = K * C + (n_vis - tail0);
        const int cap = (top_k / C) * C + C - 1;
        for (int i = threadIdx.x; i < n_vis - tail0; i += kThreads) out[K * C + i] = tail0 + i;
        for (int i = n_out + threadIdx.x; i < cap; i += kThreads) out[i] = -1;
        if (threadIdx.x == 0 && n_sel) n_sel[r] = n_out;
    }
}

template <typename T, int HH>
cudaError_t launch_t(const void* q, int q_dtype, const float* w, int H, int d, const T* k, int64_t k_row_stride,
                     int64_t k_rows, const Geom& g, int C, const int32_t* n_pooled, const int32_t* stale_pos,
                     float* pooled, int64_t pool_seq_stride, int top_k, float* scores, int64_t score_row_stride,
                     int32_t* idx, int64_t idx_row_stride, int32_t* n_sel, cudaStream_t st) {
    const int64_t n_rows = g.B;
    const int max_blocks = g.max_n_kv / C;
    const size_t smem = (size_t)(HH * d + HH + kPartFloats + blk::kRankMax) * sizeof(float);
    auto kern = block_score_topk_kernel<T, HH>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const bool vec = !(reinterpret_cast<uintptr_t>(pooled) & 15u) && d % 4 == 0;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // the most CTAs per row (a power of two, at most kMaxCl, at least 32 blocks each) whose clusters
    // are all resident at once (the occupancy query runs once per shape and device)
    static thread_local int64_t memo_rows = -1;
    static thread_local int memo_blocks = -1, memo_dev = -1, memo_cl = 1;
    int dev = 0;
    cudaGetDevice(&dev);
    int cl = kMaxCl;
    if (memo_rows == n_rows && memo_blocks == max_blocks && memo_dev == dev) {
        cl = memo_cl;
    } else {
        while (cl > 1 && max_blocks < cl * 32) cl >>= 1;
        for (; cl > 1; cl >>= 1) {
            attr[0].val.clusterDim.x = (unsigned)cl;
            cfg.gridDim = dim3((unsigned)(n_rows * cl));
            cfg.numAttrs = 1;
            int active = 0;
            if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active >= n_rows) break;
        }
        memo_rows = n_rows;
        memo_blocks = max_blocks;
        memo_dev = dev;
        memo_cl = cl;
    }
    attr[0].val.clusterDim.x = (unsigned)cl;
    cfg.gridDim = dim3((unsigned)(n_rows * cl));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, q, q_dtype, w, H, d, k, k_row_stride, k_rows, g, C, n_pooled, stale_pos,
                              pooled, pool_seq_stride, vec, top_k, scores, score_row_stride, idx, idx_row_stride,
                              n_sel);
}

template <typename T>
cudaError_t launch_h(const void* q, int q_dtype, const float* w, int H, int d, const T* k, int64_t k_row_stride,
                     int64_t k_rows, const Geom& g, int C, const int32_t* n_pooled, const int32_t* stale_pos,
                     float* pooled, int64_t pool_seq_stride, int top_k, float* scores, int64_t score_row_stride,
                     int32_t* idx, int64_t idx_row_stride, int32_t* n_sel, cudaStream_t st) {
#define LIDX_BLOCK_CASE(N)                                                                                     \
    return launch_t<T, N>(q, q_dtype, w, H, d, k, k_row_stride, k_rows, g, C, n_pooled, stale_pos, pooled,     \
                          pool_seq_stride, top_k, scores, score_row_stride, idx, idx_row_stride, n_sel, st)
    if (H <= 16) LIDX_BLOCK_CASE(16);
    if (H <= 32) LIDX_BLOCK_CASE(32);
    LIDX_BLOCK_CASE(64);
#undef LIDX_BLOCK_CASE
}

}  // namespace

// cudaErrorNotSupported: shapes the one launch does not take (the caller runs the three calls)
cudaError_t launch_block_score_topk(const void* q, int q_dtype, const float* w, int H, int d, const void* k_raw,
                                    int k_dtype, int64_t k_row_stride, int64_t k_rows, const Geom& g, int C,
                                    const int32_t* n_pooled, const int32_t* stale_pos, float* pooled,
                                    int64_t pool_seq_stride, int top_k, float* scores, int64_t score_row_stride,
                                    int32_t* idx, int64_t idx_row_stride, int32_t* n_sel, cudaStream_t st) {
    // the pooled-key scorer's split path (H in [9, 64]: 16 to 64 padded heads), one query row per
    // sequence, at most blk::kRankMax blocks per row, d within the shared-memory plan
    if (g.T != 1 || C < 2 || H < 9 || H > 64 || d < 1 || d > 256 || g.max_n_kv / C > blk::kRankMax ||
        g.max_n_kv / C < 1 || g.B < 1)
        return cudaErrorNotSupported;
    switch (k_dtype) {
        case IDX_F16:
            return launch_h(q, q_dtype, w, H, d, static_cast<const __half*>(k_raw), k_row_stride, k_rows, g, C,
                            n_pooled, stale_pos, pooled, pool_seq_stride, top_k, scores, score_row_stride, idx,
                            idx_row_stride, n_sel, st);
        case IDX_BF16:
            return launch_h(q, q_dtype, w, H, d, static_cast<const __nv_bfloat16*>(k_raw), k_row_stride, k_rows, g,
                            C, n_pooled, stale_pos, pooled, pool_seq_stride, top_k, scores, score_row_stride, idx,
                            idx_row_stride, n_sel, st);
        case IDX_F32:
            return launch_h(q, q_dtype, w, H, d, static_cast<const float*>(k_raw), k_row_stride, k_rows, g, C,
                            n_pooled, stale_pos, pooled, pool_seq_stride, top_k, scores, score_row_stride, idx,
                            idx_row_stride, n_sel, st);
        default:
            return cudaErrorNotSupported;
    }
}

}  // namespace lidx
