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
// blocks four threads per block key and writes each score both to the scores
// output and into rank 0's shared memory; after a cluster barrier rank 0 ranks
// the row's blocks and writes the selection.  Decode rows only (one query row
// per sequence: the pooled cache is per sequence, so rows of one sequence
// would pool the same blocks).
#include "block_ops.cuh"
#include "sm100_ptx.cuh"

namespace lidx {
namespace {

constexpr int kThreads = 512;   // the block rank's CTA size: rows of at most 512 blocks
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
    float* sc = part + kPartFloats;    // rank 0: the row's block scores
    __shared__ blk::RankShared rs;
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
    const uint32_t sc0 = sm100::mapa(sc, 0);
    const int je = min(j1, n_cb);
    for (int jb = j0; jb < je; jb += kThreads / 4) {
        const int j = jb + (int)(threadIdx.x >> 2), hg = threadIdx.x & 3;
        const bool valid = j < je;
        const float v = blk::score_split_sum(
            valid ? blk::score_split_part<float, HH>(qs, ws, prow + (int64_t)j * d, d, hg, vec) : 0.f);
        if (valid && hg == 0) {
            scores[r * score_row_stride + j] = v;
            sm100::st_cluster_f32(sc0 + 4u * (uint32_t)j, v);
        }
    }
    // 3. rank 0 selects once every CTA's scores are in its shared memory
    sm100::cluster_sync();
    if (rank != 0) return;
    blk::block_rank_row<kThreads>(sc, n_vis, top_k, C, idx + r * idx_row_stride, n_sel ? n_sel + r : nullptr, rs);
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
    // are all resident at once
    int cl = kMaxCl;
    while (cl > 1 && max_blocks < cl * 32) cl >>= 1;
    for (; cl > 1; cl >>= 1) {
        attr[0].val.clusterDim.x = (unsigned)cl;
        cfg.gridDim = dim3((unsigned)(n_rows * cl));
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active >= n_rows) break;
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
    // sequence, at most 512 blocks per row, d within the shared-memory plan
    if (g.T != 1 || C < 2 || H < 9 || H > 64 || d < 1 || d > 256 || g.max_n_kv / C > kThreads ||
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
