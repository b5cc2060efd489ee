// Block mean-pool of raw indexer keys:
//     p[b, beta, :] = (1/C) * sum_{t < C} k_raw[row(b, beta*C + t), :]
// for every complete block beta < floor(n_kv[b] / C).  Blocks are cuts of the
// position line measured from the sequence's first position, and the pooled
// key is the raw key's mean, before any norm or rotation (llama.cpp commit
// c88c916636, QSA commit message; llama-memory-hybrid-idx.h, kpool_layout).
//
// Incremental form: per sequence only blocks beta >= beta0 are written, with
// beta0 = min(n_pooled[b], floor(stale_pos[b]/C)) (llama-memory-hybrid-idx.h:
// pooled keys persist across batches; an edit stales every pool at or after
// it), so a decode step re-pools only what changed.
//
// One CTA of 128 threads per (block, sequence), striding over the blocks to
// (re)pool; the arithmetic of a block is blk::pool_block (block_ops.cuh), which
// the one-launch idx_block_score_topk shares.  A pure HBM stream: each raw key
// byte is read once and 1/C of it is written (as f32).
#include "block_ops.cuh"

namespace lidx {
namespace {

constexpr int kThreads = blk::kPoolThreads;

template <typename T>
__global__ void __launch_bounds__(kThreads) pool_kernel(const T* k, int64_t k_row_stride,
                                                        int64_t k_rows, Geom g, int C, int d,
                                                        float* __restrict__ pooled,
                                                        int64_t pool_seq_stride,
                                                        const int32_t* __restrict__ n_pooled,
                                                        const int32_t* __restrict__ stale_pos) {
    extern __shared__ float part[];  // [RP][d]
    const int b = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const int n_cb = seq_n_kv(g, b) / C;
    const int beta0 = blk::pool_first_block(n_pooled, stale_pos, b, C, n_cb);
    for (int beta = beta0 + (int)blockIdx.x; beta < n_cb; beta += gridDim.x)
        blk::pool_block(k, k_row_stride, k_rows, g, C, d, b, beta, part,
                        pooled + ((int64_t)b * pool_seq_stride + beta) * d);
}

template <typename T>
cudaError_t run(const T* k, int64_t k_row_stride, int64_t k_rows, const Geom& g, int C, int d,
                float* pooled, int64_t pool_seq_stride, const int32_t* n_pooled, const int32_t* stale_pos,
                cudaStream_t st) {
    const int max_blocks = g.max_n_kv / C;
    if (max_blocks == 0 || g.B == 0) return cudaSuccess;
    constexpr int V = 16 / sizeof(T);
    const int tpr = d / V;
    const int rp = kThreads / tpr;
    const size_t sm = (size_t)rp * d * sizeof(float);
    // a full pooling covers every block; an update usually re-pools few blocks per sequence, so a
    // few CTAs per sequence stride over them (most of a full-size grid would only exit)
    int gx = max_blocks < 65535 ? max_blocks : 65535;
    if (n_pooled || stale_pos) {
        int sms = sm_count();
        if (sms < 2) sms = 152;
        const int want = (2 * sms + g.B - 1) / g.B;
        if (gx > want) gx = want;
    }
    dim3 grid((unsigned)gx, (unsigned)g.B);
    return launch_pdl(pool_kernel<T>, grid, dim3(kThreads), sm, st, k, k_row_stride, k_rows, g, C, d, pooled,
                      pool_seq_stride, n_pooled, stale_pos);
}

}  // namespace

cudaError_t launch_block_pool(const void* k_raw, int k_dtype, int64_t k_row_stride, int64_t k_rows,
                              const Geom& g, int C, int d, float* pooled, int64_t pool_seq_stride,
                              const int32_t* n_pooled, const int32_t* stale_pos, cudaStream_t st) {
    switch (k_dtype) {
        case IDX_F16:
            return run(static_cast<const __half*>(k_raw), k_row_stride, k_rows, g, C, d, pooled,
                       pool_seq_stride, n_pooled, stale_pos, st);
        case IDX_BF16:
            return run(static_cast<const __nv_bfloat16*>(k_raw), k_row_stride, k_rows, g, C, d,
                       pooled, pool_seq_stride, n_pooled, stale_pos, st);
        default:
            return run(static_cast<const float*>(k_raw), k_row_stride, k_rows, g, C, d, pooled,
                       pool_seq_stride, n_pooled, stale_pos, st);
    }
}

}  // namespace lidx
