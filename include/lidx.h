/*
 * lidx.h -- C ABI of the lightning-indexer sparse-attention library (liblidx.so).
 *
 * The path: score every visible cached key with the lightning indexer, select
 * the top_k keys per query row, and run softmax attention over only those
 * keys.  Also the block-pooled variant: one mean-pooled key per block of C
 * positions, whole blocks plus the incomplete tail.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers named in the argument lists are DEVICE pointers unless said
 *    otherwise.  The caller owns every buffer; the library allocates nothing,
 *    synchronises nothing and only enqueues kernels on `stream` (NULL = the
 *    legacy default stream).  Calls are asynchronous.
 *  - Arguments are validated on the host before anything is launched.  A bad
 *    argument returns IDX_ERR_INVALID_ARG (or IDX_ERR_UNSUPPORTED for a valid
 *    but unimplemented shape/dtype) and launches nothing; idx_last_error()
 *    then returns a message for the calling thread.  Nothing aborts.
 *  - A failed launch returns IDX_ERR_CUDA.  Data-dependent faults the host
 *    cannot see (an index outside its sequence, a key row outside the
 *    allocation, a bounded wait that ran out) are never followed: the kernel
 *    skips the access and records the fault in a device status word, read by
 *    idx_device_status().
 *  - Element strides and row strides are in ELEMENTS of the named dtype.
 *  - Query rows: a batch has n_seq sequences of n_q_per_seq query rows each;
 *    query row r = b * n_q_per_seq + t belongs to sequence b.
 *  - Key positions are relative to the sequence: position j of sequence b is
 *    cache row kv_start[b] + j (or b * kv_seq_stride + j).  Indices returned
 *    by idx_topk are such positions.
 */
#ifndef LIDX_H
#define LIDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, without requiring the CUDA headers. */
typedef struct CUstream_st* idx_stream_t;

typedef enum idx_status {
    IDX_OK = 0,
    IDX_ERR_INVALID_ARG = 1,
    IDX_ERR_UNSUPPORTED = 2,
    IDX_ERR_CUDA = 3,
    IDX_ERR_TIMEOUT = 4,      /* device status only: a bounded wait ran out */
    IDX_ERR_DEVICE_BOUNDS = 5, /* device status only: an out-of-range index or row was skipped */
    IDX_ERR_INEXACT = 6        /* device status only: a query value overflowed the type the scorer
                                  converts it to (bf16 q of magnitude >= 65520 against F16 keys) */
} idx_status;

typedef enum idx_dtype {
    IDX_F32 = 0,
    IDX_F16 = 1,
    IDX_BF16 = 2
} idx_dtype;

/*
 * Batch geometry shared by the calls below.
 *   n_seq          B >= 0 sequences.
 *   n_q_per_seq    T >= 1 query rows per sequence (decode: 1).
 *   n_kv           device int32[B]: cached tokens of sequence b.  A decode
 *                  query's own key is written to the cache before scoring, so
 *                  n_kv counts it (ik_llama.cpp PR #2058, commit
 *                  "decode-correct via persistent indexer-K cache").
 *   kv_start       device int32[B] or NULL: cache row of position 0 of
 *                  sequence b.  NULL means b * kv_seq_stride.
 *   kv_seq_stride  rows between sequences when kv_start is NULL.
 *   q_pos          device int32[B*T] or NULL: position of each query row.
 *                  Key j is visible to row r iff j < n_kv[b] and, when q_pos
 *                  is given, j <= q_pos[r] (the causal mask, ik_llama.cpp PR
 *                  #2058, commit "Add GLM-5.2/DeepSeek-V3.2 DSA lightning
 *                  indexer").  n_vis(r) = min(q_pos[r] + 1, n_kv[b]), >= 0.
 *   max_n_kv       host-side bound: every n_kv[b] <= max_n_kv.  It sizes the
 *                  grids; a larger n_kv[b] is clamped to it and flagged.
 *   page_table     device int32 or NULL.  Paged caches: position j of sequence
 *                  b lives in cache row
 *                      page_table[b*page_table_stride + j/page_size]*page_size
 *                      + j % page_size
 *                  (kv_start and kv_seq_stride are then unused).  Cache cells
 *                  need not follow positions; blocks and the causal bound stay
 *                  cuts of the position line (llama.cpp commit c88c916636, QSA
 *                  commit message: blocks are cuts of the position line, not of
 *                  the cell array; ik_llama.cpp PR #2058 "UPDATE 5": several
 *                  sequences share one cell array).  A row outside the cache is
 *                  never read (flagged, as for kv_start).
 *   page_table_stride  entries per sequence in page_table.
 *   page_size      rows per page, >= 1 when page_table is given (a multiple
 *                  of 64 keeps the tensor-core scorers; other sizes run on the
 *                  CUDA cores).
 */
/* top_k = -1 selects this (see idx_topk) */
#define IDX_DEFAULT_TOP_K 2048

typedef struct idx_batch {
    int32_t n_seq;
    int32_t n_q_per_seq;
    const int32_t* n_kv;
    const int32_t* kv_start;
    int64_t kv_seq_stride;
    const int32_t* q_pos;
    int32_t max_n_kv;
    const int32_t* page_table;
    int64_t page_table_stride;
    int32_t page_size;
} idx_batch;

/*
 * idx_hadamard -- rotate rows by the orthonormal Sylvester Walsh-Hadamard
 * matrix H_d (natural order, entries (-1)^popcount(i&j)/sqrt(d)): y = H_d x.
 * Score preserving: (Hq).(Hk) = q.k (ik_llama.cpp PR #2058, commit "Add
 * GLM-5.2/DeepSeek-V3.2 DSA lightning indexer"; applied to cached keys and to
 * queries in commit "decode-correct via persistent indexer-K cache").
 *   x, y       device [n_rows] rows of d elements, row r at x + r*row_stride
 *              (y likewise).  y may equal x (in place); other overlap is
 *              not allowed.
 *   dtype      storage type of x and y; y is the exact rotation rounded
 *              once (nearest even) to dtype (16-bit types: f32 butterflies
 *              with a certified error bound, the few elements the bound
 *              cannot decide recomputed in f64; f32: computed in f64).
 *   d          32, 64, 128 or 256.
 * Errors: INVALID_ARG for x or y NULL with n_rows > 0, n_rows < 0,
 * unsupported d, row_stride < d, or x, y not 16-byte aligned or
 * row_stride*size not a multiple of 16 bytes.
 */
idx_status idx_hadamard(const void* x, void* y, idx_dtype dtype, int64_t n_rows, int32_t d,
                        int64_t row_stride, idx_stream_t stream);

/*
 * idx_score -- lightning-indexer scores
 *     s[r, j] = sum_h w[r, h] * max(0, q[r, h, :] . k[j, :])      (f32 out)
 * for every visible key j of every query row r, accumulated in f32 (ik_llama_opt
 * commit log, "openpangu: DSA lightning indexer + SWA schedule"; ReLU per head
 * before the head sum: llama.cpp commit c88c916636, QSA commit message).
 *   q          [B*T, H, d] contiguous, q_dtype.
 *   w          f32 [B*T, H]: per-row, per-head weights (the indexer projection
 *              of the token; it carries every scale).
 *   k          one shared (MQA) key row of d elements per cached token, row i
 *              at k + i*k_row_stride; k_rows = rows in the allocation.
 *   block_size 0 or 1: token keys, row r sees n_vis(r) keys.  C > 1: k holds
 *              pooled block keys (idx_block_pool) addressed by kv_start /
 *              kv_seq_stride in BLOCK rows, and row r sees floor(n_vis(r)/C)
 *              blocks (only complete blocks are scored).
 *   scores     f32, row r at scores + r*score_row_stride; entries j of
 *              visible keys are written, the rest of the row is untouched.
 *   workspace  may be NULL when idx_workspace_size(IDX_OP_SCORE, ...) is 0.
 * Supported: q_dtype, k_dtype in {F32, F16, BF16}, H <= 64, d <= 256 and
 * H*d <= 16384.  H = 64, d = 128 with F16/BF16 keys runs on the tensor cores
 * when q converts exactly to the key type: the same type, or bf16 q with F16
 * keys (bf16's 8-bit significand fits f16's 11 bits).  A bf16 q element of
 * magnitude >= 65520 does not fit f16's range: it is staged as +-inf and
 * IDX_ERR_INEXACT is recorded in the device status; elements below f16's
 * normal range (2^-14) keep their f16 rounding, an error of at most 2^-25
 * each.  Every other combination (f32 q, f16 q with BF16 keys) runs on the
 * CUDA cores in f32 with q as given.
 */
idx_status idx_score(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads,
                     int32_t head_dim, const void* k, idx_dtype k_dtype, int64_t k_row_stride,
                     int64_t k_rows, idx_batch batch, int32_t block_size, float* scores,
                     int64_t score_row_stride, void* workspace, size_t workspace_bytes,
                     idx_stream_t stream);

/*
 * idx_quantize_rows -- per-row symmetric 8-bit code of a key cache row, the
 * storage format of a quantized indexer key cache ("GLM-DSA: allow for
 * quantized indexer cache", ik_llama_opt commit log; like the q8_0 latent
 * cache there, "a storage format only": scores use the dequantized values).
 * For each row r, in f32 arithmetic (round to nearest even):
 *     scale[r] = max_c |x[r, c]| / 127
 *     q8[r, c] = clamp(rint(x[r, c] / scale[r]), -127, 127)   (0 when scale = 0)
 * so x ~= scale[r] * q8[r, c] with |error| <= scale/2.
 *   x          device [n_rows] rows of d elements at x + r*x_row_stride, x_dtype.
 *   q8         device int8, row r at q8 + r*q8_row_stride (bytes).
 *   scale      device f32 [n_rows], or NULL: each row's scale is stored inline
 *              in bytes d .. d+3 of its code row (d % 4 == 0, q8_row_stride
 *              >= d + 4; for d = 128 a 144-byte row keeps TMA alignment).
 * Errors: INVALID_ARG for NULL pointers with n_rows > 0, d < 1 or d > 1024,
 * strides < d, or q8 / q8_row_stride not 16-byte aligned.
 */
idx_status idx_quantize_rows(const void* x, idx_dtype x_dtype, int64_t n_rows, int32_t d, int64_t x_row_stride,
                             int8_t* q8, int64_t q8_row_stride, float* scale, idx_stream_t stream);

/*
 * idx_score_q8 -- idx_score over a quantized key cache (idx_quantize_rows):
 *     s[r, j] = sum_h w[r, h] * max(0, q[r, h, :] . (scale[j] * k8[j, :]))
 * i.e. the indexer score of the dequantized keys (ik_llama_opt commit log,
 * "GLM-DSA: allow for quantized indexer cache"; the score itself as in
 * idx_score).  A key row costs d + 4 bytes instead of 2d.
 *   k8         device int8 key rows, row i at k8 + i*k_row_stride (bytes).
 *   k_scale    device f32, k_scale[i] for cache row i (any sign), or NULL for
 *              inline scales (bytes head_dim .. head_dim+3 of each row, as
 *              idx_quantize_rows writes them with scale NULL).
 *   other arguments as idx_score (block_size 0/1 only).
 * H = 64, d = 128 decode rows (T = 1) with f16 or bf16 q run on the tensor
 * cores: the int8 codes are widened exactly to f16 in shared memory, q is
 * converted to f16 (exact for bf16 q inside f16's normal range; beyond it
 * IDX_ERR_INEXACT is recorded, as for idx_score), and the scale is applied
 * per head before the ReLU.  Everything else runs on the CUDA cores.
 */
idx_status idx_score_q8(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                        const int8_t* k8, int64_t k_row_stride, const float* k_scale, int64_t k_rows,
                        idx_batch batch, int32_t block_size, float* scores, int64_t score_row_stride,
                        void* workspace, size_t workspace_bytes, idx_stream_t stream);

/*
 * idx_block_pool -- mean-pooled raw key of every complete block
 *     p[b, beta, :] = (1/C) * sum_{t=beta*C}^{beta*C+C-1} k_raw[row(b, t), :]
 * for beta < floor(n_kv[b] / C).  Blocks are cuts of the position line from
 * the sequence's first position, and pooling takes the raw key, before any
 * norm or rotation (llama.cpp commit c88c916636, QSA commit message;
 * llama-memory-hybrid-idx.h, kpool_layout).  Sums in f32.
 *   k_raw      rows addressed by batch.kv_start / kv_seq_stride, k_dtype.
 *   pooled     f32, block beta of sequence b at
 *              pooled + (b*pool_seq_stride + beta)*head_dim.
 * Errors: INVALID_ARG for block_size < 1, pool_seq_stride < max_n_kv/C.
 */
idx_status idx_block_pool(const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride,
                          int64_t k_rows, idx_batch batch, int32_t block_size, int32_t head_dim,
                          float* pooled, int64_t pool_seq_stride, idx_stream_t stream);

/*
 * idx_block_pool_update -- incremental maintenance of a persistent pooled-key
 * cache: only the blocks that changed are (re)pooled.  The pooled keys live
 * across decode steps; a step appends tokens, so only blocks completed since
 * the last pooling are new, and a sequence edit from position p on regroups
 * the blocks from the one holding p, staling every pooled key at or after it
 * (llama-memory-hybrid-idx.h: "The pooled keys persist in the idx cache
 * across batches", mem_idx_stale / POS_CLEAN, get_n_kpool_new "pools to
 * re-pool this ubatch").  For sequence b, with n_cb = floor(n_kv[b]/C):
 *     beta0 = min(n_pooled[b], floor(stale_pos[b] / C))   clamped to [0, n_cb]
 * and the blocks beta0 <= beta < n_cb are written exactly as idx_block_pool
 * writes them; every other pooled row is left untouched.
 *   n_pooled   device int32 [n_seq] or NULL (= 0): complete blocks of sequence
 *              b whose pooled keys are current.  The caller keeps this count
 *              (after the call it is n_cb); the library does not write it.
 *   stale_pos  device int32 [n_seq] or NULL (= no edit): first position whose
 *              raw key changed since those blocks were pooled; IDX_POS_CLEAN
 *              means none, a negative value the whole sequence.
 * Other arguments and errors as idx_block_pool.
 */
#define IDX_POS_CLEAN INT32_MAX
idx_status idx_block_pool_update(const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride,
                                 int64_t k_rows, idx_batch batch, const int32_t* n_pooled,
                                 const int32_t* stale_pos, int32_t block_size, int32_t head_dim,
                                 float* pooled, int64_t pool_seq_stride, idx_stream_t stream);

/*
 * idx_topk -- per-row selection, positions ascending.
 * top_k = -1 means the model's configured indexer top_k ("GLM-DSA: convert
 *   sparse-attention control from env vars to CLI args": dsa_top_k default -1
 *   == the model's indexer_top_k), IDX_DEFAULT_TOP_K = 2048 for the models the
 *   pages run; idx_workspace_size maps -1 the same way.
 * Token mode (block_size 0 or 1): K = min(top_k, n_vis(r)) positions with
 *   the largest scores; equal scores: the lower position wins; -0 == +0.
 *   ("ggml_top_k(min(top_k, n_tokens))", ik_llama.cpp PR #2058.)
 * Block mode (block_size C > 1; scores are block scores from idx_score in
 *   block mode): the best min(floor(top_k/C), n_cb) complete blocks (lower
 *   block index wins ties), every token of those blocks, plus every tail
 *   token [n_cb*C, n_vis) -- exactly dense when n_vis <= top_k + C - 1
 *   (llama.cpp commit c88c916636, QSA commit message).
 *   idx        int32, row r at idx + r*idx_row_stride.  Capacity: top_k in
 *              token mode, floor(top_k/C)*C + C - 1 in block mode; entries
 *              past the selection up to that capacity are set to -1.
 *   n_sel      int32[B*T] or NULL: number of positions selected per row.
 * Scores must be finite (a NaN is ordered like a value, never trusted).
 */
idx_status idx_topk(const float* scores, int64_t score_row_stride, idx_batch batch,
                    int32_t top_k, int32_t block_size, int32_t* idx, int64_t idx_row_stride,
                    int32_t* n_sel, void* workspace, size_t workspace_bytes,
                    idx_stream_t stream);

/*
 * idx_block_score_topk -- the indexer of a block-pooled decode step in one
 * call: idx_block_pool_update (raw keys -> the persistent pooled-key cache),
 * idx_score over the pooled keys (block_size C) and idx_topk in block mode,
 * with their results bit for bit (llama.cpp commit c88c916636, QSA commit
 * message: block keys are the mean of the block's raw keys, a query keeps its
 * best floor(top_k/C) complete blocks and the tail; the pooled keys persist
 * across decode steps, llama-memory-hybrid-idx.h).  Decode rows
 * (n_q_per_seq 1) with 9 to 64 heads and at most 1024 blocks per row run as
 * one launch (a cluster of CTAs per row: each re-pools and scores its share of
 * the row's blocks, the first ranks them); other shapes run the three calls.
 *   q, w, n_heads, head_dim   as idx_score; k_raw, k_dtype, k_row_stride,
 *              k_rows, batch  the raw key cache as idx_block_pool_update reads
 *              it (batch also gives n_kv, q_pos and n_q_per_seq of the rows);
 *   n_pooled, stale_pos, block_size, pooled, pool_seq_stride  as
 *              idx_block_pool_update (pooled is updated in place and scored
 *              from: block beta of sequence b at pooled + (b*pool_seq_stride +
 *              beta)*head_dim);
 *   top_k, scores, score_row_stride, idx, idx_row_stride, n_sel  as idx_score
 *              (block scores, floor(max_n_kv / C) per row) and idx_topk in
 *              block mode.
 * Errors: those of the three calls.
 */
idx_status idx_block_score_topk(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                                const void* k_raw, idx_dtype k_dtype, int64_t k_row_stride, int64_t k_rows,
                                idx_batch batch, const int32_t* n_pooled, const int32_t* stale_pos,
                                int32_t block_size, float* pooled, int64_t pool_seq_stride, int32_t top_k,
                                float* scores, int64_t score_row_stride, int32_t* idx, int64_t idx_row_stride,
                                int32_t* n_sel, idx_stream_t stream);

/*
 * idx_score_topk -- the fused indexer + selection: idx_score (token keys)
 * followed by idx_topk, with the same results, in one call (ik_llama_opt
 * commit log, "Route DSA indexer selection through ggml_indexer_topk": the
 * selection of the lightning indexer as one op, with no per-head score
 * tensor).  Decode rows (n_q_per_seq 1) with H = 64, d = 128 16-bit keys and
 * fewer than 2 x SMs rows run fused: the tensor-core scorer also counts each
 * row's scores into a 2048-bin histogram of their order key's top 11 bits,
 * which fixes the bin of the top_k-th score exactly, so the select only
 * ranks the keys of that one bin.  Other shapes run idx_score + idx_topk.
 *   Arguments as idx_score (block_size 0) and idx_topk (token mode); scores
 *   are written as idx_score writes them.
 *   workspace  idx_workspace_size(IDX_OP_SCORE_TOPK, ...) bytes, 16-byte
 *              aligned; with less (or NULL) the call runs unfused.
 * The fused scorer zeroes its histograms itself behind a bounded barrier
 * across its CTAs (one per SM); if that barrier times out (the device was
 * shared with work that held SMs for seconds) IDX_ERR_TIMEOUT is recorded in
 * the device status and the select falls back to ranking every score, so the
 * result stays exact.
 */
idx_status idx_score_topk(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                          const void* k, idx_dtype k_dtype, int64_t k_row_stride, int64_t k_rows, idx_batch batch,
                          int32_t top_k, float* scores, int64_t score_row_stride, int32_t* idx,
                          int64_t idx_row_stride, int32_t* n_sel, void* workspace, size_t workspace_bytes,
                          idx_stream_t stream);

/*
 * sparse_attn_decode / sparse_attn_prefill -- softmax attention of each
 * query row over only its selected keys:
 *     l[h, j] = scale * q[r, h, :] . K[j, g(h), :],  p = softmax_j(l),
 *     out[r, h, :] = sum_j p[h, j] * V[j, g(h), :],   g(h) = h / (Hq / Hkv)
 * for j in idx[r, 0 : n_sel[r]] ("Gather OpenPangu DSA decode reads" and
 * "Gather OpenPangu sparse prefill attention", ik_llama_opt commit log).
 *   q          [B*T, Hq, dk] contiguous, dtype.
 *   k          row i at k + i*kv_row_stride holds [Hkv, dk] contiguous.
 *   v          row i at v + i*v_row_stride holds [Hkv, dv]; NULL selects the
 *              MLA latent form: Hkv must be 1 and V = the first dv columns
 *              of the same K row ("openpangu: MLA-latent KV cache").
 *   kv_rows    rows in the K (and V) allocation.
 *   idx/n_sel  as written by idx_topk (positions of sequence b, -1 padding
 *              ignored); n_sel[r] in [1, idx_row_stride].  A row with
 *              n_sel[r] == 0 gets zeros.
 *   out        [B*T, Hq, dv] contiguous, out_dtype (F32 or BF16).
 *   workspace  idx_workspace_size(IDX_OP_ATTN, ...) bytes (16-byte aligned)
 *              or NULL when that is 0; used for split-key partial results.
 * dtype in {F32, F16, BF16}; dk <= 576, dv <= 512, Hq % Hkv == 0.  The two
 * entry points compute the same function; decode is tuned for few rows with
 * long selections, prefill for many rows.
 */
idx_status sparse_attn_decode(const void* q, idx_dtype dtype, int32_t n_q_heads, int32_t n_kv_heads,
                              int32_t dk, int32_t dv, const void* k, const void* v,
                              int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows,
                              idx_batch batch, const int32_t* idx, int64_t idx_row_stride,
                              const int32_t* n_sel, float scale, void* out, idx_dtype out_dtype,
                              void* workspace, size_t workspace_bytes, idx_stream_t stream);

idx_status sparse_attn_prefill(const void* q, idx_dtype dtype, int32_t n_q_heads, int32_t n_kv_heads,
                               int32_t dk, int32_t dv, const void* k, const void* v,
                               int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows,
                               idx_batch batch, const int32_t* idx, int64_t idx_row_stride,
                               const int32_t* n_sel, float scale, void* out, idx_dtype out_dtype,
                               void* workspace, size_t workspace_bytes, idx_stream_t stream);

/*
 * sparse_attn_decode_noalloc -- sparse_attn_decode's 128-head MLA latent
 * attention for callers that cannot allocate device memory: programs that
 * own all device memory through their own pool or arena (serving engines,
 * frameworks embedding this library), for which a cudaMalloc would fall
 * outside their accounting and could block or synchronise the device.
 * The source pages have no counterpart to this entry point.
 *   Same arguments and result as sparse_attn_decode with v == NULL, minus
 *   the workspace: the key-split partials go to a static device array of
 *   20,000,768 bytes that belongs to the library (held by every GPU that
 *   loads it until the process exits).
 *   Supported: dtype BF16, n_q_heads 128, n_kv_heads 1, dk 576, dv 512,
 *   16-byte aligned q/k/out, kv_row_stride % 8 == 0 (else UNSUPPORTED);
 *   kv_row_stride < 576 (overlapping, zero or negative) is INVALID_ARG.
 *   On a device with at most 152 SMs (a GB300) the array covers every
 *   split of rows selecting at most 2048 keys; a call whose partials would
 *   not fit (rows selecting more keys, or a device with more SMs, where the
 *   split policy may use more units) returns INVALID_ARG without launching
 *   anything.  The array is shared by all calls and keeps
 *   the last call's contents (nothing in it must start at zero); calls whose
 *   work overlaps on the GPU race on it and must be serialised by the caller.
 *   The first call on each device, with that device current, looks up the
 *   array's device address; make that call before any stream capture.
 */
idx_status sparse_attn_decode_noalloc(const void* q, idx_dtype dtype, int32_t n_q_heads, int32_t n_kv_heads,
                                      int32_t dk, int32_t dv, const void* k, int64_t kv_row_stride,
                                      int64_t kv_rows, idx_batch batch, const int32_t* idx,
                                      int64_t idx_row_stride, const int32_t* n_sel, float scale, void* out,
                                      idx_dtype out_dtype, idx_stream_t stream);

/*
 * sparse_decode_step -- one decode step of the sparse attention: the
 * indexer's scores and top-k selection (idx_score_topk) followed by the
 * attention over the selected keys (sparse_attn_decode), with the results of
 * those two calls (scores, idx, n_sel and out are all written).  The pages'
 * fused indexer + top-k ("Route DSA indexer selection through
 * ggml_indexer_topk") feeding the gathered decode ("Gather OpenPangu DSA
 * decode reads", ik_llama_opt commit log).
 *   Indexer arguments as idx_score_topk; attention arguments as
 *   sparse_attn_decode (q_attn with attn_dtype, n_q_heads, n_kv_heads, dk,
 *   dv, k_attn, v_attn, strides and kv_rows).
 *   workspace  idx_workspace_size(IDX_OP_DECODE_STEP, n_rows, max_n_kv,
 *              top_k, n_q_heads, dv) bytes, 16-byte aligned.
 * Few short decode rows run as ONE launch (a grid of 2-CTA clusters resident
 * at once: each CTA scores a share of the key tiles, the CTA finishing a row
 * selects it, each cluster then attends one (row, key split) unit, and the
 * splits are merged after a grid barrier): n_q_per_seq 1, at most 32 rows,
 * max_n_kv <= 16384, the indexer at 64 heads x 128 with 16-bit keys (q of
 * the keys' type, or BF16 q with F16 keys), the 128-head MLA latent
 * attention (BF16, dk 576, dv 512, v_attn NULL), 16-byte aligned tensors,
 * and rows x key splits no more than the clusters the device holds at once.
 * The scores, the selection and (with the same key splits) the output are
 * bit for bit those of the two calls.  Anything else runs the two calls.
 * The fused launch waits on flags other CTAs of the same launch raise (all
 * bounded, ~2 s; a timeout records IDX_ERR_TIMEOUT in the device status).
 * Its flags and counters use one of 256 slots of a library-owned device
 * array, taken round-robin per call; more than 256 fused calls in flight on
 * one device at once (across streams) would share a slot and must not run.
 */
idx_status sparse_decode_step(const void* q, idx_dtype q_dtype, const float* w, int32_t n_heads, int32_t head_dim,
                              const void* k, idx_dtype k_dtype, int64_t k_row_stride, int64_t k_rows,
                              idx_batch batch, int32_t top_k, float* scores, int64_t score_row_stride, int32_t* idx,
                              int64_t idx_row_stride, int32_t* n_sel, const void* q_attn, idx_dtype attn_dtype,
                              int32_t n_q_heads, int32_t n_kv_heads, int32_t dk, int32_t dv, const void* k_attn,
                              const void* v_attn, int64_t kv_row_stride, int64_t v_row_stride, int64_t kv_rows,
                              float scale, void* out, idx_dtype out_dtype, void* workspace, size_t workspace_bytes,
                              idx_stream_t stream);

/*
 * sparse_decode_step_fused -- 1 when a sparse_decode_step call with these
 * sizes runs as one launch on the current device (given the supported
 * dtypes, head counts, alignment and a workspace of
 * idx_workspace_size(IDX_OP_DECODE_STEP, ...) bytes), else 0.  Host only;
 * the first call per device queries how many clusters the device holds.
 */
int32_t sparse_decode_step_fused(int64_t n_rows, int32_t n_q_per_seq, int32_t max_n_kv, int32_t top_k,
                                 int64_t idx_row_stride);

/* Operation selectors for idx_workspace_size. */
enum {
    IDX_OP_SCORE = 0,
    IDX_OP_TOPK = 1,
    IDX_OP_ATTN_DECODE = 2,
    IDX_OP_ATTN_PREFILL = 3,
    IDX_OP_SCORE_TOPK = 4,
    IDX_OP_DECODE_STEP = 5
};

/*
 * idx_workspace_size -- bytes of device workspace an operation needs for the
 * given sizes (0 when none).  n_rows = B*T query rows; the other arguments are
 * the same as the call's.  Pure host arithmetic; never fails (returns 0 for
 * nonsense sizes, which the call itself then rejects).
 */
size_t idx_workspace_size(int32_t op, int64_t n_rows, int32_t max_n_kv, int32_t top_k,
                          int32_t n_q_heads, int32_t dv);

/* Message for the last non-OK status returned on the calling thread. */
const char* idx_last_error(void);

/*
 * idx_device_status -- synchronise the current device and return the first
 * data-dependent fault recorded by a kernel since the last reset
 * (IDX_ERR_DEVICE_BOUNDS, IDX_ERR_TIMEOUT) or IDX_OK; reset != 0 clears it.
 * Returns IDX_ERR_CUDA if the synchronisation itself fails.
 */
idx_status idx_device_status(int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* LIDX_H */
