// lidx_oracle.cpp -- plain C++17 CPU oracle of the lightning-indexer
// sparse-attention path (score -> causal bound -> top-k -> sparse attention,
// and the block-pooled variant).
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
// CPU-baseline / reference legs load this library.  It includes no CUDA header
// and shares no source with the GPU library; it is a second, independent
// restatement of the method next to the numpy oracle (lidx_oracle.py), and the
// pins in tests/test_oracle_pins.py run against both.
//
// Every input is read as stored (f16 / bf16 / f32 widened exactly to double)
// and every sum is taken in double, in the index order the definition names;
// OpenMP only spreads independent query rows over the host cores.
//
// Sources (page title, then the part of the page):
//  * ik_llama.cpp PR #2058 (GLM-DSA lightning indexer), commit "Add
//    GLM-5.2/DeepSeek-V3.2 DSA lightning indexer": per-head relu(q_h . k)
//    weighted by the indexer projection and summed over heads, the causal
//    mask, top_k(min(top_k, n_tokens)); the Walsh-Hadamard rotation is
//    orthonormal, so (Hq).(Hk) = q.k.
//  * same PR, commit "decode-correct via persistent indexer-K cache": the
//    decode key is in the cache before scoring; the cache holds rotated keys.
//  * ik_llama_opt commit log, "openpangu: DSA lightning indexer + SWA
//    schedule" (score = sum_g w_g relu(q_g . k)), "Gather OpenPangu DSA decode
//    reads" (softmax over only the gathered rows) and "openpangu: MLA-latent
//    KV cache" (the value is the leading 512 columns of the latent row);
//    "GLM-DSA: allow for quantized indexer cache" (a storage format only).
//  * llama.cpp commit c88c916636 (QSA), commit message: one mean-pooled raw
//    key per block of compress_ratio positions, a budget of whole blocks plus
//    the incomplete tail, block scores expanded to members by a gather.
//  * llama-memory-hybrid-idx.h: pooled keys persist across batches; an edit
//    from position p stales every pooled key at or after p's block.
//
// Readings where the pages leave a step open (the same as the numpy oracle):
// ties go to the lower position (lower block index); -0 == +0; the selection
// is returned in ascending position order padded with -1; w is one f32 weight
// per (query row, head) and carries every scale; the block budget is
// floor(top_k / C) whole blocks with the tail outside it; the Hadamard
// rotation is exact and rounded once to the storage type; the int8 cache
// stores scale = max|x| / 127 and codes rint(x / scale) clamped to +-127, in
// f32; attention over an empty selection is 0 (the batch form only).
#include <omp.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// storage formats of the arrays handed in
enum Fmt { F64 = 0, F32 = 1, F16 = 2, BF16 = 3, I8 = 4 };

// IEEE binary16 bit pattern -> its exact value
double widen_f16(uint16_t h) {
    const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = std::ldexp((double)m, -24);                 // subnormal: m * 2^-24
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = std::ldexp((double)(1024 + m), e - 25);     // (1.m) * 2^(e-15)
    return sign ? -v : v;
}

// bfloat16 bit pattern -> its exact value (the top half of an f32)
double widen_bf16(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// element i of an array stored in `fmt` (I8: the integer code itself)
double elem(const void* p, int fmt, int64_t i) {
    switch (fmt) {
        case F64: return static_cast<const double*>(p)[i];
        case F32: return (double)static_cast<const float*>(p)[i];
        case F16: return widen_f16(static_cast<const uint16_t*>(p)[i]);
        case BF16: return widen_bf16(static_cast<const uint16_t*>(p)[i]);
        default: return (double)static_cast<const int8_t*>(p)[i];
    }
}

// Round x to the storage format once, to nearest with ties to even: a value
// with 2^E <= |x| < 2^(E+1) is rounded to a multiple of 2^(E - p + 1), with E
// clamped at the smallest normal exponent (subnormal spacing); beyond the
// largest finite value it becomes +-inf.
double round_storage(double x, int fmt) {
    if (fmt == F64 || x == 0.0 || !std::isfinite(x)) return x;
    int p, emin;
    double fmax;
    if (fmt == F32) {
        p = 24; emin = -126; fmax = (double)FLT_MAX;
    } else if (fmt == F16) {
        p = 11; emin = -14; fmax = 65504.0;
    } else {
        p = 8; emin = -126; fmax = std::ldexp(255.0, 120);   // 0x1.fep127
    }
    int e = 0;
    std::frexp(x, &e);                // |x| = m * 2^e with m in [0.5, 1)
    int E = e - 1;
    if (E < emin) E = emin;
    const int qexp = E - (p - 1);
    const double y = std::ldexp(std::nearbyint(std::ldexp(x, -qexp)), qexp);
    return std::fabs(y) > fmax ? std::copysign(INFINITY, x) : y;
}

}  // namespace

extern "C" {

int oracle_threads(void) { return omp_get_max_threads(); }

void oracle_round_storage(const double* x, int64_t n, int fmt, double* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = round_storage(x[i], fmt);
}

void oracle_widen(const void* x, int fmt, int64_t n, double* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = elem(x, fmt, i);
}

// ---------------------------------------------------------------------------
// S1: Walsh-Hadamard rotation.  H_d[i][j] = (-1)^popcount(i & j) / sqrt(d)
// (Sylvester, natural order, orthonormal and symmetric).
// ---------------------------------------------------------------------------
void oracle_hadamard_matrix(int d, double* h) {
    const double inv = 1.0 / std::sqrt((double)d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) h[(int64_t)i * d + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -inv : inv;
}

// y_r = H_d x_r = (sum_j (-1)^popcount(i & j) x_r[j]) / sqrt(d) for each row: the +-1 sums in
// double (exact for stored 16-bit values, so an exactly cancelling sum stays 0), then one
// division, then rounded once to store_fmt (F64: no rounding)
void oracle_hadamard(const double* x, int64_t n_rows, int d, int store_fmt, double* y) {
    const double sqrt_d = std::sqrt((double)d);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j)
                acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -x[r * d + j] : x[r * d + j];
            y[r * d + i] = round_storage(acc / sqrt_d, store_fmt);
        }
    }
}

// ---------------------------------------------------------------------------
// S3: keys visible to a query: every cached key in decode (the query's own key
// is already cached), j <= q_pos under the causal mask.
// ---------------------------------------------------------------------------
int64_t oracle_visible_count(int64_t n_kv, int causal, int64_t q_pos) {
    if (!causal) return n_kv;
    const int64_t lim = q_pos + 1;
    return lim < 0 ? 0 : (lim < n_kv ? lim : n_kv);
}

// ---------------------------------------------------------------------------
// S2: s[r, j] = sum_h w[r, h] * max(0, sum_c q[r, h, c] * k[key_off[r] + j, c])
// for j < n_vis[r]; dot products and the head sum in double, stored as f32
// with -0 made +0.  Int8 keys (k_fmt I8) are dequantized exactly: code * scale
// of their row.
//   q       [R, H, d] in q_fmt;  w  [R, H] double
//   k       cache rows of d elements, row i at element i * k_row_stride
//   out     row r at out + r * out_stride
// ---------------------------------------------------------------------------
void oracle_scores(int64_t R, int H, int d, const void* q, int q_fmt, const double* w, const void* k, int k_fmt,
                   int64_t k_row_stride, const float* k_scale, const int64_t* key_off, const int32_t* n_vis,
                   float* out, int64_t out_stride) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        // q of this row with the head index fastest, so that the per-head sums
        // below run side by side (each still summed over c in order)
        std::vector<double> qt((size_t)d * H), kk(d), acc(H);
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < d; ++c) qt[(size_t)c * H + h] = elem(q, q_fmt, (r * H + h) * (int64_t)d + c);
        for (int64_t j = 0; j < n_vis[r]; ++j) {
            const int64_t row = key_off[r] + j;
            const double sc = k_fmt == I8 ? (double)k_scale[row] : 1.0;
            for (int c = 0; c < d; ++c) kk[c] = elem(k, k_fmt, row * k_row_stride + c) * sc;
            std::fill(acc.begin(), acc.end(), 0.0);
            for (int c = 0; c < d; ++c)
                for (int h = 0; h < H; ++h) acc[h] += qt[(size_t)c * H + h] * kk[c];
            double s = 0.0;
            for (int h = 0; h < H; ++h) s += w[r * H + h] * (acc[h] > 0.0 ? acc[h] : 0.0);
            float f = (float)s;
            if (f == 0.0f) f = 0.0f;   // canonical +0
            out[r * out_stride + j] = f;
        }
    }
}

// ---------------------------------------------------------------------------
// S4: the min(top_k, n_vis) best visible keys: a stable sort of positions by
// score, descending (equal scores keep ascending position, so the lower
// position wins; -0 and +0 compare equal), the first K taken and returned in
// ascending position order; entries K .. top_k-1 are -1.
// Returns 0, or 1 if a score is not finite.
// ---------------------------------------------------------------------------
static int topk_row(const float* s, int64_t n, int64_t top_k, int32_t* idx, int32_t* n_sel) {
    for (int64_t j = 0; j < n; ++j)
        if (!std::isfinite(s[j])) return 1;
    std::vector<int32_t> order((size_t)n);
    for (int64_t j = 0; j < n; ++j) order[j] = (int32_t)j;
    std::stable_sort(order.begin(), order.end(), [s](int32_t a, int32_t b) { return s[a] > s[b]; });
    const int64_t K = std::min<int64_t>(top_k, n);
    std::sort(order.begin(), order.begin() + K);
    for (int64_t i = 0; i < top_k; ++i) idx[i] = i < K ? order[i] : -1;
    *n_sel = (int32_t)K;
    return 0;
}

int oracle_topk(int64_t R, const float* scores, int64_t score_stride, const int32_t* n_vis, int top_k, int32_t* idx,
                int64_t idx_stride, int32_t* n_sel) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r)
        bad |= topk_row(scores + r * score_stride, n_vis[r], top_k, idx + r * idx_stride, n_sel + r);
    return bad;
}

// ---------------------------------------------------------------------------
// S5: p[beta, c] = (1/C) sum_{t = beta*C}^{beta*C + C - 1} k[t, c] for the
// complete blocks beta < floor(n_kv / C), blocks cut from position 0; summed
// in double, stored as f32.
// ---------------------------------------------------------------------------
static void pool_block(const void* k, int fmt, int64_t stride, int C, int d, int64_t beta, float* dst) {
    for (int c = 0; c < d; ++c) {
        double sum = 0.0;
        for (int t = 0; t < C; ++t) sum += elem(k, fmt, (beta * C + t) * stride + c);
        dst[c] = (float)(sum / C);
    }
}

void oracle_block_pool(const void* k, int fmt, int64_t stride, int64_t n_kv, int C, int d, float* pooled) {
    const int64_t n_cb = n_kv / C;
#pragma omp parallel for schedule(static)
    for (int64_t beta = 0; beta < n_cb; ++beta) pool_block(k, fmt, stride, C, d, beta, pooled + beta * d);
}

// Persistent pooled keys after one maintenance step: rows beta0 .. n_cb-1 are
// pooled afresh, with beta0 = min(n_pooled, floor(stale_pos / C)) (a negative
// stale_pos: 0; has_stale 0: no edit) clamped to [0, n_cb]; every other row of
// prev is copied unchanged.  prev and out hold n_rows rows of d floats.
void oracle_block_pool_update(const float* prev, int64_t n_rows, const void* k, int fmt, int64_t stride,
                              int64_t n_kv, int C, int d, int64_t n_pooled, int has_stale, int64_t stale_pos,
                              float* out) {
    std::memcpy(out, prev, (size_t)n_rows * d * sizeof(float));
    const int64_t n_cb = n_kv / C;
    int64_t beta0 = n_pooled > 0 ? n_pooled : 0;
    if (has_stale) beta0 = std::min<int64_t>(beta0, stale_pos < 0 ? 0 : stale_pos / C);
    beta0 = std::min(beta0, n_cb);
    for (int64_t beta = beta0; beta < n_cb; ++beta) pool_block(k, fmt, stride, C, d, beta, out + beta * d);
}

// ---------------------------------------------------------------------------
// S6: block selection.  The best min(floor(top_k / C), n_cb) complete blocks
// (block score descending, lower block index first on ties), every token of
// them, then every tail token [n_cb*C, n_vis); ascending; padded with -1 to
// the capacity floor(top_k/C)*C + C - 1.  Returns 1 on a non-finite score.
// ---------------------------------------------------------------------------
static int64_t block_capacity(int top_k, int C) { return (int64_t)(top_k / C) * C + C - 1; }

int oracle_block_select(int64_t R, const float* bs, int64_t bs_stride, const int32_t* n_vis, int top_k, int C,
                        int32_t* idx, int64_t idx_stride, int32_t* n_sel) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r) {
        const float* s = bs + r * bs_stride;
        const int64_t n = n_vis[r], n_cb = n / C;
        int32_t* out = idx + r * idx_stride;
        bool finite = true;
        for (int64_t b = 0; b < n_cb; ++b) finite = finite && std::isfinite(s[b]);
        if (!finite) {
            bad |= 1;
            continue;
        }
        std::vector<int32_t> order((size_t)n_cb);
        for (int64_t b = 0; b < n_cb; ++b) order[b] = (int32_t)b;
        std::stable_sort(order.begin(), order.end(), [s](int32_t a, int32_t b) { return s[a] > s[b]; });
        const int64_t nb = std::min<int64_t>(top_k / C, n_cb);
        std::sort(order.begin(), order.begin() + nb);
        int64_t m = 0;
        for (int64_t i = 0; i < nb; ++i)
            for (int t = 0; t < C; ++t) out[m++] = order[i] * C + t;
        for (int64_t t = n_cb * C; t < n; ++t) out[m++] = (int32_t)t;
        n_sel[r] = (int32_t)m;
        for (int64_t i = m; i < block_capacity(top_k, C); ++i) out[i] = -1;
    }
    return bad;
}

// The same selection in the expansion form: every member of a complete block
// takes its block's score (a gather), the top floor(top_k/C)*C members are
// taken under the token rule (score descending, lower position first), and
// the tail is always kept.
int oracle_block_select_expanded(int64_t R, const float* bs, int64_t bs_stride, const int32_t* n_vis, int top_k,
                                 int C, int32_t* idx, int64_t idx_stride, int32_t* n_sel) {
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r) {
        const float* s = bs + r * bs_stride;
        const int64_t n = n_vis[r], n_cb = n / C, members = n_cb * C;
        const int64_t budget = (int64_t)(top_k / C) * C;
        std::vector<float> tok((size_t)members);
        for (int64_t t = 0; t < members; ++t) tok[t] = s[t / C];
        std::vector<int32_t> kept((size_t)std::max<int64_t>(budget, 1));
        int32_t nk = 0;
        if (topk_row(tok.data(), members, budget, kept.data(), &nk)) {
            bad |= 1;
            continue;
        }
        int32_t* out = idx + r * idx_stride;
        int64_t m = 0;
        for (int32_t i = 0; i < nk; ++i) out[m++] = kept[i];
        for (int64_t t = members; t < n; ++t) out[m++] = (int32_t)t;
        n_sel[r] = (int32_t)m;
        for (int64_t i = m; i < block_capacity(top_k, C); ++i) out[i] = -1;
    }
    return bad;
}

// ---------------------------------------------------------------------------
// S7 / S8: softmax attention of each query head over only the selected keys.
// For query head h of row r, kv head g = h / (Hq / Hkv):
//     l_s = scale * sum_c q[r, h, c] * K[row_s, g, c]
//     p_s = exp(l_s - max l) / sum exp(l - max l)
//     out[r, h, c] = sum_s p_s * V[row_s, g, c]
// with row_s = key_off[r] + idx[r, s] for s < n_sel[r].  V NULL is the MLA
// latent form: V = the first dv columns of the same K row.  Everything in
// double; a row with n_sel 0 gets 0.  Returns 1 if an index is negative.
// ---------------------------------------------------------------------------
int oracle_attention(int64_t R, int Hq, int Hkv, int dk, int dv, const void* q, int q_fmt, const void* K, int k_fmt,
                     int64_t k_row_stride, const void* V, int v_fmt, int64_t v_row_stride, const int64_t* key_off,
                     const int32_t* idx, int64_t idx_stride, const int32_t* n_sel, double scale, double* out) {
    const int G = Hq / Hkv;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r) {
        const int64_t S = n_sel[r];
        double* o = out + r * (int64_t)Hq * dv;
        std::fill(o, o + (int64_t)Hq * dv, 0.0);
        bool ok = true;
        for (int64_t s = 0; s < S; ++s) ok = ok && idx[r * idx_stride + s] >= 0;
        if (!ok) {
            bad |= 1;
            continue;
        }
        if (S == 0) continue;
        std::vector<double> ks((size_t)S * dk), vs((size_t)S * dv), qt((size_t)dk * G), l((size_t)G * S),
            acc(G);
        for (int g = 0; g < Hkv; ++g) {
            // the selected rows of kv head g, widened
            for (int64_t s = 0; s < S; ++s) {
                const int64_t row = key_off[r] + idx[r * idx_stride + s];
                for (int c = 0; c < dk; ++c) ks[s * dk + c] = elem(K, k_fmt, row * k_row_stride + (int64_t)g * dk + c);
                for (int c = 0; c < dv; ++c)
                    vs[s * dv + c] = V ? elem(V, v_fmt, row * v_row_stride + (int64_t)g * dv + c) : ks[s * dk + c];
            }
            // the query heads of this group, head index fastest
            for (int i = 0; i < G; ++i)
                for (int c = 0; c < dk; ++c)
                    qt[(size_t)c * G + i] = elem(q, q_fmt, (r * Hq + (int64_t)g * G + i) * dk + c);
            // logits: each head's sum over c in order, the heads side by side
            for (int64_t s = 0; s < S; ++s) {
                std::fill(acc.begin(), acc.end(), 0.0);
                for (int c = 0; c < dk; ++c)
                    for (int i = 0; i < G; ++i) acc[i] += qt[(size_t)c * G + i] * ks[s * dk + c];
                for (int i = 0; i < G; ++i) l[(size_t)i * S + s] = scale * acc[i];
            }
            for (int i = 0; i < G; ++i) {
                double* li = &l[(size_t)i * S];
                double m = li[0];
                for (int64_t s = 1; s < S; ++s) m = std::max(m, li[s]);
                double den = 0.0;
                for (int64_t s = 0; s < S; ++s) {
                    li[s] = std::exp(li[s] - m);
                    den += li[s];
                }
                double* oh = o + ((int64_t)g * G + i) * dv;
                for (int64_t s = 0; s < S; ++s) {
                    const double p = li[s] / den;
                    for (int c = 0; c < dv; ++c) oh[c] += p * vs[s * dv + c];
                }
            }
        }
    }
    return bad;
}

// ---------------------------------------------------------------------------
// Quantized indexer cache (storage format).  Per row, in f32 with round to
// nearest even: scale = max_c |x_c| / 127, code_c = clamp(rint(x_c / scale),
// -127, 127); an all-zero row has scale 0 and codes 0.
// ---------------------------------------------------------------------------
void oracle_quantize_rows(const void* x, int fmt, int64_t n, int d, int64_t stride, int8_t* q8, float* scale) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < d; ++c) amax = std::max(amax, std::fabs((float)elem(x, fmt, r * stride + c)));
        const float sc = amax / 127.0f;
        scale[r] = sc;
        for (int c = 0; c < d; ++c) {
            int8_t code = 0;
            if (sc > 0.0f) {
                const float ratio = (float)elem(x, fmt, r * stride + c) / sc;
                float v = std::nearbyint(ratio);
                v = v > 127.0f ? 127.0f : (v < -127.0f ? -127.0f : v);
                code = (int8_t)v;
            }
            q8[r * d + c] = code;
        }
    }
}

// the keys the quantized cache represents: scale[r] * code (exact in double)
void oracle_dequantize_rows(const int8_t* q8, const float* scale, int64_t n, int d, double* out) {
    for (int64_t r = 0; r < n; ++r)
        for (int c = 0; c < d; ++c) out[r * d + c] = (double)q8[r * d + c] * (double)scale[r];
}

}  // extern "C"
