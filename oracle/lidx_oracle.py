"""Plain float64 oracle of the lightning-indexer sparse-attention path.

TEST INFRASTRUCTURE ONLY (see the package docstring): only tests, the smoke
check and the bench's CPU-baseline leg may use it.

Sources (page title, then the part of the page):

* ik_llama.cpp PR #2058 (GLM-DSA lightning indexer), commit "Add
  GLM-5.2/DeepSeek-V3.2 DSA lightning indexer": indexer score
  ``relu(k . q_h)`` weighted per head by the indexer projection and summed over
  heads, plus the causal mask, then ``top_k(min(top_k, n_tokens))``; the
  Walsh-Hadamard rotation leaves ``(Hq).(Hk) = q.k`` unchanged.
* same PR, commit "decode-correct via persistent indexer-K cache": decode keys
  are written to the cache before scoring, so a decode query sees every cached
  key including its own; the rotated key is what the cache holds.
* ik_llama_opt commit log (src/llama.cpp), "openpangu: DSA lightning indexer +
  SWA schedule": ``score = sum_g w_g * relu(q_g . k)`` computed in f32, causal
  masked, exact top-k; below top_k visible keys the layer is exactly dense.
* same log, "Gather OpenPangu DSA decode reads" and "openpangu: MLA-latent KV
  cache": attention is a plain softmax over only the gathered rows; the MLA
  value is the first 512 columns of the same 576-wide latent row.
* llama.cpp commit c88c916636 (block-pooled indexer, QSA), commit message: one
  mean-pooled raw key per block of compress_ratio positions, a budget of whole
  blocks plus the incomplete tail, exactly dense below
  top_k + compress_ratio - 1 tokens, block scores expanded to members by a
  gather, blocks cut on the position line.

Readings where the pages leave a step open are stated beside each function.
"""

from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------

# (significand bits incl. the implicit one, minimum normal exponent, largest finite)
_FORMATS = {
    "f32": (24, -126, float(np.finfo(np.float32).max)),
    "f16": (11, -14, 65504.0),
    "bf16": (8, -126, float.fromhex("0x1.fep127")),
}


def round_to_storage(x, fmt: str) -> np.ndarray:
    """Round float64 values to ``fmt`` ("f32", "f16", "bf16"), nearest-even,
    directly from float64 (one rounding), and return them widened to float64.

    Needed where the method stores an intermediate in the cache dtype: the
    rotated indexer key is what the F16 cache holds (ik_llama.cpp PR #2058,
    commit "decode-correct via persistent indexer-K cache").  Overflow gives
    +-inf.  Written from the IEEE-754 definition: a value with exponent e
    (2**e <= |x| < 2**(e+1)) is rounded to a multiple of 2**(e - p + 1), and
    below the normal range to a multiple of 2**(emin - p + 1).
    """
    p, emin, fmax = _FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    ax = np.abs(x)
    nz = ax > 0
    # exponent of each value, clamped at the normal minimum (subnormal spacing)
    e = np.zeros_like(x)
    e[nz] = np.floor(np.log2(ax[nz]))
    # log2 can be off by one ulp near powers of two: fix e so 2**e <= |x| < 2**(e+1)
    lo = np.ldexp(1.0, e.astype(np.int64))
    e = np.where(nz & (lo > ax), e - 1, e)
    lo = np.ldexp(1.0, e.astype(np.int64))
    e = np.where(nz & (ax >= 2.0 * lo), e + 1, e)
    e = np.maximum(e, emin)
    quantum_exp = (e - (p - 1)).astype(np.int64)
    scaled = np.ldexp(x, -quantum_exp)            # exact: a power-of-two scale
    out = np.ldexp(np.rint(scaled), quantum_exp)  # np.rint rounds half to even
    out = np.where(np.abs(out) > fmax, np.copysign(np.inf, x), out)
    return out


# ---------------------------------------------------------------------------
# S1: Walsh-Hadamard rotation
# ---------------------------------------------------------------------------

def hadamard_matrix(d: int) -> np.ndarray:
    """Orthonormal Sylvester-Hadamard matrix of order ``d`` (a power of two),
    natural order: H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]], scaled by
    1/sqrt(d) so that H @ H = I (ik_llama.cpp PR #2058, commit "decode-correct
    via persistent indexer-K cache": orthonormal, symmetric, H*H = I; the
    K-shift commit of the same series builds it "with the identical Sylvester
    construction")."""
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / math.sqrt(d)


def hadamard_rotate(x, store: str | None = None) -> np.ndarray:
    """Rotate every length-d row (last axis) of ``x`` by H_d: y = H x.

    ``store`` names the storage dtype the rotated rows are written back in
    ("bf16", "f16", "f32"); the rotation is done in float64 -- the +-1 sums
    first, then one division by sqrt(d) -- and rounded once.
    Score invariance: (Hq).(Hk) = q.k because H is orthonormal (ik_llama.cpp
    PR #2058, commit "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer",
    simplifications list)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    signs = hadamard_matrix(d) * math.sqrt(d)      # the +-1 Sylvester matrix (entries exact)
    signs = np.round(signs)
    # H x = (S x) / sqrt(d): the +-1 sums of stored values are exact in double, so an exactly
    # cancelling sum stays exactly 0; then one division
    y = (x @ signs.T) / math.sqrt(d)
    if store is not None:
        y = round_to_storage(y, store)
    return y


# ---------------------------------------------------------------------------
# S3: visibility
# ---------------------------------------------------------------------------

def visible_count(n_kv: int, q_pos: int | None) -> int:
    """Number of keys a query row sees.

    Decode (``q_pos`` None): every cached key, the query's own key included,
    because the decode key is written to the cache before scoring (ik_llama.cpp
    PR #2058, commit "decode-correct via persistent indexer-K cache").
    Causal prefill: key j is visible iff j <= q_pos ("+ base causal mask",
    commit "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer").  Visibility is a
    bound, never -inf arithmetic (ik_llama_opt log, "openpangu: keep DSA
    zero-trick sources finite": 0 * -inf = NaN broke the mask)."""
    if q_pos is None:
        return int(n_kv)
    return int(max(0, min(int(q_pos) + 1, int(n_kv))))


# ---------------------------------------------------------------------------
# S2: indexer score
# ---------------------------------------------------------------------------

def indexer_scores(q, w, k) -> np.ndarray:
    """score_j = sum_h w_h * max(0, q_h . k_j) for every key row j.

    ``q`` [H, d], ``w`` [H], ``k`` [n, d]; all widened to float64 as stored.
    ReLU is applied to each head's dot product before the head sum
    (llama.cpp commit c88c916636, QSA commit message: "rectifies each head's dot
    product before summing over heads"; ik_llama_opt log, "openpangu: DSA
    lightning indexer + SWA schedule": score = sum_g w_g * relu(q_g . k)).
    Reading: ``w`` is one weight per (query row, head) -- the output of the
    indexer projection of that token -- and carries every scale; nothing else
    multiplies the score.

    Computed in float64, returned as float32 (the pages sum in f32), with -0
    made +0 so that the order key is unique.
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros(0, dtype=np.float32)
    dots = k @ q.T                        # [n, H]: q_h . k_j
    s = np.maximum(dots, 0.0) @ w         # sum_h w_h relu(.)
    s32 = s.astype(np.float32)
    s32[s32 == 0] = np.float32(0.0)       # canonical +0
    return s32


# ---------------------------------------------------------------------------
# S4: top-k selection
# ---------------------------------------------------------------------------

def topk_select(scores, n_vis: int, top_k: int) -> np.ndarray:
    """Positions of the min(top_k, n_vis) best visible keys, ascending.

    "ggml_top_k(min(top_k, n_tokens))" (ik_llama.cpp PR #2058, commit "Add
    GLM-5.2/DeepSeek-V3.2 DSA lightning indexer").  Order: score descending,
    and among equal scores the lower position first (the pages leave ties
    open; the lower position wins).  The result is returned sorted by
    position: only the set matters to the attention that follows ("Gather
    OpenPangu DSA decode reads" in the ik_llama_opt log gathers rows in any
    order and runs a plain softmax over them).
    """
    s = np.asarray(scores, dtype=np.float32)[:n_vis].astype(np.float64)
    if not np.all(np.isfinite(s)):
        raise ValueError("scores must be finite")
    kk = min(int(top_k), int(n_vis))
    if kk <= 0:
        return np.zeros(0, dtype=np.int64)
    pos = np.arange(n_vis)
    # stable ordering: primary key -score (ascending), secondary position
    order = np.lexsort((pos, -s))
    return np.sort(order[:kk]).astype(np.int64)


# ---------------------------------------------------------------------------
# S5 / S6: block-pooled indexer
# ---------------------------------------------------------------------------

def quantize_rows(x):
    """Per-row symmetric 8-bit codes of key rows, with an f32 scale per row.

    The storage format of a quantized indexer key cache ("GLM-DSA: allow for
    quantized indexer cache", ik_llama_opt commit log; like the q8_0 latent
    cache described there, it is "a storage format only" and the scores use
    the dequantized values).  Reading: one scale per key row,
        scale = max_c |x_c| / 127,   q_c = clamp(rint(x_c / scale), -127, 127)
    taken in float32 with round-to-nearest-even (the integer decisions are made
    in the precision the kernel makes them in); an all-zero row gets scale 0
    and codes 0.  Returns (int8 codes, float32 scales).
    """
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    q = np.zeros(x32.shape, dtype=np.int8)
    nz = scale > 0
    if np.any(nz):
        ratio = (x32[nz] / scale[nz][:, None]).astype(np.float32)
        q[nz] = np.clip(np.rint(ratio), -127, 127).astype(np.int8)
    return q, scale


def dequantize_rows(q8, scale) -> np.ndarray:
    """Key rows as the quantized cache represents them: scale_j * q8[j, c], in float64."""
    return np.asarray(q8, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[..., None]


def block_pool(k_raw, C: int, n_kv: int) -> np.ndarray:
    """Mean of the C raw keys of each complete block, stored as float32.

    Block beta covers positions [beta*C, (beta+1)*C) of the sequence: blocks
    are cuts of the position line measured from the sequence's first position
    (llama.cpp commit c88c916636, QSA commit message; llama-memory-hybrid-idx.h,
    kpool_layout comment: pools are fixed by the positions relative to the
    sequence's first one).  Only complete blocks are pooled; the remaining
    n_kv mod C tokens are the tail.  The pooled key is the mean of the raw
    keys, taken before any norm or rotation (the same commit message).
    """
    k_raw = np.asarray(k_raw, dtype=np.float64)
    n_cb = int(n_kv) // int(C)
    d = k_raw.shape[-1]
    if n_cb == 0:
        return np.zeros((0, d), dtype=np.float32)
    blocks = k_raw[: n_cb * C].reshape(n_cb, C, d)
    return blocks.mean(axis=1).astype(np.float32)


def block_pool_update(pooled_prev, k_raw, C: int, n_kv: int, n_pooled: int, stale_pos=None) -> np.ndarray:
    """Persistent pooled keys after one maintenance step.

    The pooled keys persist across batches, a batch only appends complete
    blocks, and an edit of the sequence from position p on regroups the blocks
    from the one holding p, so every pooled key at or after it is stale
    (llama-memory-hybrid-idx.h: "The pooled keys persist in the idx cache
    across batches", mem_idx_stale with POS_CLEAN, and get_n_kpool_new, the
    pools to re-pool this ubatch).  With n_cb = floor(n_kv / C) and
        beta0 = min(n_pooled, floor(stale_pos / C))   (a negative stale_pos: 0)
    clamped to [0, n_cb], blocks beta0 .. n_cb-1 take the block means of the
    current raw keys (block_pool) and every other row of pooled_prev is kept.
    stale_pos None means no edit.  Returns a new float32 array.
    """
    out = np.array(pooled_prev, dtype=np.float32, copy=True)
    n_cb = int(n_kv) // int(C)
    beta0 = max(int(n_pooled), 0)
    if stale_pos is not None:
        beta0 = min(beta0, 0 if stale_pos < 0 else int(stale_pos) // int(C))
    beta0 = min(beta0, n_cb)
    if n_cb > beta0:
        out[beta0:n_cb] = block_pool(k_raw, C, n_kv)[beta0:n_cb]
    return out


def block_select(block_scores, n_vis: int, top_k: int, C: int) -> np.ndarray:
    """Token positions kept by the block-pooled indexer, ascending.

    Keep the best min(floor(top_k / C), n_cb) complete blocks (score
    descending, lower block index first on ties) and every tail token
    [n_cb*C, n_vis) (llama.cpp commit c88c916636, QSA commit message: "keeps a
    budget of the best blocks, plus the tail of tokens that do not yet form a
    complete block").  Readings: the budget is floor(top_k / C) whole blocks;
    the tail is outside the budget.  With those, every block fits -- the result
    is dense -- exactly when n_vis <= top_k + C - 1 and C divides top_k.
    """
    n_cb = int(n_vis) // int(C)
    bs = np.asarray(block_scores, dtype=np.float32)[:n_cb].astype(np.float64)
    if not np.all(np.isfinite(bs)):
        raise ValueError("block scores must be finite")
    nb = min(int(top_k) // int(C), n_cb)
    order = np.lexsort((np.arange(n_cb), -bs))
    chosen = np.sort(order[:nb])
    toks = [np.arange(b * C, (b + 1) * C) for b in chosen]
    toks.append(np.arange(n_cb * C, int(n_vis)))
    return np.concatenate(toks).astype(np.int64)


def block_select_expanded(block_scores, n_vis: int, top_k: int, C: int) -> np.ndarray:
    """The same selection in the pages' expansion form.

    Every member of a complete block gets its block's score by a gather, the
    tail is always kept, and the top floor(top_k/C)*C of the block members
    are taken under the token tie rule (score descending, lower position
    first).  "Since the budget is a whole number of blocks and a block's
    members tie exactly, the cut still lands on a block boundary" (llama.cpp
    commit c88c916636, QSA commit message).  Tests assert that this equals
    :func:`block_select`.
    """
    n_cb = int(n_vis) // int(C)
    bs = np.asarray(block_scores, dtype=np.float32)[:n_cb]
    member_block = np.arange(n_cb * C) // C           # gather index
    tok_scores = bs[member_block]
    kept = topk_select(tok_scores, n_cb * C, (int(top_k) // int(C)) * int(C))
    tail = np.arange(n_cb * C, int(n_vis))
    return np.concatenate([kept, tail]).astype(np.int64)


# ---------------------------------------------------------------------------
# S7 / S8: softmax attention over a selected set
# ---------------------------------------------------------------------------

def attention_over(q, K, V, scale: float) -> np.ndarray:
    """Plain softmax attention of query heads over the given rows.

    ``q`` [G, dk], ``K`` [S, dk], ``V`` [S, dv] -> [G, dv] in float64:
    l = scale * q K^T, p = softmax(l) over the S rows, o = p V.  The max is
    subtracted before exp (it cancels exactly in the normalisation).  This is
    the "maskless softmax over ... selected rows" of "Gather OpenPangu DSA
    decode reads" (ik_llama_opt log).  S = 0 is not a valid input.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        raise ValueError("attention over an empty set")
    logits = scale * (q @ K.T)                     # [G, S]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    return p @ V


def sparse_attention_mla(q, latent, sel, scale: float, dv: int = 512) -> np.ndarray:
    """MLA attention of one query row over the selected latent rows.

    ``q`` [Hq, 576] (absorbed query), ``latent`` [n, 576] rows of the form
    [ckv 512 | roped k_pe 64], ``sel`` positions.  Logits use the whole 576-wide
    row; the value is its first ``dv`` = 512 columns (ik_llama_opt log,
    "openpangu: MLA-latent KV cache" and "Gather OpenPangu DSA decode reads":
    values derived from the gathered k rows).  Returns [Hq, dv] float64.
    """
    latent = np.asarray(latent, dtype=np.float64)
    rows = latent[np.asarray(sel, dtype=np.int64)]
    return attention_over(q, rows, rows[:, :dv], scale)


def sparse_attention_gqa(q, K, V, sel, scale: float) -> np.ndarray:
    """GQA/MQA attention of one query row over the selected positions.

    ``q`` [Hq, dk]; ``K`` [n, Hkv, dk]; ``V`` [n, Hkv, dv]; query head h reads
    kv head h // (Hq / Hkv) (the attention cells of llama-memory-hybrid-idx.h:
    "cell j is one token in both" caches).  Returns [Hq, dv] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, hkv = q.shape[0], K.shape[1]
    g = hq // hkv
    sel = np.asarray(sel, dtype=np.int64)
    out = np.zeros((hq, V.shape[2]))
    for j in range(hkv):
        out[j * g:(j + 1) * g] = attention_over(q[j * g:(j + 1) * g], K[sel, j], V[sel, j], scale)
    return out


def dense_attention_gqa(q, K, V, n_vis: int, scale: float) -> np.ndarray:
    """Attention over every visible key: the dense path the sparse one equals
    when top_k >= n_vis (ik_llama.cpp PR #2058: "indexer is an exact no-op
    when top_k>=n_tokens")."""
    return sparse_attention_gqa(q, K, V, np.arange(n_vis), scale)


def dense_attention_mla(q, latent, n_vis: int, scale: float, dv: int = 512) -> np.ndarray:
    """Dense MLA attention over every visible latent row."""
    return sparse_attention_mla(q, latent, np.arange(n_vis), scale, dv)


# ---------------------------------------------------------------------------
# the whole decode step for one query row
# ---------------------------------------------------------------------------

def decode_pipeline_mla(q_idx, w, k_cache, n_kv, top_k, q_attn, latent, scale, dv=512):
    """Score -> select -> sparse MLA attention for one decode query.

    Returns (scores f32 [n_kv], selected positions, output [Hq, dv] float64).
    """
    s = indexer_scores(q_idx, w, np.asarray(k_cache)[:n_kv])
    sel = topk_select(s, n_kv, top_k)
    out = sparse_attention_mla(q_attn, latent, sel, scale, dv)
    return s, sel, out
