"""Pins of the CPU oracles against what the pages and the mathematics fix.

Each test ties an oracle function to something other than its own code: a
hand-worked example (tests/golden), a closed form, a library routine that
computes the same thing by another method, brute-force enumeration on tiny
inputs, or an invariant the pages state.  Every pin runs against both
oracles -- the numpy one and the C++ one -- through the fixture ``O``; the last
tests also hold the two against each other.  All run on the CPU.
"""

import itertools
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import oracle.cpp


@pytest.fixture(params=["numpy", "cpp"])
def O(request):
    return oracle if request.param == "numpy" else oracle.cpp


def _lnfix(x):
    return [[math.log(3.0) if v == "ln3" else float(v) for v in row] for row in x]


# ---------------------------------------------------------------- rounding

def test_round_f16_matches_numpy_half(O):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 5, 20000),
                        [0.0, -0.0, 65504.0, 65519.0, 65520.0, 6.1e-5, 5.96e-8, 2.98e-8, 2.99e-8]])
    ours = O.round_to_storage(x, "f16")
    ref = x.astype(np.float16).astype(np.float64)       # numpy rounds double -> half directly
    np.testing.assert_array_equal(ours, ref)


def test_round_bf16_matches_torch_for_float32_values(O):
    # for values exact in float32, torch's float32 -> bfloat16 cast is a single RNE rounding
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(50000, generator=g) * torch.exp(torch.randn(50000, generator=g) * 8)).float()
    ref = x.to(torch.bfloat16).double().numpy()
    ours = O.round_to_storage(x.double().numpy(), "bf16")
    np.testing.assert_array_equal(ours, ref)


def test_round_ties_to_even_closed_form(O):
    # bf16 spacing at 1 is 2**-7: 1 + 2**-8 is a tie -> 1 (even); 1 + 3*2**-8 -> 1 + 2**-6
    assert O.round_to_storage([1 + 2 ** -8], "bf16")[0] == 1.0
    assert O.round_to_storage([1 + 3 * 2 ** -8], "bf16")[0] == 1 + 2 ** -6
    # f16 spacing at 1 is 2**-10
    assert O.round_to_storage([1 + 2 ** -11], "f16")[0] == 1.0
    assert O.round_to_storage([1 + 3 * 2 ** -11], "f16")[0] == 1 + 2 ** -9
    assert O.round_to_storage([1e6], "f16")[0] == math.inf


# ---------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("d", [1, 2, 8, 32, 128])
def test_hadamard_matrix_equals_scipy(O, d):
    np.testing.assert_allclose(O.hadamard_matrix(d), scipy.linalg.hadamard(d) / math.sqrt(d), rtol=0, atol=1e-15)


def test_hadamard_matrix_closed_form_entries(O):
    d = 128
    h = O.hadamard_matrix(d)
    i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
    sign = np.vectorize(lambda a: -1.0 if bin(a).count("1") % 2 else 1.0)(i & j)
    np.testing.assert_array_equal(h * math.sqrt(d), sign)


def test_hadamard_orthonormal_symmetric(O):
    h = O.hadamard_matrix(128)
    np.testing.assert_allclose(h @ h, np.eye(128), atol=1e-13)
    np.testing.assert_array_equal(h, h.T)


def _fwht(v):
    # butterfly fast Walsh-Hadamard transform (natural order), independent of the matrix build
    v = list(v)
    h = 1
    while h < len(v):
        for i in range(0, len(v), 2 * h):
            for j in range(i, i + h):
                a, b = v[j], v[j + h]
                v[j], v[j + h] = a + b, a - b
        h *= 2
    return np.array(v) / math.sqrt(len(v))


def test_hadamard_rotate_equals_butterfly_fwht(O):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128))
    y = O.hadamard_rotate(x)
    for r in range(5):
        np.testing.assert_allclose(y[r], _fwht(x[r]), atol=1e-12)
    # basis vector e_0 maps to the constant 1/sqrt(d)
    e0 = np.zeros(128); e0[0] = 1
    np.testing.assert_allclose(O.hadamard_rotate(e0), np.full(128, 1 / math.sqrt(128)), atol=1e-15)


def test_hadamard_round_trip_and_score_invariance(O):
    rng = np.random.default_rng(4)
    q = rng.standard_normal((8, 128)); k = rng.standard_normal((300, 128)); w = rng.standard_normal(8)
    np.testing.assert_allclose(O.hadamard_rotate(O.hadamard_rotate(q)), q, atol=1e-12)
    s0 = O.indexer_scores(q, w, k)
    s1 = O.indexer_scores(O.hadamard_rotate(q), w, O.hadamard_rotate(k))
    np.testing.assert_allclose(s1, s0, rtol=1e-6, atol=1e-6)


def test_hadamard_exact_cancellation_gives_zero(O):
    # H x = (S x) / sqrt(d) with S the +-1 Sylvester matrix: x = e_0 + e_1 gives (1 + (-1)^(i&1)) / sqrt(d),
    # exactly 0 at every odd i and exactly 2/sqrt(d) at every even i, also after rounding
    for d in (32, 64, 128):
        x = np.zeros(d); x[0] = x[1] = 1.0
        y = O.hadamard_rotate(x)
        assert np.all(y[1::2] == 0.0)
        np.testing.assert_allclose(y[0::2], 2 / math.sqrt(d), rtol=1e-15)
        assert np.all(O.hadamard_rotate(x, store="bf16")[1::2] == 0.0)


def test_hadamard_cancelling_bf16_row_worked_example(O, golden):
    g = golden["hadamard_cancel"]
    x = np.array(g["x"])
    assert np.all(O.round_to_storage(x, "bf16") == x)         # the inputs are stored bf16 values
    signs = np.array([(-1) ** bin(g["index"] & j).count("1") for j in range(g["d"])])
    assert float(np.sum(signs * x)) == 0.0                    # the signed sum cancels exactly
    y = O.hadamard_rotate(x[None])[0]
    assert y[g["index"]] == g["expected"]
    assert O.hadamard_rotate(x[None], store="bf16")[0][g["index"]] == g["expected"]


def test_hadamard_store_rounds_once(O):
    rng = np.random.default_rng(5)
    x = O.round_to_storage(rng.standard_normal((4, 128)), "bf16")
    y = O.hadamard_rotate(x, store="bf16")
    np.testing.assert_array_equal(y, O.round_to_storage(O.hadamard_rotate(x), "bf16"))


# ---------------------------------------------------------------- score

def test_score_worked_example(O, golden):
    g = golden["score"]
    s = O.indexer_scores(np.array(g["q"], float), np.array(g["w"]), np.array(g["k"], float))
    assert s.dtype == np.float32
    np.testing.assert_array_equal(s, np.array(g["expected"], np.float32))


def test_score_closed_form_unit_query(O):
    # one head, weight 1, q = e_c  ->  score_j = relu(k_jc)
    rng = np.random.default_rng(6)
    k = rng.standard_normal((50, 16))
    for c in (0, 7, 15):
        q = np.zeros((1, 16)); q[0, c] = 1.0
        np.testing.assert_array_equal(O.indexer_scores(q, [1.0], k), np.maximum(k[:, c], 0).astype(np.float32))


def test_score_relu_before_head_sum_and_homogeneity(O):
    rng = np.random.default_rng(7)
    q = rng.standard_normal((4, 8)); k = rng.standard_normal((40, 8)); w = rng.uniform(0.1, 1, 4)
    s = O.indexer_scores(q, w, k).astype(np.float64)
    # positive homogeneity: scaling one head's query by a > 0 scales only its term
    s2 = O.indexer_scores(q * np.array([[3.0], [1], [1], [1]]), w * np.array([1 / 3.0, 1, 1, 1]), k)
    np.testing.assert_allclose(s2, s, rtol=1e-6, atol=1e-6)
    # head permutation invariance
    p = [2, 0, 3, 1]
    np.testing.assert_allclose(O.indexer_scores(q[p], w[p], k), s, rtol=1e-6, atol=1e-6)
    # every dot negative -> score exactly 0 (relu per head), even with negative weights
    assert np.all(O.indexer_scores(-np.abs(q), -w, np.abs(k)) == 0)
    # linear in w
    np.testing.assert_allclose(O.indexer_scores(q, 2 * w, k), 2 * s, rtol=1e-6, atol=1e-6)
    # negative zero is canonicalised
    z = O.indexer_scores(np.ones((1, 2)), [-1.0], np.array([[-1.0, -1.0]]))
    assert np.signbit(z[0]) == False  # noqa: E712


# ---------------------------------------------------------------- top-k

def test_topk_worked_example(O, golden):
    g = golden["topk"]
    for c in g["cases"]:
        got = O.topk_select(np.array(g["scores"], np.float32), c["n_vis"], c["top_k"])
        assert got.tolist() == c["expected"], c


def _valid_topk_sets(s, k):
    """All size-k subsets S with: every i in S beats every j outside S, where i
    beats j iff s_i > s_j or (s_i == s_j and i < j)."""
    n = len(s)
    out = []
    for S in itertools.combinations(range(n), k):
        rest = [j for j in range(n) if j not in S]
        if all(s[i] > s[j] or (s[i] == s[j] and i < j) for i in S for j in rest):
            out.append(list(S))
    return out


def test_topk_brute_force_enumeration_with_ties(O):
    rng = np.random.default_rng(8)
    for trial in range(300):
        n = int(rng.integers(1, 10))
        s = rng.integers(-2, 3, n).astype(np.float32)      # many exact ties
        n_vis = int(rng.integers(1, n + 1))
        k = int(rng.integers(1, n + 2))
        kk = min(k, n_vis)
        sets = _valid_topk_sets(s[:n_vis].tolist(), kk)
        assert len(sets) == 1                               # the tie rule makes it unique
        assert O.topk_select(s, n_vis, k).tolist() == sets[0]


def test_topk_equals_python_stable_sort(O):
    rng = np.random.default_rng(9)
    for _ in range(20):
        n = int(rng.integers(1, 3000))
        s = np.round(rng.standard_normal(n), 1).astype(np.float32)
        k = int(rng.integers(1, 400))
        ref = sorted(sorted(range(n), key=lambda j: (-float(s[j]), j))[:k])
        assert O.topk_select(s, n, k).tolist() == ref


def test_topk_negative_zero_ties_with_zero(O):
    s = np.array([-0.0, 0.0, -0.0, 1.0], np.float32)
    assert O.topk_select(s, 4, 2).tolist() == [0, 3]


# ---------------------------------------------------------------- blocks

def test_block_pool_worked_example(O, golden):
    g = golden["block_pool"]
    got = O.block_pool(np.array(g["k_raw"], float), g["C"], len(g["k_raw"]))
    np.testing.assert_array_equal(got, np.array(g["expected"], np.float32))


def test_block_pool_closed_forms(O):
    # C = 1: pooled keys are the keys; a linear ramp pools to the block midpoint
    rng = np.random.default_rng(10)
    k = O.round_to_storage(rng.standard_normal((33, 4)), "f32")
    np.testing.assert_array_equal(O.block_pool(k, 1, 33), k.astype(np.float32))
    t = np.arange(64, dtype=float)[:, None] * np.ones((1, 3))
    np.testing.assert_array_equal(O.block_pool(t, 8, 64)[:, 0], (np.arange(8) * 8 + 3.5).astype(np.float32))
    assert O.block_pool(t, 8, 7).shape == (0, 3)


def test_block_select_worked_example(O, golden):
    g = golden["block_select"]
    for c in g["cases"]:
        got = O.block_select(np.array(c["block_scores"], np.float32), c["n_vis"], g["top_k"], g["C"])
        assert got.tolist() == c["expected"], c
        got2 = O.block_select_expanded(np.array(c["block_scores"], np.float32), c["n_vis"], g["top_k"], g["C"])
        assert got2.tolist() == c["expected"], c


def test_block_selection_equals_expansion_and_whole_blocks(O):
    rng = np.random.default_rng(11)
    for _ in range(400):
        C = int(rng.choice([1, 2, 3, 4, 8]))
        top_k = int(rng.integers(1, 40))
        n_vis = int(rng.integers(0, 80))
        n_cb = n_vis // C
        bs = rng.integers(-2, 3, n_cb).astype(np.float32)   # exact ties between blocks
        a = O.block_select(bs, n_vis, top_k, C)
        b = O.block_select_expanded(bs, n_vis, top_k, C)
        assert a.tolist() == b.tolist()
        # whole blocks + the complete tail
        body = a[a < n_cb * C]
        assert len(body) % C == 0
        for blk in set((body // C).tolist()):
            assert set(range(blk * C, blk * C + C)) <= set(body.tolist())
        assert set(range(n_cb * C, n_vis)) <= set(a.tolist())
        assert len(body) == min(top_k // C, n_cb) * C


def test_block_dense_threshold_both_sides(O):
    rng = np.random.default_rng(12)
    for C in (2, 4, 64):
        for top_k in (C, 4 * C, 32 * C):
            n = top_k + C - 1                     # dense: every token kept
            bs = rng.standard_normal(n // C).astype(np.float32)
            assert O.block_select(bs, n, top_k, C).tolist() == list(range(n))
            n = top_k + C                         # one block too many: not dense
            bs = rng.standard_normal(n // C).astype(np.float32)
            assert len(O.block_select(bs, n, top_k, C)) == top_k


def test_block_select_brute_force_blocks(O):
    rng = np.random.default_rng(13)
    for _ in range(200):
        C = int(rng.integers(1, 4)); n_vis = int(rng.integers(1, 16)); top_k = int(rng.integers(1, 12))
        n_cb = n_vis // C
        bs = rng.integers(0, 3, n_cb).astype(np.float32)
        nb = min(top_k // C, n_cb)
        sets = _valid_topk_sets(bs.tolist(), nb) if nb > 0 else [[]]
        assert len(sets) == 1
        expect = [t for b in sets[0] for t in range(b * C, b * C + C)] + list(range(n_cb * C, n_vis))
        assert O.block_select(bs, n_vis, top_k, C).tolist() == expect


# ---------------------------------------------------------------- attention

def test_attention_worked_examples(O, golden):
    g = golden["attention"]["gqa"]
    out = O.attention_over(np.array(g["q"], float), np.array(_lnfix(g["K"])), np.array(g["V"], float), g["scale"])
    np.testing.assert_allclose(out, g["expected"], rtol=1e-14)
    m = golden["attention"]["mla"]
    out = O.sparse_attention_mla(np.array(m["q"], float), np.array(_lnfix(m["latent"])), [0, 1], m["scale"], m["dv"])
    np.testing.assert_allclose(out, m["expected"], rtol=1e-14)


def test_dense_attention_equals_torch_sdpa_causal_gqa(O):
    # library routine: scaled_dot_product_attention in float64 with a causal mask
    g = torch.Generator().manual_seed(14)
    T, Hq, Hkv, dk, dv = 24, 8, 2, 16, 12
    q = torch.randn(T, Hq, dk, generator=g, dtype=torch.float64)
    K = torch.randn(T, Hkv, dk, generator=g, dtype=torch.float64)
    V = torch.randn(T, Hkv, dv, generator=g, dtype=torch.float64)
    scale = 1 / math.sqrt(dk)
    Kr = K.repeat_interleave(Hq // Hkv, dim=1)
    Vr = V.repeat_interleave(Hq // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), Kr.transpose(0, 1), Vr.transpose(0, 1), is_causal=True, scale=scale).transpose(0, 1)
    for t in range(T):
        out = O.dense_attention_gqa(q[t].numpy(), K.numpy(), V.numpy(), O.visible_count(T, t), scale)
        np.testing.assert_allclose(out, ref[t].numpy(), rtol=1e-12, atol=1e-12)


def test_attention_closed_forms(O):
    rng = np.random.default_rng(15)
    K = rng.standard_normal((10, 2, 8)); V = rng.standard_normal((10, 2, 5))
    q = rng.standard_normal((4, 8))
    # one selected key: the output is that key's value, for every head of the group
    out = O.sparse_attention_gqa(q, K, V, [6], 0.3)
    np.testing.assert_allclose(out[:2], np.tile(V[6, 0], (2, 1)), rtol=1e-14)
    np.testing.assert_allclose(out[2:], np.tile(V[6, 1], (2, 1)), rtol=1e-14)
    # zero query: uniform weights -> mean of the selected values
    out = O.sparse_attention_gqa(np.zeros((4, 8)), K, V, [1, 4, 9], 1.0)
    np.testing.assert_allclose(out[0], V[[1, 4, 9], 0].mean(0), rtol=1e-13)
    # MLA: value is the leading dv columns of the same rows
    lat = rng.standard_normal((12, 20))
    out = O.sparse_attention_mla(np.zeros((3, 20)), lat, [0, 5], 1.0, dv=16)
    np.testing.assert_allclose(out[1], lat[[0, 5], :16].mean(0), rtol=1e-13)


def test_sparse_equals_dense_when_topk_covers_visible(O):
    # exact no-op when top_k >= visible keys (ik_llama.cpp PR #2058 validation)
    rng = np.random.default_rng(16)
    n, H, d = 40, 4, 16
    q = rng.standard_normal((H, d)); w = rng.standard_normal(H); k = rng.standard_normal((n, d))
    qa = rng.standard_normal((8, 24)); lat = rng.standard_normal((n, 24))
    for n_vis in (1, 7, 40):
        s, sel, out = O.decode_pipeline_mla(q, w, k, n_vis, 64, qa, lat, 0.2, dv=16)
        assert sel.tolist() == list(range(n_vis))
        np.testing.assert_array_equal(out, O.dense_attention_mla(qa, lat, n_vis, 0.2, dv=16))


def test_visible_count(O):
    assert O.visible_count(100, None) == 100
    assert O.visible_count(100, 0) == 1
    assert O.visible_count(100, 99) == 100
    assert O.visible_count(100, 500) == 100
    assert O.visible_count(100, -1) == 0


def test_attention_large_logits_limit(O):
    # logits of order 1e4: softmax is the one-hot of the largest logit, so o = v of that key
    rng = np.random.default_rng(17)
    K = rng.standard_normal((6, 1, 4)); V = rng.standard_normal((6, 1, 3))
    q = rng.standard_normal((1, 4))
    out = O.sparse_attention_gqa(q, K, V, [0, 2, 3, 5], 1e4)
    best = [0, 2, 3, 5][int(np.argmax(K[[0, 2, 3, 5], 0] @ q[0]))]
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0], V[best, 0], rtol=1e-9, atol=1e-12)


def test_block_pool_update_worked_example(O, golden):
    g = golden["block_pool_update"]
    prev = np.zeros((4, 1), np.float32)
    prev[:2, 0] = g["pooled_before"]
    k = np.array(g["k_raw_after"], float)[:, None]
    got = O.block_pool_update(prev, k, g["C"], len(k), g["n_pooled"], g["stale_pos"])
    np.testing.assert_array_equal(got[:3, 0], np.array(g["expected"], np.float32))
    assert got[3, 0] == 0.0          # rows past the complete blocks are untouched


@pytest.mark.parametrize("n_prev,n_new,stale", [(0, 100, None), (64, 100, None), (64, 100, 37), (96, 130, 95),
                                                 (96, 96, 0), (40, 200, -1), (200, 200, None), (128, 131, 127)])
def test_block_pool_update_equals_full_pool_after_edits(O, n_prev, n_new, stale):
    # invariant: pool the old keys, edit positions >= stale, append to n_new, update
    # -> identical to pooling the new keys from scratch; rows before beta0 keep their bits
    rng = np.random.default_rng(n_prev * 1000 + n_new)
    C, d = 8, 5
    k_old = rng.standard_normal((max(n_prev, n_new), d))
    prev = np.full((40, d), 123.0, np.float32)
    nb_prev = n_prev // C
    prev[:nb_prev] = O.block_pool(k_old, C, n_prev)
    k_new = k_old.copy()
    if stale is not None:
        k_new[max(stale, 0):] = rng.standard_normal(k_new[max(stale, 0):].shape)
    got = O.block_pool_update(prev, k_new, C, n_new, nb_prev, stale)
    n_cb = n_new // C
    np.testing.assert_array_equal(got[:n_cb], O.block_pool(k_new, C, n_new))
    beta0 = min(nb_prev, n_cb if stale is None else (0 if stale < 0 else stale // C))
    np.testing.assert_array_equal(got[:beta0], prev[:beta0])
    assert np.all(got[n_cb:] == prev[n_cb:])


def test_block_pool_update_without_stale_marker_keeps_old_blocks(O):
    # an edit the caller does not report is not seen: blocks before n_pooled stay as they were
    C, d = 4, 3
    k = np.arange(48.0).reshape(16, d)
    prev = O.block_pool(k, C, 16)
    k2 = k.copy()
    k2[0] += 100.0
    got = O.block_pool_update(prev, k2, C, 16, 4, None)
    np.testing.assert_array_equal(got, prev)
    got = O.block_pool_update(prev, k2, C, 16, 4, 0)
    np.testing.assert_array_equal(got, O.block_pool(k2, C, 16))


def test_quantize_rows_worked_values(O):
    # amax 127 -> scale exactly 1, so the codes are rint(x) with ties to even
    x = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 126.6, -127.0, 0.49]])
    q, s = O.quantize_rows(x)
    assert s[0] == np.float32(1.0)
    np.testing.assert_array_equal(q[0], np.array([127, 2, 4, -2, 0, 127, -127, 0], np.int8))
    q, s = O.quantize_rows(np.zeros((2, 5)))
    assert np.all(s == 0) and np.all(q == 0)


def test_quantize_rows_invariants(O):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((200, 128)).astype(np.float32) * rng.uniform(1e-3, 50, (200, 1)).astype(np.float32)
    q, s = O.quantize_rows(x)
    assert q.dtype == np.int8 and np.all(np.abs(q.astype(int)) <= 127)
    assert np.all(np.abs(q).max(axis=1) == 127)                   # the largest entry maps to +-127
    err = np.abs(x.astype(np.float64) - O.dequantize_rows(q, s))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))


def test_scores_of_quantized_keys_within_the_dequantization_bound(O):
    # |relu(a) - relu(b)| <= |a - b| and |q_h . (k - k_hat)| <= ||q_h||_1 * scale / 2
    rng = np.random.default_rng(6)
    H, d, n = 8, 64, 50
    q = rng.standard_normal((H, d))
    w = rng.standard_normal(H)
    k = rng.standard_normal((n, d))
    k8, sc = O.quantize_rows(k)
    exact = O.indexer_scores(q, w, k).astype(np.float64)
    quant = O.indexer_scores(q, w, O.dequantize_rows(k8, sc)).astype(np.float64)
    bound = np.abs(w) @ np.abs(q).sum(axis=1) * sc.astype(np.float64) / 2
    assert np.all(np.abs(exact - quant) <= bound + 1e-5 * np.abs(exact) + 1e-6)
    assert np.max(np.abs(exact - quant)) > 0                       # the codes are not the keys


def test_dequantize_negative_scale_worked_example(O, golden):
    g = golden["quantized_keys"]
    k = O.dequantize_rows(np.array(g["codes"], np.int8), np.array(g["scale"], np.float32))
    np.testing.assert_array_equal(k, np.array(g["dequantized"]))
    s = O.indexer_scores(np.array(g["q"], float), np.array(g["w"]), k)
    np.testing.assert_array_equal(s, np.array(g["expected_scores"], np.float32))
    if hasattr(O, "scores_batch"):
        # the batch form reads the int8 codes and their scales as stored
        s8 = O.scores_batch(np.array(g["q"], float)[None], np.array(g["w"])[None], np.array(g["codes"], np.int8),
                            [0], [2], k_scale=np.array(g["scale"], np.float32))
        np.testing.assert_array_equal(s8[0], np.array(g["expected_scores"], np.float32))


# ---------------------------------------------------------------- the two oracles against each other

def _f32_ulp(x):
    return np.spacing(np.abs(np.asarray(x, np.float32))).astype(np.float64)


def test_oracles_agree_on_scores_and_selection():
    # independent implementations (numpy matmuls vs C++ loops): the same double values up to summation
    # order, so the f32 scores differ by at most one rounding step; on the same scores the selections,
    # both block forms and the pooled keys are identical
    rng = np.random.default_rng(20)
    cpp = oracle.cpp
    for n, H, d in ((1, 1, 1), (37, 4, 32), (700, 64, 128)):
        q = rng.standard_normal((H, d)); w = rng.standard_normal(H) / 8; k = rng.standard_normal((n, d))
        a, b = oracle.indexer_scores(q, w, k), cpp.indexer_scores(q, w, k)
        assert np.all(np.abs(a.astype(np.float64) - b) <= _f32_ulp(a))
        for top_k in (1, 5, 64, 2048):
            assert oracle.topk_select(a, n, top_k).tolist() == cpp.topk_select(a, n, top_k).tolist()
    for C in (1, 3, 64):
        kr = rng.standard_normal((300, 16))
        pa, pb = oracle.block_pool(kr, C, 300), cpp.block_pool(kr, C, 300)
        assert np.all(np.abs(pa.astype(np.float64) - pb) <= _f32_ulp(pa))
        bs = rng.integers(-3, 4, 300 // C).astype(np.float32)
        for n_vis in (0, C - 1, 150, 300):
            for top_k in (C, 7 * C, 2048):
                assert oracle.block_select(bs, n_vis, top_k, C).tolist() == cpp.block_select(bs, n_vis, top_k, C).tolist()
    x = rng.standard_normal((50, 128)).astype(np.float32) * 3
    qa, sa = oracle.quantize_rows(x)
    qb, sb = cpp.quantize_rows(x)
    np.testing.assert_array_equal(qa, qb)
    np.testing.assert_array_equal(sa, sb)


def test_oracles_agree_on_attention_and_hadamard():
    rng = np.random.default_rng(21)
    cpp = oracle.cpp
    q = rng.standard_normal((16, 40)); lat = rng.standard_normal((90, 40)); sel = rng.permutation(90)[:33]
    np.testing.assert_allclose(cpp.sparse_attention_mla(q, lat, sel, 0.3, dv=32),
                               oracle.sparse_attention_mla(q, lat, sel, 0.3, dv=32), rtol=1e-12, atol=1e-13)
    K = rng.standard_normal((50, 4, 24)); V = rng.standard_normal((50, 4, 20)); qg = rng.standard_normal((8, 24))
    np.testing.assert_allclose(cpp.sparse_attention_gqa(qg, K, V, sel[sel < 50], 0.2),
                               oracle.sparse_attention_gqa(qg, K, V, sel[sel < 50], 0.2), rtol=1e-12, atol=1e-13)
    x = rng.standard_normal((20, 128))
    np.testing.assert_allclose(cpp.hadamard_rotate(x), oracle.hadamard_rotate(x), rtol=0, atol=1e-13)


def test_cpp_batch_forms_read_storage_types_exactly():
    # the batch functions read f16 / bf16 / int8 caches as stored: the same as widening first
    rng = np.random.default_rng(22)
    cpp = oracle.cpp
    R, H, d, n = 3, 8, 32, 200
    q = torch.randn(R, H, d, dtype=torch.float64).to(torch.bfloat16)
    w = rng.standard_normal((R, H))
    k = torch.randn(n, d, dtype=torch.float64).to(torch.float16)
    n_vis = [200, 17, 0]
    s = cpp.scores_batch(q, w, k, [0, 5, 0], n_vis)
    for r in range(R):
        ref = cpp.indexer_scores(q[r].double().numpy(), w[r], k.double().numpy()[[0, 5, 0][r]:][:n_vis[r]])
        np.testing.assert_array_equal(s[r, :n_vis[r]], ref)
    k8, sc = cpp.quantize_rows(k.double().numpy())
    s8 = cpp.scores_batch(q, w, k8, [0, 0, 0], [200, 200, 200], k_scale=sc)
    np.testing.assert_array_equal(s8[1], cpp.indexer_scores(q[1].double().numpy(), w[1], cpp.dequantize_rows(k8, sc)))
    lat = torch.randn(n, 40, dtype=torch.float64).to(torch.bfloat16)
    idx = np.array([[3, 9, 150], [0, 1, -1]])
    qa = torch.randn(2, 4, 40, dtype=torch.float64).to(torch.bfloat16)
    out = cpp.attention_batch(qa, lat, None, [0, 10], idx, [3, 2], 0.25, 1, dv=32)
    np.testing.assert_array_equal(out[0], cpp.sparse_attention_mla(qa[0].double().numpy(), lat.double().numpy(),
                                                                   [3, 9, 150], 0.25, dv=32))
    np.testing.assert_array_equal(out[1], cpp.sparse_attention_mla(qa[1].double().numpy(), lat.double().numpy()[10:],
                                                                   [0, 1], 0.25, dv=32))
