"""Pins for the oracle's indexer scores, index top-k and sparse attention (DeepSeek V4.1 Compressed
sparse attention atlas page, "All 25 steps": Indexer, re-scored / Sparse attention; deepseek_v41_ref::attn
rustdoc page: sparse_attn; Join rows atlas page).

Scores: closed forms with one or two heads.  Top-k: a brute-force rank count, constructed ties and
signed zeros, and the selection invariants.  Attention: torch's scaled_dot_product_attention (a
library routine) with the sink as one extra key of value zero, and closed forms of the sink.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf(orc, a):
    return orc.f32_to_bf16(np.asarray(a, np.float32))


# ---------------------------------------------------------------------------- indexer scores

def test_scores_one_head_is_relu_dot(orc):
    rng = np.random.default_rng(10)
    q = _bf(orc, rng.standard_normal((3, 1, 16)))
    K = _bf(orc, rng.standard_normal((40, 16)))
    S = orc.index_scores(q, np.ones((3, 1), np.float32), K, np.full(3, 1000, np.int32), 1, 40)
    dots = orc.bf16_to_f32(q)[:, 0].astype(np.float64) @ orc.bf16_to_f32(K).astype(np.float64).T
    assert np.allclose(S, np.maximum(dots, 0.0), rtol=1e-6, atol=1e-6)
    assert (S[dots < 0] == 0).all()


def test_scores_head_weights_apply_after_relu(orc):
    rng = np.random.default_rng(11)
    q1 = rng.standard_normal((2, 1, 8)).astype(np.float32)
    q = _bf(orc, np.concatenate([q1, -q1], axis=1))  # head 1 = -head 0
    K = _bf(orc, rng.standard_normal((30, 8)))
    w = np.array([[2.0, 3.0], [-1.0, 0.5]], np.float32)
    S = orc.index_scores(q, w, K, np.full(2, 100, np.int32), 1, 30)
    d = orc.bf16_to_f32(q)[:, 0].astype(np.float64) @ orc.bf16_to_f32(K).astype(np.float64).T
    # ReLU(d) w0 + ReLU(-d) w1: each position gets exactly one head's weight
    want = np.where(d > 0, d * w[:, :1], -d * w[:, 1:])
    assert np.allclose(S, want, rtol=1e-6, atol=1e-6)


def test_scores_validity(orc):
    q = _bf(orc, np.ones((1, 1, 4)))
    K = _bf(orc, np.ones((20, 4)))
    # causal limit: j < floor((pos + 1) / ratio); pos 10, ratio 4 -> j < 2
    S = orc.index_scores(q, np.ones((1, 1), np.float32), K, np.array([10]), 4, 20)
    assert np.isfinite(S[0, :2]).all() and np.isneginf(S[0, 2:]).all()
    # published length caps it too
    S = orc.index_scores(q, np.ones((1, 1), np.float32), K, np.array([1000]), 1, 5)
    assert np.isfinite(S[0, :5]).all() and np.isneginf(S[0, 5:]).all()
    # candidate block mask: block b covers j in [4b, 4b + 4)
    cand = np.array([[1, 0, 1, 0, 0]], np.uint8)
    S = orc.index_scores(q, np.ones((1, 1), np.float32), K, np.array([1000]), 1, 20, cand, 4)
    fin = np.isfinite(S[0])
    assert list(np.nonzero(fin)[0]) == [0, 1, 2, 3, 8, 9, 10, 11]


def test_join_rows_geometry(orc):
    g = json.load(open(os.path.join(GOLD, "join_rows.json")))
    q = _bf(orc, np.ones((1, 1, 4)))
    K = _bf(orc, np.ones((600, 4)))
    S = orc.index_scores(q, np.ones((1, 1), np.float32), K, np.array([g["pos"]]), g["ratio"], 600)
    n_valid = int(np.isfinite(S).sum())
    assert n_valid == g["compressed_positions"]
    assert g["window"] + n_valid == g["rows"]


# ---------------------------------------------------------------------------- top-k

def _brute_topk_set(S, valid, K):
    """Position j is chosen iff fewer than K valid positions beat it (higher score, or the same
    score and a lower index)."""
    n = len(S)
    chosen = []
    for j in range(n):
        if not valid[j]:
            continue
        beat = sum(1 for i in range(n) if valid[i] and (S[i] > S[j] or (S[i] == S[j] and i < j)))
        if beat < K:
            chosen.append(j)
    return set(chosen)


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(orc, seed):
    rng = np.random.default_rng(100 + seed)
    Lc, K = 37, 8
    S = rng.integers(-3, 4, (5, Lc)).astype(np.float32) * 0.5  # many ties
    S[:, 3] = -0.0
    S[:, 4] = 0.0
    pos = np.array([20, 60, 147, 9, 3], np.int32)
    cand = rng.integers(0, 2, (5, 10)).astype(np.uint8)
    for c in (None, cand):
        out = orc.index_topk(S, K, pos, 4, 30, c, 4, offset=128)
        for t in range(5):
            valid = [j < (pos[t] + 1) // 4 and j < 30 and (c is None or c[t, j // 4]) for j in range(Lc)]
            want = _brute_topk_set(S[t], valid, K)
            got = [v - 128 for v in out[t] if v >= 0]
            assert set(got) == want and len(got) == len(want)
            assert list(out[t][len(got):]) == [-1] * (K - len(got))
            # selection order: score descending, index ascending
            keys = [(-S[t, j], j) for j in got]
            assert keys == sorted(keys)


def test_topk_ties_and_signed_zero(orc):
    S = np.zeros((1, 20), np.float32)
    S[0, ::2] = -0.0
    out = orc.index_topk(S, 5, np.array([100]), 1, 20)
    assert list(out[0]) == [0, 1, 2, 3, 4]
    # fewer valid than K: all of them, then -1
    out = orc.index_topk(S, 8, np.array([4]), 1, 20)
    assert list(out[0]) == [0, 1, 2, 3, 4, -1, -1, -1]


# ---------------------------------------------------------------------------- sparse attention

def _sdpa_with_sink(q, G, sink, scale):
    """torch SDPA over the rows G plus one extra key whose score is the sink and whose value is 0."""
    qt = torch.from_numpy(q.astype(np.float64))[:, None, :]           # [H, 1, d]
    n, d = G.shape
    k = torch.cat([torch.from_numpy(G.astype(np.float64)), torch.zeros(1, d, dtype=torch.float64)])
    v = k.clone()
    H = q.shape[0]
    mask = torch.zeros(H, 1, n + 1, dtype=torch.float64)
    mask[:, 0, n] = torch.from_numpy(sink.astype(np.float64))
    out = torch.nn.functional.scaled_dot_product_attention(qt, k[None].expand(H, -1, -1), v[None].expand(H, -1, -1),
                                                           attn_mask=mask, scale=scale)
    return out[:, 0].numpy()


@pytest.mark.parametrize("seed", range(3))
def test_sparse_attn_matches_sdpa_with_sink_key(orc, seed):
    rng = np.random.default_rng(200 + seed)
    H, hd, Na, Nb = 4, 32, 9, 13
    q = _bf(orc, rng.standard_normal((2, H, hd)) * 2)
    ra = _bf(orc, rng.standard_normal((Na, hd)))
    rb = _bf(orc, rng.standard_normal((Nb, hd)))
    sink = rng.standard_normal(H).astype(np.float32)
    idx = np.array([[0, -1, 3, 8, 9, 21, -1, 15], [-1, -1, 2, 2, 10, 11, 12, 20]], np.int32)
    scale = 1.0 / math.sqrt(hd)
    o = orc.bf16_to_f32(orc.sparse_attn(q, ra, rb, idx, sink, scale))
    Y = np.concatenate([orc.bf16_to_f32(ra), orc.bf16_to_f32(rb)])
    for t in range(2):
        G = Y[[i for i in idx[t] if i >= 0]]
        want = _sdpa_with_sink(orc.bf16_to_f32(q[t]), G, sink, scale)
        assert np.allclose(o[t], want, rtol=2 ** -7, atol=1e-6)


def test_sparse_attn_sink_closed_forms(orc):
    hd, H = 4, 2
    G = _bf(orc, [[1.0, 2.0, -3.0, 0.5]])
    q = np.zeros((1, H, hd), np.uint16)  # every score is 0
    # one row, score 0: A = 1 / (e^s + 1); sink ln 3 -> 1/4, sink -inf-like -> 1
    sink = np.array([math.log(3.0), -1e30], np.float32)
    o = orc.bf16_to_f32(orc.sparse_attn(q, G, None, np.array([[0]], np.int32), sink, 0.5))
    g = orc.bf16_to_f32(G[0])
    assert np.allclose(o[0, 0], g / 4, rtol=2 ** -8) and np.array_equal(o[0, 1], g)
    # n identical rows: O = g * n / (e^s + n)
    o = orc.bf16_to_f32(orc.sparse_attn(q, np.repeat(G, 5, 0), None, np.array([[0, 1, 2, 3, 4]], np.int32), sink, 0.5))
    assert np.allclose(o[0, 0], g * 5 / 8, rtol=2 ** -8)
    # nothing selected: O = 0
    o = orc.sparse_attn(q, G, None, np.array([[-1, -1]], np.int32), sink, 0.5)
    assert (o == 0).all()


def test_sparse_attn_scale_two_rows(orc):
    # hd = 4 -> scale 1/2; q = (2, 0, 0, 0): S_1 = 1 for G_1 = e_0, S_2 = 0 for G_2 = e_1; sink absent
    q = _bf(orc, [[[2.0, 0, 0, 0]]])
    G = _bf(orc, [[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    o = orc.bf16_to_f32(orc.sparse_attn(q, G, None, np.array([[0, 1]], np.int32), np.array([-1e30], np.float32), 0.5))
    e = math.e
    assert abs(o[0, 0, 0] - e / (e + 1)) < 2 ** -8 and abs(o[0, 0, 1] - 1 / (e + 1)) < 2 ** -8


def test_sparse_attn_rows_permutation_invariant(orc):
    rng = np.random.default_rng(7)
    q = _bf(orc, rng.standard_normal((1, 3, 16)))
    G = _bf(orc, rng.standard_normal((10, 16)))
    sink = rng.standard_normal(3).astype(np.float32)
    a = orc.sparse_attn(q, G, None, np.array([[0, 1, 2, 3, 4, 5]], np.int32), sink, 0.25)
    b = orc.sparse_attn(q, G, None, np.array([[5, 3, -1, 1, 0, 4, 2]], np.int32), sink, 0.25)
    assert np.allclose(orc.bf16_to_f32(a), orc.bf16_to_f32(b), rtol=2 ** -8, atol=1e-7)


def test_sparse_attn_rejects_bad_index(orc):
    q = np.zeros((1, 1, 4), np.uint16)
    G = np.zeros((2, 4), np.uint16)
    with pytest.raises(ValueError):
        orc.sparse_attn(q, G, None, np.array([[2]], np.int32), np.zeros(1, np.float32), 0.5)
