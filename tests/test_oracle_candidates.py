"""Pins of the oracle's candidate-source block mask, on the CPU.

The pages say the candidate-source layer publishes a block-level candidate mask ([queries][cand_width])
that later index sources apply, chosen by a top-k over blocks (candidate_block_size,
candidate_topk_blocks), but print no block score.  The reading: a block scores the largest valid
indexer score inside it.  Pinned here against a brute-force restatement in numpy (block maxima,
then a full sort with the lower block first on ties), on random scores, on exact ties and -0, with
fewer blocks than the count, and with the causal limit cutting a block; blocks without a valid
position are never marked.
"""
import numpy as np
import pytest


def _brute(S, pos, ratio, clen, cb, K, width):
    n, L = S.shape
    out = np.zeros((n, width), np.uint8)
    for t in range(n):
        limit = min((int(pos[t]) + 1) // ratio, clen)
        blocks = []
        for b in range(width):
            js = [j for j in range(b * cb, min((b + 1) * cb, limit))]
            if js:
                m = max(float(S[t, j]) for j in js)
                blocks.append((-(m + 0.0), b))  # -0 and +0 alike
        blocks.sort()
        for _, b in blocks[:K]:
            out[t, b] = 1
    return out


@pytest.mark.parametrize("n,L,clen,ratio,cb,K,start", [(6, 256, 256, 2, 8, 5, 300), (4, 512, 400, 4, 64, 3, 1700),
                                                        (3, 64, 64, 1, 8, 20, 40), (5, 128, 100, 2, 16, 2, 150)])
def test_candidate_blocks_brute_force(orc, n, L, clen, ratio, cb, K, start):
    rng = np.random.default_rng(n + L)
    S = rng.standard_normal((n, L)).astype(np.float32)
    S[:, ::5] = np.round(S[:, ::5])  # exact ties between blocks
    S[:, ::11] = -0.0
    pos = (start + np.arange(n)).astype(np.int32)
    width = -(-L // cb)
    got = orc.candidate_blocks(S, pos, ratio, clen, cb, K, width)
    assert np.array_equal(got, _brute(S, pos, ratio, clen, cb, K, width))


def test_candidate_blocks_invariants(orc):
    rng = np.random.default_rng(3)
    n, L, cb, K = 8, 200, 8, 6
    S = rng.standard_normal((n, L)).astype(np.float32)
    pos = np.array([3, 9, 15, 40, 80, 120, 300, 1000], np.int32)
    width = -(-L // cb)
    m = orc.candidate_blocks(S, pos, 2, L, cb, K, width)
    for t in range(n):
        limit = min((int(pos[t]) + 1) // 2, L)
        n_blocks = -(-limit // cb)
        assert m[t].sum() == min(K, n_blocks)
        assert (m[t, n_blocks:] == 0).all()  # no block past the causal limit
    # the block holding the row's best valid score is always a candidate
    for t in range(n):
        limit = min((int(pos[t]) + 1) // 2, L)
        if limit:
            assert m[t, int(np.argmax(S[t, :limit])) // cb] == 1
