"""GPU parity of the candidate source's block mask against the oracle.

Kernel level: csa_candidate_blocks on the oracle's f32 scores (ties, -0, causal limits cutting
blocks, fewer blocks than the count, the config's 8-position blocks and 2048 kept blocks) must equal
orc.candidate_blocks bit for bit.  Layer level: a ratio-2 index source that is also the candidate
source publishes a mask from its own scores; it must be a valid top-K of the oracle's block scores
(exact wherever the K-th and (K+1)-th block scores are further apart than the score tolerance), and
a later index source that applies it must match the oracle given the same mask.
"""
import numpy as np
import pytest
import torch

from csa_inputs import Geometry, activations, latent_cache, positions, ring_rows, weights
from _helpers import assert_close_bf16, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_attn_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("B,T,start,L,clen,ratio,cb,K", [
    (4, 1, 1000, 512, 500, 2, 64, 4),
    (2, 1, 65535, 16384, 16384, 4, 64, 64),
    (1, 1, 32767, 16384, 16384, 2, 8, 2048),      # the config's blocks of 8, 2048 kept
    (1, 40, 0, 64, 64, 1, 8, 3),                  # prefill: limits cut blocks, early rows have none
    (3, 1, 200, 128, 100, 2, 16, 20),             # fewer blocks than the count
])
def test_candidate_blocks_bit_exact(csa, orc, B, T, start, L, clen, ratio, cb, K):
    rng = np.random.default_rng(B * 7 + L)
    S = rng.standard_normal((B * T, L)).astype(np.float32)
    S[:, ::5] = np.round(S[:, ::5] * 2) / 2
    S[:, ::13] = -0.0
    pos = positions(B, T, start)
    width = -(-L // cb)
    want = orc.candidate_blocks(S, pos, ratio, clen, cb, K, width)
    mask = torch.full((B * T, width), 7, dtype=torch.uint8, device="cuda")
    csa.candidate_blocks(to_dev(S), B, T, start, clen, ratio, cb, K, mask)
    assert np.array_equal(to_np(mask), want)


def _block_scores(S_row, cb, width):
    out = np.full(width, -np.inf)
    for c in range(width):
        seg = S_row[c * cb:(c + 1) * cb]
        seg = seg[np.isfinite(seg)]
        if seg.size:
            out[c] = seg.max()
    return out


def test_candidate_source_then_index_source(csa, orc):
    g = Geometry(dim=128, n_heads=4, head_dim=64, rope_dim=16, q_rank=64, o_rank=32, groups=2, window=8,
                 index_heads=16, index_hd=128, index_topk=16, cand_block=8, cand_topk_blocks=5, max_seq=1024,
                 max_tokens=1, max_batch=4)
    gd = g.as_dict()
    B, T, start, L, clen = 4, 1, 700, 384, 300
    width = L // g.cand_block
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor)
    Z, KI = latent_cache(g, B, L, seed_base=3300)
    ring0 = orc.act_quant(ring_rows(g, B))[0]
    pos = positions(B, T, start)
    ctx = csa.Context(gd)
    K = g.index_topk
    # layer 1: index source and candidate source
    w1 = weights(g, with_indexer=True, norm_ones=False, seed_base=1200)
    x1 = activations(g, B, T, seed_base=2300)
    role1 = dict(ratio=2, is_index_source=1, is_candidate_source=1)
    mask_d = torch.full((B * T, width), 9, dtype=torch.uint8, device="cuda")
    sel_d = torch.full((B * T, K), -7, dtype=torch.int32, device="cuda")
    sh = csa.Shared(to_dev(Z), to_dev(KI), clen, sel_d, K, mask_d)
    dbg = dict(scores=torch.full((B * T, L), float("nan"), device="cuda"))
    ctx.forward({k: to_dev(v) for k, v in w1.items()}, role1, to_dev(ring0), to_dev(x1), start, shared=sh, debug=dbg)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    got_mask = to_np(mask_d)
    # the mask is the GPU's own scores' block top-K, bit for bit
    S_gpu = to_np(dbg["scores"]).astype(np.float32)
    S_gpu = np.where(np.isnan(S_gpu), -np.inf, S_gpu).astype(np.float32)
    assert np.array_equal(got_mask, orc.candidate_blocks(S_gpu, pos, 2, clen, g.cand_block, g.cand_topk_blocks, width))
    # and a valid block top-K of the oracle's scores
    res1 = orc.attn_forward(gd, role1, w1, ring0.copy(), x1, start, tab,
                            dict(compress_kv=Z, index_k=KI, compress_len=clen, topk_idxs=np.zeros((B * T, K), np.int32)))
    for r in range(B * T):
        bs = _block_scores(res1["scores"][r], g.cand_block, width)
        valid = np.isfinite(bs)
        tol = 2e-2 * np.abs(bs[valid]).max()
        chosen = np.nonzero(got_mask[r])[0]
        assert len(chosen) == min(g.cand_topk_blocks, int(valid.sum())) and valid[chosen].all()
        order = sorted(np.nonzero(valid)[0], key=lambda c: (-bs[c], c))
        if len(order) > g.cand_topk_blocks:
            kth = bs[order[g.cand_topk_blocks - 1]]
            if kth - bs[order[g.cand_topk_blocks]] > tol:
                assert set(chosen) == set(order[:g.cand_topk_blocks])
            else:
                assert bs[chosen].min() >= kth - tol
    # layer 2: an index source that applies the published mask
    w2 = weights(g, with_indexer=True, norm_ones=False, seed_base=1300)
    x2 = activations(g, B, T, seed_base=2400)
    role2 = dict(ratio=2, is_index_source=1, uses_candidates=1)
    out2 = ctx.forward({k: to_dev(v) for k, v in w2.items()}, role2, to_dev(ring0), to_dev(x2), start, shared=sh)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    for b in range(B):
        res2 = orc.attn_forward(gd, role2, w2, ring0[b:b + 1].copy(), x2[b:b + 1], start, tab,
                                dict(compress_kv=Z[b:b + 1], index_k=KI[b:b + 1], compress_len=clen,
                                     topk_idxs=np.zeros((T, K), np.int32), candidates=got_mask[b * T:(b + 1) * T]),
                                debug=False)
        assert_close_bf16(to_np(out2)[b], res2["out"][0], what="index source under the published mask")
    ctx.close()
