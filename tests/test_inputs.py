"""The seeded synthetic inputs follow their stated recipe: deterministic per seed, the stated
distributions and shapes, candidate masks that keep exactly the stated number of causal blocks and
nothing past the causal limit, and fp8 weight storage made of finite codes and tile scales in range.
"""
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from csa_inputs import (WORKLOADS, Geometry, activations, candidate_mask, fp8_weight, latent_cache,  # noqa: E402
                        positions, weights)


def _f(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_seeded_and_deterministic():
    g = Geometry(dim=256, n_heads=4, head_dim=64, rope_dim=16, q_rank=64, o_rank=32, groups=2, window=8,
                 index_heads=4, index_hd=32, index_topk=8, cand_block=4, max_seq=64, max_tokens=8, max_batch=2)
    a, b = weights(g), weights(g)
    assert a.keys() == b.keys() and all(np.array_equal(a[k], b[k]) for k in a)
    assert np.array_equal(activations(g, 2, 3), activations(g, 2, 3))
    # distinct tensors draw from distinct seeds
    assert not np.array_equal(a["wq_a"][:4, :4], a["wkv"][:4, :4])


def test_distributions_at_full_width():
    """x ~ N(0, 1); a projection [out, in] ~ N(0, 1/in); Z and K^I ~ N(0, 1); sink ~ N(0, 1) in f32;
    the norm weights are ones."""
    g = WORKLOADS["reindex_decode_r2"].geom
    w = weights(g)
    for name, fan_in in (("wq_a", g.dim), ("wq_b", g.q_rank), ("wo_b", g.groups * g.o_rank)):
        v = _f(w[name])
        assert v.shape[1] == fan_in
        assert abs(v.std() * math.sqrt(fan_in) - 1.0) < 0.02 and abs(v.mean()) * math.sqrt(fan_in) < 0.01
    assert w["sink"].dtype == np.float32 and w["sink"].shape == (g.n_heads,)
    assert (w["q_norm"] == 1).all() and (w["kv_norm"] == 1).all()
    x = _f(activations(g, 4, 1))
    assert x.shape == (4, 1, g.dim) and abs(x.std() - 1) < 0.03 and abs(x.mean()) < 0.03
    Z, KI = latent_cache(g, 2, 500)
    assert Z.shape == (2, 500, g.head_dim) and KI.shape == (2, 500, g.index_hd)
    assert abs(_f(Z).std() - 1) < 0.02 and abs(_f(KI).std() - 1) < 0.02


def test_candidate_masks_keep_exactly_the_stated_causal_blocks():
    for name in ("reindex_decode_r2", "longctx_decode_r4"):
        wl = WORKLOADS[name]
        g = wl.geom
        L = wl.compress_len
        width = -(-L // g.cand_block)
        pos = positions(wl.batch, wl.tokens, wl.start_pos)
        m = candidate_mask(wl.batch * wl.tokens, pos, wl.ratio, L, g.cand_block, width, wl.cand_keep, 1015)
        assert m.dtype == np.uint8 and m.shape == (wl.batch * wl.tokens, width)
        for r in range(m.shape[0]):
            limit = min((int(pos[r]) + 1) // wl.ratio, L)
            nb = -(-limit // g.cand_block)
            want = int(wl.cand_keep) if wl.cand_keep >= 1 else math.ceil(nb * wl.cand_keep)
            assert int(m[r].sum()) == min(want, nb)
            assert not m[r, nb:].any()
        # seeded: the same seed gives the same mask, another seed another one
        assert np.array_equal(m, candidate_mask(m.shape[0], pos, wl.ratio, L, g.cand_block, width, wl.cand_keep,
                                                1015))
        assert not np.array_equal(m, candidate_mask(m.shape[0], pos, wl.ratio, L, g.cand_block, width,
                                                    wl.cand_keep, 1016))


def test_fp8_weight_storage_in_range():
    codes, scales = fp8_weight((257, 129), 3)
    assert codes.dtype == np.uint8 and codes.shape == (257, 129)
    assert not ((codes == 0x7F) | (codes == 0xFF)).any()  # no NaN codes
    assert len(np.unique(codes)) > 200  # spread over the finite codes
    assert scales.dtype == np.float32 and scales.shape == (3, 2)
    e = np.log2(scales.astype(np.float64))
    assert (e >= -12).all() and (e < -4).all()
