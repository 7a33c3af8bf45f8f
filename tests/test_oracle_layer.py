"""Pins for the oracle's layer forward (DeepSeek V4.1 Compressed sparse attention atlas page:
Attention.forward excerpt, "All 25 steps", the parameter table; metrale_model_arch::attn_v41 docs:
roles, shared selection, refusals).

The projections are checked against torch matmuls and torch's rms_norm in float64 (library
routines), the grouped output against a dense product with the block-diagonal expansion of wo_a,
the parameter accounting against the page's table, the Reindex reuse against the index source.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from csa_inputs import WORKLOADS, Geometry, activations, candidate_mask, latent_cache, positions, weights

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _f64(orc, u16):
    return torch.from_numpy(orc.bf16_to_f32(u16).astype(np.float64))


def _bf16(x):
    return x.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_param_counts_full_width(orc):
    g = json.load(open(os.path.join(GOLD, "param_counts.json")))
    c = orc.param_counts(g["geometry"], with_indexer=True)
    comp = g["components"]
    assert c[:6] == [comp["query_compression"], comp["query_heads"], comp["window_keys_and_values"],
                     comp["indexer_rescored"], comp["sparse_attention"], comp["grouped_output"]]
    assert c[6] == g["per_instance_total"]
    assert c[6] * g["groups_of_layers"] == g["total_over_groups"]
    # the shapes the synthetic weights take are the ones counted
    w = weights(Geometry(dim=64, n_heads=4, head_dim=32, rope_dim=8, q_rank=16, o_rank=8, groups=2, window=4,
                         index_heads=2, index_hd=8), with_indexer=True)
    small = dict(dim=64, n_heads=4, head_dim=32, rope_dim=8, q_rank=16, o_rank=8, groups=2, window=4, eps=1e-6,
                 index_heads=2, index_hd=8, index_topk=4, cand_block=2)
    c = orc.param_counts(small, True)
    assert c[6] == sum(v.size for v in w.values())


def _tiny_setup(orc, ratio=2, index_source=True, cand=True, B=2, T=6, start_pos=0, L=16, seed=1000):
    geom = Geometry(dim=96, n_heads=4, head_dim=64, rope_dim=16, q_rank=48, o_rank=24, groups=2, window=8,
                    index_heads=4, index_hd=32, index_topk=8, cand_block=4, max_seq=256)
    g = geom.as_dict()
    w = weights(geom, with_indexer=True, seed_base=seed, norm_ones=False)
    x = activations(geom, B, T, seed_base=seed)
    Z, KI = latent_cache(geom, B, L, seed_base=seed)
    tab = orc.rope_table(g["rope_dim"], g["max_seq"], g["compress_rope_theta"] if ratio else g["rope_theta"])
    pos = positions(B, T, start_pos)
    shared = dict(compress_kv=Z, index_k=KI, compress_len=L, topk_idxs=np.full((B * T, 8), -7, np.int32))
    if cand:
        shared["candidates"] = candidate_mask(B * T, pos, ratio, L, 4, -(-L // 4), 0.5, seed + 15)
    role = dict(ratio=ratio, is_index_source=index_source, uses_candidates=cand)
    return geom, g, w, x, tab, shared, role


def test_projection_paths_match_torch(orc):
    geom, g, w, x, tab, shared, role = _tiny_setup(orc)
    ring = np.zeros((2, 8, 64), np.uint16)
    r = orc.attn_forward(g, role, w, ring, x, 0, tab, shared)
    X = _f64(orc, x.reshape(12, 96))
    # qr = RMSNorm(x wq_a^T) * q_norm, each stage rounded to bf16
    qa = _bf16(X @ _f64(orc, w["wq_a"]).T)
    qr = _bf16(torch.nn.functional.rms_norm(_f64(orc, qa), (48,), torch.from_numpy(w["q_norm"].astype(np.float64)),
                                            eps=g["eps"]))
    assert np.array_equal(r["qr"], qr)
    # q before RoPE = qr wq_b^T; the rope part is rotated, the rest is the plain product
    qb = _bf16(_f64(orc, qr) @ _f64(orc, w["wq_b"]).T).reshape(12, 4, 64)
    assert np.array_equal(r["q"][..., :48], qb[..., :48])
    # indexer query and head weights: q^I = qr W_IQ^T, w^I = (x W_IW^T) / sqrt(dI * Hi)
    assert np.array_equal(r["qI"], _bf16(_f64(orc, qr) @ _f64(orc, w["idx_wq_b"]).T))
    wraw = orc.bf16_to_f32(_bf16(X @ _f64(orc, w["idx_wproj"]).T)).astype(np.float64)
    assert np.allclose(r["wI"], wraw / math.sqrt(32 * 4), rtol=1e-7)
    # the kv row: RMSNorm(x wkv^T) * kv_norm, rope tail rotated, then the fp8 round trip; its
    # untouched head (before the tail) equals act_quant of the plain product
    ka = _bf16(X @ _f64(orc, w["wkv"]).T)
    kn = _bf16(torch.nn.functional.rms_norm(_f64(orc, ka), (64,), torch.from_numpy(w["kv_norm"].astype(np.float64)),
                                            eps=g["eps"]))
    krot = orc.apply_rotary(kn, 16, positions(2, 6, 0), tab)
    kq, codes, se = orc.act_quant(krot)
    assert np.array_equal(r["kv"], kq) and np.array_equal(r["kv_codes"], codes) and np.array_equal(r["kv_scale"], se)


def test_grouped_output_is_block_diagonal_dense(orc):
    geom, g, w, x, tab, shared, role = _tiny_setup(orc)
    ring = np.zeros((2, 8, 64), np.uint16)
    r = orc.attn_forward(g, role, w, ring, x, 0, tab, shared)
    ob = orc.apply_rotary(r["o"].reshape(12 * 4, 64), 16, positions(2, 6, 0), tab, inverse=True, rows_per_pos=4)
    O = _f64(orc, ob.reshape(12, 256))
    woa = _f64(orc, w["wo_a"])  # [G*o_rank, gw] = [48, 128]
    bd = torch.zeros(48, 256, dtype=torch.float64)
    bd[:24, :128] = woa[:24]
    bd[24:, 128:] = woa[24:]
    og = _bf16(O @ bd.T)
    assert np.array_equal(r["og"], og)
    out = _bf16(_f64(orc, og) @ _f64(orc, w["wo_b"]).T)
    assert np.array_equal(r["out"].reshape(12, 96), out)


def test_attention_inputs_joined(orc):
    """sparse_attn over [chunk rows; Z] with J = [window; I + T] equals the layer's o."""
    geom, g, w, x, tab, shared, role = _tiny_setup(orc)
    ring = np.zeros((2, 8, 64), np.uint16)
    r = orc.attn_forward(g, role, w, ring, x, 0, tab, shared)
    for b in range(2):
        rows_a = r["kv"][b * 6:(b + 1) * 6]
        idx = r["idx"][b * 6:(b + 1) * 6]
        assert (idx[:, 8:][idx[:, 8:] >= 0] >= 6).all()  # compressed entries offset by |W| = T
        o = orc.sparse_attn(r["q"][b * 6:(b + 1) * 6], rows_a, shared["compress_kv"][b], idx, w["sink"],
                            1 / math.sqrt(64))
        assert np.array_equal(o, r["o"][b * 6:(b + 1) * 6])
    # the published selection is the layer's compressed columns
    assert np.array_equal(shared["topk_idxs"], r["idx"][:, 8:])


def test_reindex_reuse_matches_index_source(orc):
    geom, g, w, x, tab, shared, role = _tiny_setup(orc, start_pos=0)
    ring = np.zeros((2, 8, 64), np.uint16)
    src = orc.attn_forward(g, role, w, ring.copy(), x, 0, tab, shared)
    reuse_role = dict(ratio=2, is_index_source=False, uses_candidates=False)
    w2 = dict(w)
    w2.pop("idx_wq_b")
    w2.pop("idx_wproj")
    re = orc.attn_forward(g, reuse_role, w2, ring.copy(), x, 0, tab, shared)
    assert np.array_equal(re["idx"], src["idx"]) and np.array_equal(re["out"], src["out"])


def test_decode_ratio2_selection(orc):
    B, L = 2, 16
    geom, g, w, x, tab, shared, role = _tiny_setup(orc, B=B, T=1, start_pos=29, L=L)
    ring = orc.act_quant(np.ascontiguousarray(np.random.default_rng(3).integers(0, 2 ** 14, (B, 8, 64)).astype(np.uint16)))[0]
    r = orc.attn_forward(g, role, w, ring, x, 29, tab, shared)
    # decode window: the ring oldest first; compressed: j < min(floor(30/2), L) = 15 under the mask
    assert list(r["idx"][0, :8]) == [(30 + k) % 8 for k in range(8)]
    for b in range(B):
        sel = [v - 8 for v in r["idx"][b, 8:] if v >= 0]
        allowed = [j for j in range(15) if shared["candidates"][b, j // 4]]
        assert set(sel) <= set(allowed) and len(sel) == min(8, len(allowed))


def test_refusals(orc):
    geom, g, w, x, tab, shared, role = _tiny_setup(orc)
    ring = np.zeros((2, 8, 64), np.uint16)
    with pytest.raises(ValueError):  # ratio > 0 without a published latent cache
        orc.attn_forward(g, role, w, ring, x, 0, tab, dict(shared, compress_kv=None))
    with pytest.raises(ValueError):  # decode takes one query per sequence
        orc.attn_forward(g, role, w, ring, x, 5, tab, shared)
    with pytest.raises(ValueError):  # reuse layer without a published selection
        orc.attn_forward(g, dict(ratio=2, is_index_source=False), w, ring, x, 0, tab, dict(shared, topk_idxs=None))


def test_tok_mask_gives_same_rows(orc):
    geom, g, w, x, tab, shared, role = _tiny_setup(orc, T=10)
    full = orc.attn_forward(g, role, w, np.zeros((2, 8, 64), np.uint16), x, 0, tab, dict(shared, topk_idxs=np.zeros((20, 8), np.int32)))
    mask = np.zeros(20, np.uint8)
    mask[[3, 9, 14]] = 1
    ring = np.zeros((2, 8, 64), np.uint16)
    part = orc.attn_forward(g, role, w, ring, x, 0, tab, dict(shared, topk_idxs=np.zeros((20, 8), np.int32)),
                            tok_mask=mask)
    for r in (3, 9, 14):
        assert np.array_equal(part["out"].reshape(20, -1)[r], full["out"].reshape(20, -1)[r])
    ring_full = np.zeros((2, 8, 64), np.uint16)
    orc.attn_forward(g, role, w, ring_full, x, 0, tab, dict(shared, topk_idxs=np.zeros((20, 8), np.int32)))
    assert np.array_equal(ring, ring_full)
