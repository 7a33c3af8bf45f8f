"""GPU parity of the compressor (the kv-source role) against the oracle's orc_compress.

csa_compress runs over a prefill chunk and then decode steps that close further groups, at the
model's width (dim 5120, 512 features with a 64-feature rotary part, index keys of 128) for ratios 4,
2 and 1, and the results are compared with the oracle driven through the same calls:
  * compress_len, published after every call: exact;
  * the partial group (f32 kv and scores, -inf in empty slots): within f32 summation error;
  * the normed rows y and the index keys (bf16): within the bf16 output tolerance;
  * the latent rows (RoPE, then the fp8 round trip): within one e4m3 step, as the window rows,
    since their bf16 inputs may differ by the f32 products' summation order.
A kv source that is also an index source then runs as a whole layer (prefill and decode), with the
oracle composing its compressor and its attention the same way.
The pooling formula is a reading (the pages name the step but print none): this checks the kernels
against the oracle's reading, not against the real model.
"""
import math

import numpy as np
import pytest
import torch

from csa_inputs import (Geometry, activations, candidate_mask, compressor_weights, positions, ring_rows, weights)
from _helpers import assert_close_bf16, bf, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_attn_gb300 as m
    m.lib()
    return m


def _fp8_rows_close(got, want, what):
    g, w = bf(got).astype(np.float64), bf(want).astype(np.float64)
    rms = np.sqrt(np.mean(w * w, axis=-1, keepdims=True))
    step = 0.13 * np.maximum(np.abs(g), np.abs(w)) + 2.0 ** -7 * rms + 1e-6
    assert (np.abs(g - w) <= step).all(), "%s: %d elements beyond one e4m3 step" % (what, int((np.abs(g - w) > step).sum()))
    assert np.linalg.norm(g - w) <= 2e-2 * np.linalg.norm(w) + 1e-6, what


def _dev_w(w):
    return {k: to_dev(v) for k, v in w.items()}


def _kv_state(B, ratio, g, L):
    z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device="cuda")
    return dict(comp_kv=z(B, ratio, g.head_dim), comp_score=z(B, ratio, g.head_dim),
                latent=z(B, L, g.head_dim, dt=torch.bfloat16), index_keys=z(B, L, g.index_hd, dt=torch.bfloat16))


@pytest.mark.parametrize("ratio,T0,steps", [(4, 64, 5), (2, 33, 3), (1, 16, 2)])
def test_compress_matches_oracle(csa, orc, ratio, T0, steps):
    g = Geometry(max_seq=256, max_tokens=64, max_batch=2)
    gd = g.as_dict()
    B, L = 2, g.max_seq // ratio
    w = compressor_weights(g, ratio, seed_base=5000 + ratio)
    x = activations(g, B, T0 + steps, seed_base=5100 + ratio)
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor)
    ctx = csa.Context(gd)
    ring = torch.zeros(B, g.window, g.head_dim, dtype=torch.bfloat16, device="cuda")
    st = _kv_state(B, ratio, g, L)
    ctx.state_init(ring, B, kv_state=st)
    wd = _dev_w(w)
    role = dict(ratio=ratio, is_kv_source=1)
    sh = csa.Shared(None, None, 0, None, g.index_topk)
    y_d = torch.zeros(B, L, g.head_dim, dtype=torch.bfloat16, device="cuda")
    o_kv, o_sc = orc.compress_state(B, ratio, g.head_dim)
    o_Z = np.zeros((B, L, g.head_dim), np.uint16)
    o_KI = np.zeros((B, L, g.index_hd), np.uint16)
    o_Y = np.zeros((B, L, g.head_dim), np.uint16)
    o_w = dict(wkv=w["comp_wkv"], wgate=w.get("comp_wgate"), norm=w["comp_norm"], wk=w["idx_wk"], k_norm=w["idx_k_norm"])
    n = 0
    for start, T in [(0, T0)] + [(T0 + i, 1) for i in range(steps)]:
        xs = np.ascontiguousarray(x[:, start:start + T])
        ctx.compress(wd, role, ring, st, to_dev(xs), start, shared=sh, y_dbg=y_d)
        n = orc.compress(gd, ratio, o_w, o_kv, o_sc, xs, start, tab, o_Z, o_KI, n, o_Y)
        torch.cuda.synchronize()
        assert sh.compress_len == n == (start + T) // ratio
    assert ctx.status() == 0
    got_kv, got_sc = to_np(st["comp_kv"]), to_np(st["comp_score"])
    assert np.array_equal(np.isneginf(got_sc), np.isneginf(o_sc))
    fin = np.isfinite(o_sc)
    if ratio > 1:
        scale = np.abs(o_kv).max() + 1e-30
        assert np.abs(got_kv - o_kv).max() <= 1e-5 * scale
        if fin.any():
            assert np.abs(got_sc[fin] - o_sc[fin]).max() <= 1e-5 * (np.abs(o_sc[fin]).max() + 1e-30)
    assert_close_bf16(to_np(y_d)[:, :n], o_Y[:, :n], what="normed rows")
    assert_close_bf16(to_np(st["index_keys"])[:, :n], o_KI[:, :n], what="index keys")
    _fp8_rows_close(to_np(st["latent"])[:, :n], o_Z[:, :n], "latent rows")
    assert (to_np(st["latent"])[:, n:] == 0).all()  # no unfinished group is published
    ctx.close()


def test_kv_source_layer(csa, orc):
    """A ratio-4 layer that is kv source and index source: prefill of 48 tokens, then decode steps
    at 48..51 (the last closes group 12), on a small geometry; each call's output against the oracle's
    compressor followed by its layer forward over the published caches.  index_topk 16 takes every
    valid group, so the comparison does not hinge on near-equal index scores (the cut itself is
    tested with the indexer)."""
    g = Geometry(dim=256, n_heads=4, head_dim=64, rope_dim=16, q_rank=64, o_rank=32, groups=2, window=8,
                 index_heads=16, index_hd=128, index_topk=16, cand_block=4, max_seq=128, max_tokens=48, max_batch=2)
    gd = g.as_dict()
    B, ratio, L = 2, 4, 32
    w = weights(g, with_indexer=True, norm_ones=False)
    cw = compressor_weights(g, ratio, seed_base=5300)
    x = activations(g, B, 52, seed_base=5400)
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor)
    role = dict(ratio=ratio, is_kv_source=1, is_index_source=1)
    ctx = csa.Context(gd)
    wd = _dev_w(dict(w, **cw))
    ring_d = torch.zeros(B, g.window, g.head_dim, dtype=torch.bfloat16, device="cuda")
    st = _kv_state(B, ratio, g, L)
    ctx.state_init(ring_d, B, kv_state=st)
    o_kv, o_sc = orc.compress_state(B, ratio, g.head_dim)
    o_Z = np.zeros((B, L, g.head_dim), np.uint16)
    o_KI = np.zeros((B, L, g.index_hd), np.uint16)
    o_w = dict(wkv=cw["comp_wkv"], wgate=cw["comp_wgate"], norm=cw["comp_norm"], wk=cw["idx_wk"],
               k_norm=cw["idx_k_norm"])
    ring_o = np.zeros((B, g.window, g.head_dim), np.uint16)
    n = 0
    for start, T in ((0, 48), (48, 1), (49, 1), (50, 1), (51, 1)):
        xs = np.ascontiguousarray(x[:, start:start + T])
        NT = B * T
        sel_d = torch.full((NT, g.index_topk), -7, dtype=torch.int32, device="cuda")
        sh = csa.Shared(None, None, n, sel_d, g.index_topk)
        out = ctx.forward(wd, role, ring_d, to_dev(xs), start, shared=sh, kv_state=st)
        torch.cuda.synchronize()
        n = orc.compress(gd, ratio, o_w, o_kv, o_sc, xs, start, tab, o_Z, o_KI, n)
        assert sh.compress_len == n and sh.has_topk
        res = orc.attn_forward(gd, dict(ratio=ratio, is_index_source=1), w, ring_o, xs, start, tab,
                               dict(compress_kv=o_Z, index_k=o_KI, compress_len=n,
                                    topk_idxs=np.zeros((NT, g.index_topk), np.int32)), debug=False)
        assert_close_bf16(to_np(out), res["out"], what="kv-source layer out @%d" % start)
    assert ctx.status() == 0
    _fp8_rows_close(to_np(st["latent"])[:, :n], o_Z[:, :n], "latent rows")
    ctx.close()
