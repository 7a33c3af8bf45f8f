"""Pins of the oracle's compressor (the kv-source role), on the CPU.

The pages give the compressor's weights and state -- f32 kv and gate [hd, dim] at ratio > 1, bf16 kv
at ratio 1; a partial group of f32 kv and score [ratio, hd] whose scores start at -inf; the latent and
index-key caches; compress_len, the number of groups written, which only grows -- but not its pooling
formula, so the oracle's agreement with the real model is unpinned.  What the pages and mathematics
do fix is checked here, each check chosen so that a plausible slip fails it:
  * the products are x Wkv^T and x Wgate^T rounded once to f32 (numpy in float64);
  * equal scores pool to the mean of the group's rows, one dominant score selects its row, and two
    rows pool to the closed-form softmax mixture (an off-by-one in the slot, a dropped exponential or
    a sum over the wrong axis fails one of them);
  * the normed row, the index key and the latent row are the pinned primitives composed in order
    (RMSNorm; linear_bf16 then RMSNorm; RoPE at the group's first position then the fp8 round trip);
  * compress_len counts complete groups only, an unfinished group publishes nothing and leaves -inf
    scores in its unwritten slots;
  * splitting a sequence into a prefill and decode steps (or any chunks) gives the very same rows.
"""
import math

import numpy as np
import pytest
import torch

from csa_inputs import Geometry


def _geom():
    return Geometry(dim=64, n_heads=4, head_dim=64, rope_dim=16, q_rank=32, o_rank=32, groups=2, window=8,
                    index_heads=4, index_hd=32, max_seq=256)


def _weights(orc, g, ratio, seed=0, gate_scale=1.0):
    rng = np.random.default_rng(seed)
    hd, dim = g.head_dim, g.dim
    w = dict(norm=(1 + 0.1 * rng.standard_normal(hd)).astype(np.float32),
             wk=orc.f32_to_bf16((rng.standard_normal((g.index_hd, hd)) / math.sqrt(hd)).astype(np.float32)),
             k_norm=(1 + 0.1 * rng.standard_normal(g.index_hd)).astype(np.float32))
    if ratio > 1:
        w["wkv"] = (rng.standard_normal((hd, dim)) / math.sqrt(dim)).astype(np.float32)
        w["wgate"] = (gate_scale * rng.standard_normal((hd, dim)) / math.sqrt(dim)).astype(np.float32)
    else:
        w["wkv"] = orc.f32_to_bf16((rng.standard_normal((hd, dim)) / math.sqrt(dim)).astype(np.float32))
    return w


def _x(orc, B, T, dim, seed=1):
    return orc.f32_to_bf16(np.random.default_rng(seed).standard_normal((B, T, dim)).astype(np.float32))


def _run(orc, g, ratio, w, x, chunks):
    """The compressor over x in the given chunks [(start, T), ...] from an empty state."""
    B = x.shape[0]
    gd = g.as_dict()
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta)
    kv, sc = orc.compress_state(B, ratio, g.head_dim)
    L = g.max_seq // ratio
    Z = np.full((B, L, g.head_dim), 0x7fc1, np.uint16)  # sentinel: rows never written stay NaN
    KI = np.full((B, L, g.index_hd), 0x7fc1, np.uint16)
    Y = np.zeros((B, L, g.head_dim), np.uint16)
    n = 0
    lens = []
    for start, T in chunks:
        n = orc.compress(gd, ratio, w, kv, sc, np.ascontiguousarray(x[:, start:start + T]), start, tab, Z, KI, n, Y)
        lens.append(n)
    return dict(kv=kv, sc=sc, Z=Z, KI=KI, Y=Y, lens=lens, tab=tab)


def _bf(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rms_bf16(v, w, eps):
    """RMSNorm of an f32 row with f32 arithmetic semantics and a bf16 result (torch's rounding)."""
    v = np.asarray(v, np.float64)
    y = v / np.sqrt(np.mean(v * v) + eps) * np.asarray(w, np.float64)
    return torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("ratio", [2, 4])
def test_state_holds_f32_products(orc, ratio):
    g = _geom()
    w = _weights(orc, g, ratio)
    x = _x(orc, 1, ratio - 1, g.dim)  # one unfinished group: the state keeps every product
    r = _run(orc, g, ratio, w, x, [(0, ratio - 1)])
    xf = _bf(x[0])
    assert np.array_equal(r["kv"][0, :ratio - 1], (xf @ w["wkv"].astype(np.float64).T).astype(np.float32))
    assert np.array_equal(r["sc"][0, :ratio - 1], (xf @ w["wgate"].astype(np.float64).T).astype(np.float32))
    assert np.isneginf(r["sc"][0, ratio - 1:]).all() and (r["kv"][0, ratio - 1:] == 0).all()
    assert r["lens"] == [0]
    assert (r["Z"] == 0x7fc1).all() and (r["KI"] == 0x7fc1).all()  # nothing published


def test_equal_scores_pool_to_the_mean(orc):
    g, ratio = _geom(), 4
    w = _weights(orc, g, ratio)
    w["wgate"] = np.zeros_like(w["wgate"])
    x = _x(orc, 1, ratio, g.dim, seed=3)
    r = _run(orc, g, ratio, w, x, [(0, ratio)])
    k = (_bf(x[0]) @ w["wkv"].astype(np.float64).T).astype(np.float32).astype(np.float64)
    z = k.mean(0).astype(np.float32)
    assert np.array_equal(r["Y"][0, 0], _rms_bf16(z, w["norm"], g.eps))


def test_dominant_score_selects_its_row(orc):
    g, ratio = _geom(), 4
    w = _weights(orc, g, ratio)
    x = _x(orc, 1, ratio, g.dim, seed=4)
    # the gate of slot 2's token is huge on every feature: its row wins the softmax outright
    w["wgate"] = np.zeros_like(w["wgate"])
    xf = _bf(x[0])
    w["wgate"][:] = (1e4 * np.sign(xf[2]) / np.abs(xf[2]).sum()).astype(np.float32)[None, :]
    r = _run(orc, g, ratio, w, x, [(0, ratio)])
    s = xf @ w["wgate"].astype(np.float64).T
    assert (s[2] - np.delete(s, 2, 0).max(0) > 200).all()
    k = (xf @ w["wkv"].astype(np.float64).T).astype(np.float32)
    assert np.array_equal(r["Y"][0, 0], _rms_bf16(k[2], w["norm"], g.eps))


def test_two_rows_pool_to_the_softmax_mixture(orc):
    g, ratio = _geom(), 2
    w = _weights(orc, g, ratio, gate_scale=3.0)
    x = _x(orc, 1, ratio, g.dim, seed=5)
    r = _run(orc, g, ratio, w, x, [(0, ratio)])
    xf = _bf(x[0])
    k = (xf @ w["wkv"].astype(np.float64).T).astype(np.float32).astype(np.float64)
    s = (xf @ w["wgate"].astype(np.float64).T).astype(np.float32).astype(np.float64)
    a = 1.0 / (1.0 + np.exp(s[1] - s[0]))  # weight of row 0
    z = (a * k[0] + (1 - a) * k[1]).astype(np.float32)
    got = _bf(r["Y"][0, 0])
    want = _bf(_rms_bf16(z, w["norm"], g.eps))
    # the closed form rounds differently from the max-shifted sum: at most one bf16 step apart
    assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-30)


@pytest.mark.parametrize("ratio", [1, 2, 4])
def test_rows_compose_the_pinned_primitives(orc, ratio):
    g = _geom()
    w = _weights(orc, g, ratio)
    T = 3 * ratio + 1
    x = _x(orc, 2, T, g.dim, seed=6)
    r = _run(orc, g, ratio, w, x, [(0, T)])
    for b in range(2):
        for j in range(3):
            y = r["Y"][b, j:j + 1]
            ki = orc.rmsnorm(orc.linear_bf16(y, w["wk"]), w["k_norm"], g.eps)
            assert np.array_equal(r["KI"][b, j], ki[0])
            z = orc.apply_rotary(y, g.rope_dim, np.array([j * ratio], np.int32), r["tab"])
            z = orc.act_quant(z)[0]
            assert np.array_equal(r["Z"][b, j], z[0])
    if ratio == 1:  # no pooling: the normed row is RMSNorm(linear_bf16(x, Wkv))
        for t in range(T):
            want = orc.rmsnorm(orc.linear_bf16(x[0, t:t + 1], w["wkv"]), w["norm"], g.eps)
            assert np.array_equal(r["Y"][0, t], want[0])


@pytest.mark.parametrize("ratio", [2, 4])
def test_compress_len_counts_complete_groups(orc, ratio):
    g = _geom()
    w = _weights(orc, g, ratio)
    T0 = 2 * ratio + 1
    x = _x(orc, 1, T0 + 2 * ratio, g.dim, seed=7)
    chunks = [(0, T0)] + [(p, 1) for p in range(T0, T0 + 2 * ratio)]
    r = _run(orc, g, ratio, w, x, chunks)
    want = [T0 // ratio] + [(p + 1) // ratio for p in range(T0, T0 + 2 * ratio)]
    assert r["lens"] == want
    n = want[-1]
    assert (r["Z"][0, n:] == 0x7fc1).all() and (r["Z"][0, :n] != 0x7fc1).any(axis=1).all()
    # the next group is open: its unwritten slots hold -inf scores
    open_slots = (T0 + 2 * ratio) % ratio
    assert np.isneginf(r["sc"][0, open_slots:]).all()


@pytest.mark.parametrize("ratio", [1, 2, 4])
def test_chunks_give_the_same_rows(orc, ratio):
    g = _geom()
    w = _weights(orc, g, ratio)
    T = 6 * ratio + 3
    x = _x(orc, 2, T, g.dim, seed=8)
    one = _run(orc, g, ratio, w, x, [(0, T)])
    split = _run(orc, g, ratio, w, x, [(0, 5), (5, 2 * ratio + 1)] + [(p, 1) for p in range(2 * ratio + 6, T)])
    for k in ("Z", "KI", "Y", "kv", "sc"):
        assert np.array_equal(one[k], split[k]), k
    assert one["lens"][-1] == split["lens"][-1] == T // ratio
