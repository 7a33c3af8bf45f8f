"""Pins for the oracle's RoPE table and rotation and for the window ring (deepseek_v41_ref::attn
rustdoc page: freqs_cis, apply_rotary, window_topk_idxs, WindowCache and the 12-into-8 ring fixture).
"""
import json
import math
import os

import numpy as np
import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_rope_table_closed_form(orc):
    # one pair (rd = 2) turns at frequency theta^0 = 1: the angle is the position itself
    t = orc.rope_table(2, 4000, 10000.0)
    p = np.arange(4000, dtype=np.float64)
    assert np.array_equal(t[:, 0, 0], np.cos(p).astype(np.float32))
    assert np.array_equal(t[:, 0, 1], np.sin(p).astype(np.float32))
    # rd = 64, theta = 10000: pair 16 turns at 10000^(-1/2) = 1/100 per position
    t = orc.rope_table(64, 1001, 10000.0)
    assert abs(float(t[1000, 16, 0]) - math.cos(10.0)) < 1e-7
    assert abs(float(t[1000, 16, 1]) - math.sin(10.0)) < 1e-7
    # position 0 is the identity rotation
    assert (t[0, :, 0] == 1.0).all() and (t[0, :, 1] == 0.0).all()


def test_rope_yarn_structure(orc):
    # no interpolation while the table fits the original length
    a = orc.rope_table(64, 4096, 160000.0, orig_seq=65536, factor=16.0)
    b = orc.rope_table(64, 4096, 160000.0)
    assert np.array_equal(a, b)
    # beyond it: the fastest pairs keep their frequency, the slowest are divided by the factor
    y = orc.rope_table(64, 65537 + 7, 160000.0, orig_seq=65536, factor=16.0)
    f = 160000.0 ** (-2.0 * np.arange(32) / 64)
    ang = np.arctan2(y[1, :, 1].astype(np.float64), y[1, :, 0].astype(np.float64))
    assert abs(ang[0] - f[0]) < 1e-6 and abs(ang[1] - f[1]) < 1e-6
    assert abs(ang[31] - f[31] / 16.0) < 1e-9
    assert np.all(np.diff(ang) < 0)  # still monotone in the pair index


def test_rope_yarn_pairs_by_rotation_count(orc):
    """YaRN's frequency classes (Peng et al., 2023): a pair that completes at least beta_fast turns over
    the original length keeps its frequency, one that completes at most beta_slow turns runs at
    frequency / factor, and the pairs in between lie strictly between the two."""
    L, theta, factor, rd = 65536, 160000.0, 16.0, 64
    y = orc.rope_table(rd, L + 2, theta, orig_seq=L, factor=factor, beta_fast=32.0, beta_slow=1.0)
    f = theta ** (-2.0 * np.arange(rd // 2) / rd)
    turns = L * f / (2 * math.pi)
    ang = np.arctan2(y[1, :, 1].astype(np.float64), y[1, :, 0].astype(np.float64))  # position 1: the frequency
    fast, slow = turns >= 32.0, turns <= 1.0
    assert fast.any() and slow.any() and (~fast & ~slow).any()
    assert np.allclose(ang[fast], f[fast], rtol=2e-7, atol=0)
    assert np.allclose(ang[slow], f[slow] / factor, rtol=2e-7, atol=0)
    mid = ~fast & ~slow
    assert np.all(ang[mid] < f[mid] * (1 - 1e-6)) and np.all(ang[mid] > f[mid] / factor * (1 + 1e-6))


@pytest.mark.parametrize(
    "rd,theta,L,factor,beta_fast,beta_slow",
    [
        (64, 160000.0, 65536, 16.0, 32.0, 1.0),  # the compressed layers' rope constants
        (64, 10000.0, 4096, 40.0, 32.0, 1.0),  # the YaRN paper's long-context extension of a 4k model
        (32, 10.0, 1024, 8.0, 32.0, 1.0),  # the ceiling index past rd - 1: the ramp is cut there
    ],
)
def test_rope_yarn_ramp_weights(orc, rd, theta, L, factor, beta_fast, beta_slow):
    """YaRN's blend inside the ramp (Peng et al., 2023, frequency interpolation by parts): pair i runs
    at f_i (1 - w_i) + (f_i / factor) w_i with w_i = clamp((i - lo) / (hi - lo), 0, 1), lo the last
    pair index (counted on past rd / 2 where needed) that still completes beta_fast turns over the
    original length, hi the first that completes at most beta_slow, capped at rd - 1.  Both ends are
    found here by searching the rotation counts, not from the closed-form index, and the weights are
    read back from the table's angle at position 1."""
    y = orc.rope_table(rd, L + 2, theta, orig_seq=L, factor=factor, beta_fast=beta_fast, beta_slow=beta_slow)
    idx = np.arange(4 * rd, dtype=np.float64)
    turns = L * theta ** (-2.0 * idx / rd) / (2 * math.pi)  # strictly decreasing in the index
    lo = max(int(np.nonzero(turns >= beta_fast)[0].max()) if (turns >= beta_fast).any() else 0, 0)
    hi = min(int(np.nonzero(turns <= beta_slow)[0].min()), rd - 1)
    assert hi > lo
    half = rd // 2
    i = np.arange(half, dtype=np.float64)
    f = theta ** (-2.0 * i / rd)
    ang = np.arctan2(y[1, :, 1].astype(np.float64), y[1, :, 0].astype(np.float64))
    w = (1.0 - ang / f) / (1.0 - 1.0 / factor)  # 0: the pair keeps f_i, 1: it runs at f_i / factor
    expect = np.clip((i - lo) / (hi - lo), 0.0, 1.0)
    assert np.all(np.abs(w - expect) < 2e-6), np.abs(w - expect).max()
    # the ramp is really exercised: some pairs strictly inside it
    assert ((expect > 0) & (expect < 1)).sum() >= 3


def test_rotary_adjacent_pairs_and_inverse(orc):
    rd, hd = 16, 64
    tab = orc.rope_table(rd, 64, 10000.0)
    x = np.zeros((1, hd), np.float32)
    x[0, hd - rd] = 1.0  # first element of the rotated tail: real part of pair 0
    xb = orc.f32_to_bf16(x)
    y = orc.bf16_to_f32(orc.apply_rotary(xb, rd, np.array([5]), tab))
    # adjacent pairs: (1, 0) -> (cos 5, sin 5) in elements (hd-rd, hd-rd+1); the rest untouched
    assert y[0, hd - rd] == orc.bf16_to_f32(orc.f32_to_bf16(np.float32(math.cos(5.0))))
    assert y[0, hd - rd + 1] == orc.bf16_to_f32(orc.f32_to_bf16(np.float32(math.sin(5.0))))
    assert (y[0, hd - rd + 2:] == 0).all() and (y[0, : hd - rd] == 0).all()
    rng = np.random.default_rng(5)
    v = orc.f32_to_bf16(rng.standard_normal((300, hd)).astype(np.float32))
    pos = rng.integers(0, 64, 300).astype(np.int32)
    r = orc.apply_rotary(v, rd, pos, tab)
    assert np.array_equal(r[:, : hd - rd], v[:, : hd - rd])
    back = orc.apply_rotary(r, rd, pos, tab, inverse=True)
    vf, bf = orc.bf16_to_f32(v).astype(np.float64), orc.bf16_to_f32(back).astype(np.float64)
    # forward then inverse: identity up to two bf16 roundings of each element
    assert np.all(np.abs(bf - vf) <= 2 ** -7 * (np.abs(vf) + np.abs(vf[:, ::-1]).max()) + 1e-30)
    # a rotation keeps each pair's modulus up to bf16 rounding
    rv = orc.bf16_to_f32(r).astype(np.float64)[:, hd - rd:].reshape(300, rd // 2, 2)
    vv = vf[:, hd - rd:].reshape(300, rd // 2, 2)
    assert np.allclose(np.hypot(rv[..., 0], rv[..., 1]), np.hypot(vv[..., 0], vv[..., 1]), rtol=2 ** -7, atol=1e-6)


def test_rotary_rounds_each_product_to_f32(orc):
    """The complex product rounds each product and each sum to f32 on its own ([ref-attn] apply_rotary:
    the pairs multiplied in f32).  With a = b = 1 + 2^-7 and (c, s) = (1 + 2^-23, 1), a c = 1 + 2^-7 +
    2^-23 + 2^-30 rounds to 1 + 2^-7 + 2^-23, so re = fl(a c) - fl(b s) is exactly 2^-23; a fused
    multiply-add, or a wider sum, keeps the 2^-30 and gives 2^-23 (1 + 2^-7), another bf16 value."""
    u = 2.0 ** -7
    x = orc.f32_to_bf16(np.array([[1 + u, 1 + u]], np.float32))
    tab = np.array([[[1 + 2.0 ** -23, 1.0]]], np.float32)
    y = orc.apply_rotary(x, 2, np.array([0], np.int32), tab)
    bits = lambda v: int(orc.f32_to_bf16(np.array([v], np.float32))[0])
    re_bits = int(y[0, 0])
    assert re_bits == bits(2.0 ** -23)
    assert re_bits != bits(2.0 ** -23 * (1 + u))
    # im = fl(fl(a s) + fl(b c)) = fl(2 + 2^-6 + 2^-23): a tie in f32, to even: 2 + 2^-6
    assert int(y[0, 1]) == bits(2 + 2.0 ** -6)


def test_rotary_composes_angles(orc):
    rd, hd = 8, 8
    tab = orc.rope_table(rd, 64, 10000.0)
    x = orc.f32_to_bf16(np.tile(np.array([1.0, 0.0], np.float32), (1, 4)))
    y = orc.bf16_to_f32(orc.apply_rotary(x, rd, np.array([7]), tab)).astype(np.float64)
    f = 10000.0 ** (-2.0 * np.arange(4) / 8)
    assert np.allclose(y[0, 0::2], np.cos(7 * f), atol=4e-3) and np.allclose(y[0, 1::2], np.sin(7 * f), atol=4e-3)


def test_ring_fixture_helpers(orc):
    g = json.load(open(os.path.join(GOLD, "ring_fixture.json")))
    W, T = g["window"], g["prefill_tokens"]
    rows = np.zeros((T, 4), np.uint16)
    rows[:, 0] = np.arange(T) + 100  # tag rows by token
    ring = np.zeros((W, 4), np.uint16)
    orc.ring_write(ring, rows, 0)
    assert list(ring[:, 0] - 100) == g["slot_token_after_prefill"]
    for d in g["decode"]:
        r = np.full((1, 4), 100 + d["pos"], np.uint16)
        before = ring.copy()
        orc.ring_write(ring, r, d["pos"])
        changed = np.nonzero((ring != before).any(1))[0]
        assert list(changed) == [d["write_slot"]]
        if "read_slots_oldest_first" in d:
            assert list(orc.window_idx_decode(d["pos"], W)) == d["read_slots_oldest_first"]
            # oldest first means ascending token order along the read
            toks = ring[orc.window_idx_decode(d["pos"], W), 0] - 100
            assert list(toks) == list(range(d["pos"] - W + 1, d["pos"] + 1))


def test_window_idx_prefill_and_young_ring(orc):
    idx = orc.window_idx_prefill(12, 8)
    assert list(idx[0]) == [-1] * 7 + [0]
    assert list(idx[3]) == [-1] * 4 + [0, 1, 2, 3]
    assert list(idx[11]) == list(range(4, 12))
    # a decode step before the ring is full: slots never written are -1
    assert list(orc.window_idx_decode(2, 8)) == [-1] * 5 + [0, 1, 2]
    assert list(orc.window_idx_decode(7, 8)) == list(range(8))


def test_ring_fixture_through_layer(orc):
    """The fixture's three regimes in order through one ring, with the layer's own kv rows."""
    from csa_inputs import WORKLOADS, weights, activations
    wl = WORKLOADS["tiny_ratio0"]
    g = wl.geom.as_dict()
    fx = json.load(open(os.path.join(GOLD, "ring_fixture.json")))
    w = weights(wl.geom, with_indexer=False)
    x = activations(wl.geom, 1, 14)
    tab = orc.rope_table(g["rope_dim"], g["max_seq"], g["rope_theta"])
    ring = np.zeros((1, g["window"], g["head_dim"]), np.uint16)
    r0 = orc.attn_forward(g, dict(ratio=0), w, ring, x[:, :12], 0, tab)
    kv = r0["kv"]
    for slot, tok in enumerate(fx["slot_token_after_prefill"]):
        assert np.array_equal(ring[0, slot], kv[tok])
    for step in fx["decode"]:
        p = step["pos"]
        r = orc.attn_forward(g, dict(ratio=0), w, ring, x[:, p:p + 1], p, tab)
        assert np.array_equal(ring[0, step["write_slot"]], r["kv"][0])
        if "read_slots_oldest_first" in step:
            assert list(r["idx"][0]) == step["read_slots_oldest_first"]
    # prefill window selection is the chunk's causal window
    assert list(r0["idx"][11]) == list(range(4, 12)) and list(r0["idx"][2]) == [-1] * 5 + [0, 1, 2]
