"""The benchmark's selection sizes and algorithmic bytes, the numerators of its bandwidth figures,
against closed forms of the workloads (no GPU).

The per-token bytes restate the measurement's definitions: sparse attention reads q (H hd bf16) and
each gathered row (hd bf16) once, writes o (H hd bf16) and reads its index row (int32); the indexer
reads Q^I (Hi dI bf16), w^I (Hi f32), the mask row and each valid key (dI bf16) once and writes each
valid score (f32); the top-k reads the mask row and each valid score and writes K int32 indices.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from csa_inputs import WORKLOADS, candidate_mask, positions  # noqa: E402


def _shared(wl):
    g = wl.geom
    if not wl.ratio:
        return None
    L = wl.compress_len
    cand = None
    if wl.uses_candidates:
        pos = positions(wl.batch, wl.tokens, wl.start_pos)
        cand = candidate_mask(wl.batch * wl.tokens, pos, wl.ratio, L, g.cand_block, -(-L // g.cand_block),
                              wl.cand_keep, 1015)
    return dict(L=L, cand=cand)


def test_prefill_counts_closed_form():
    """4096 queries at t = 0..4095, ratio 4, 1024 latent rows, window 128, K = 512, no mask: query t
    gathers min(t+1, 128) window rows and min(floor((t+1)/4), 512) compressed ones."""
    import bench
    wl = WORKLOADS["prefill_r4"]
    rows, n_valid = bench.selection_counts(wl, _shared(wl))
    # sum_{n=1..4096} min(n, 128) = 128*129/2 + (4096-128)*128
    window = 128 * 129 // 2 + (4096 - 128) * 128
    # floor(n/4) for n = 1..4095 takes 0 three times and each m = 1..1023 four times; n = 4096 gives 1024
    valid = 4 * (1023 * 1024 // 2) + 1024
    # capped at 512 from n = 2048 on: n = 1..2047 sum to 4 * (0 + ... + 511), n = 2048..4096 give 512 each
    capped = 4 * (511 * 512 // 2) + (4096 - 2047) * 512
    assert n_valid == valid == 2096128
    assert rows == window + capped == 2088512


def test_long_context_counts_and_bytes_closed_form():
    """64 queries at p = 65535, ratio 4, 16384 latent rows, 64 of 256 blocks of 64 kept (all full), four
    layers: 128 + 512 gathered rows and 4096 valid keys a query."""
    import bench
    wl = WORKLOADS["longctx_decode_r4"]
    g = wl.geom
    sh = _shared(wl)
    assert (sh["cand"].sum(1) == 64).all()
    rows, n_valid = bench.selection_counts(wl, sh)
    assert rows == 64 * (128 + 512) and n_valid == 64 * 4096
    attn, idx, topk = bench.algorithmic_bytes(wl, sh, (rows, n_valid))
    NT, H, hd, Hi, dI, K, W, cw = 64, g.n_heads, g.head_dim, g.index_heads, g.index_hd, g.index_topk, g.window, 256
    per_layer_attn = NT * (2 * H * hd * 2 + (W + K) * 4) + rows * hd * 2
    per_layer_idx = NT * (Hi * dI * 2 + Hi * 4 + cw) + n_valid * (dI * 2 + 4)
    per_layer_topk = NT * (cw + K * 4) + n_valid * 4
    assert (attn, idx, topk) == (4 * per_layer_attn, 4 * per_layer_idx, 4 * per_layer_topk)
    assert attn + idx + topk == 481591296


def test_reindex_decode_counts_follow_the_mask():
    """32 queries at p = 1000, ratio 2, 500 latent rows (valid j < 500), blocks of 64 with four of the
    eight causal blocks kept: a kept block holds 64 valid keys, except the last (448..499), which holds
    52; every query gathers its 128 window rows and all of its valid keys (at most 256 < K)."""
    import bench
    wl = WORKLOADS["reindex_decode_r2"]
    sh = _shared(wl)
    cand = sh["cand"]
    assert cand.shape == (32, 8) and (cand.sum(1) == 4).all()
    last_kept = int(cand[:, 7].astype(np.int64).sum())
    rows, n_valid = bench.selection_counts(wl, sh)
    assert n_valid == 32 * 4 * 64 - 12 * last_kept
    assert rows == 32 * 128 + n_valid


def test_projection_bytes_match_the_parameter_table():
    """The projections' algorithmic bytes of the Reindex decode step: every projection weight of the
    layer once (the pages' parameter table, less the sink and the two norm vectors, which are not
    projection weights), plus the 32 tokens' activations in and out of the four stages, bf16."""
    import json
    import bench
    wl = WORKLOADS["reindex_decode_r2"]
    g = wl.geom
    pc = json.load(open(os.path.join(ROOT, "tests", "golden", "param_counts.json")))
    weights = pc["per_instance_total"] - g.n_heads - g.q_rank - g.head_dim  # sink, q_norm, kv_norm
    M = wl.batch * wl.tokens
    acts = M * ((g.dim + g.q_rank + g.head_dim + g.index_heads)  # proj x: x in; qr, kv, w^I out
                + (g.q_rank + g.n_heads * g.head_dim + g.index_heads * g.index_hd)  # proj qr: qr in; q, q^I out
                + (g.n_heads * g.head_dim + g.groups * g.o_rank)  # wo_a: O in, og out
                + (g.groups * g.o_rank + g.dim))  # wo_b: og in, out
    got = bench.projection_bytes(wl)
    assert set(got) == {"proj x", "proj qr", "wo_a", "wo_b"}
    assert sum(got.values()) == 2 * (weights + acts) == 270403584


def test_prefill_scored_pairs_closed_form():
    """The indexer's scored pairs at prefill: only the queries with more than K = 512 valid positions
    are scored (the others' selections take every position).  floor((t+1)/4) > 512 from t = 2051 on;
    each value v = 513..1023 occurs for four consecutive t, and 1024 once (t = 4095)."""
    import bench
    wl = WORKLOADS["prefill_r4"]
    want = 4 * sum(range(513, 1024)) + 1024
    assert bench.scored_pairs(wl, _shared(wl)) == want == 1570816
    # with a candidate mask every valid pair is scored
    wl2 = WORKLOADS["longctx_decode_r4"]
    sh2 = _shared(wl2)
    assert bench.scored_pairs(wl2, sh2) == bench.selection_counts(wl2, sh2)[1]

