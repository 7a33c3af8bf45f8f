"""GPU parity of the whole layer (attn_v41_forward through the C ABI) against the CPU oracle.

Small geometries run every token; the full-width workloads compare sampled queries (the oracle
computes those rows one by one) in the launch configuration the benchmark times.  Tolerances:
layer and attention outputs atol/rtol 2e-2 plus a relative error norm of 1e-2; fp8-rounded rows at
most one e4m3 step apart (the projections feeding them round differently); window indices exact;
the compressed selection equal to the oracle's wherever the K-th and (K+1)-th oracle scores are
further apart than the score tolerance, otherwise a valid top-K within that tolerance.
"""
import math

import numpy as np
import pytest
import torch

from csa_inputs import (WORKLOADS, Geometry, activations, candidate_mask, latent_cache, positions, ring_rows,
                        weights)
from _helpers import assert_close_bf16, assert_same_selection, bf, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_attn_gb300 as m
    m.lib()
    return m


def _dev_weights(w):
    return {k: to_dev(v) for k, v in w.items()}


def _assert_fp8_rows_close(got, want, what):
    """fp8-rounded rows whose bf16 inputs differ by the projections' rounding: each element within one
    e4m3 step of the oracle's, plus one bf16 ulp of the row's RMS (the RoPE tail subtracts products
    of O(1) values, so a one-ulp input difference is absolute, not relative to the result)."""
    g, w = bf(got).astype(np.float64), bf(want).astype(np.float64)
    rms = np.sqrt(np.mean(w * w, axis=-1, keepdims=True))
    step = 0.13 * np.maximum(np.abs(g), np.abs(w)) + 2.0 ** -7 * rms + 1e-6
    bad = np.abs(g - w) > step
    if bad.any():
        idx = np.argwhere(bad)
        r0 = idx[0][:-1]
        rows = sorted(set(tuple(i[:-1]) for i in idx))
        raise AssertionError("%s: %d elements more than one e4m3 step apart in %d rows %s...; first row %s: "
                             "got %s want %s at cols %s" % (what, len(idx), len(rows), rows[:8], tuple(r0),
                                                            g[tuple(r0)][bad[tuple(r0)]][:8],
                                                            w[tuple(r0)][bad[tuple(r0)]][:8],
                                                            np.nonzero(bad[tuple(r0)])[0][:8]))
    assert np.linalg.norm(g - w) <= 2e-2 * np.linalg.norm(w) + 1e-6, what


def _check_selection(got, S_row, K, offset, tol):
    """got: the GPU's selection row (j + offset, -1 padded); S_row: oracle scores (-inf = invalid)."""
    valid = np.isfinite(S_row)
    n = int(valid.sum())
    sel = [v - offset for v in got if v >= 0]
    assert len(sel) == min(n, K) and len(set(sel)) == len(sel)
    assert all(valid[j] for j in sel)
    if n <= K:
        assert set(sel) == set(np.nonzero(valid)[0])
        return
    order = sorted(np.nonzero(valid)[0], key=lambda j: (-S_row[j], j))
    kth, nxt = S_row[order[K - 1]], S_row[order[K]]
    if kth - nxt > tol:
        assert set(sel) == set(order[:K])
    else:
        assert min(S_row[j] for j in sel) >= kth - tol


def _dbg(NT, g, L, with_idx_cols):
    H, hd = g.n_heads, g.head_dim
    z = lambda *s, dt=torch.bfloat16: torch.zeros(*s, dtype=dt, device="cuda")
    return dict(q=z(NT, H, hd), kv=z(NT, hd), kv_codes=z(NT, hd, dt=torch.uint8), kv_scale=z(NT, hd // 32, dt=torch.int8),
                idx=torch.full((NT, with_idx_cols), -9, dtype=torch.int32, device="cuda"),
                scores=torch.full((NT, max(L, 1)), float("nan"), device="cuda"), o=z(NT, H, hd),
                og=z(NT, g.groups * g.o_rank), qr=z(NT, g.q_rank), qI=z(NT, max(g.index_heads * g.index_hd, 1)),
                wI=z(NT, max(g.index_heads, 1), dt=torch.float32))


def _compare_rows(res, dbg, rows, g, what):
    NT = len(rows)
    out = res["out"].reshape(-1, g.dim)[rows]
    assert_close_bf16(to_np(dbg["__out"]).reshape(-1, g.dim)[rows], out, what=what + " out")
    assert_close_bf16(to_np(dbg["o"])[rows], res["o"][rows], what=what + " o")
    assert_close_bf16(to_np(dbg["q"])[rows], res["q"][rows], what=what + " q")
    _assert_fp8_rows_close(to_np(dbg["kv"])[rows], res["kv"][rows], what + " kv")


def _compare_indexer_inputs(res, dbg, grows, rows, what):
    """The indexer's query q^I = qr W_IQ^T (bf16) and head weights w^I = bf16(x W_IW^T) / sqrt(dI Hi)
    (f32), read back from the forward: within the bf16 output tolerance, as their inputs differ by the
    projections' rounding."""
    assert_close_bf16(to_np(dbg["qI"])[grows], res["qI"][rows], what=what + " qI")
    wg = to_np(dbg["wI"])[grows].astype(np.float64)
    wo = res["wI"][rows].astype(np.float64)
    assert np.all(np.abs(wg - wo) <= 2e-2 * np.abs(wo) + 2e-2 * np.abs(wo).max()), what + " wI"


# ------------------------------------------------------------------------------------- tiny

def test_tiny_ratio0_prefill_then_decode(csa, orc):
    """The ring fixture's three regimes through one cache, GPU against oracle."""
    wl = WORKLOADS["tiny_ratio0"]
    g = wl.geom
    gd = g.as_dict()
    w = weights(g, with_indexer=False)
    x = activations(g, 1, 14)
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.rope_theta)
    ring_o = np.zeros((1, g.window, g.head_dim), np.uint16)
    ctx = csa.Context(gd)
    wd = _dev_weights(w)
    ring_d = torch.zeros((1, g.window, g.head_dim), dtype=torch.bfloat16, device="cuda")
    ctx.state_init(ring_d, 1)
    for start, T in ((0, 12), (12, 1), (13, 1)):
        xs = x[:, start:start + T] if start else x[:, :12]
        res = orc.attn_forward(gd, dict(ratio=0), w, ring_o, xs, start, tab)
        dbg = _dbg(T, g, 1, g.window)
        out = ctx.forward(wd, dict(ratio=0), ring_d, to_dev(xs), start, debug=dbg)
        torch.cuda.synchronize()
        dbg["__out"] = out
        _compare_rows(res, dbg, np.arange(T), g, "tiny@%d" % start)
        assert np.array_equal(to_np(dbg["idx"]), res["idx"])
        _assert_fp8_rows_close(to_np(ring_d), ring_o, "ring@%d" % start)
    assert ctx.status() == 0


def _small_geom():
    return Geometry(dim=96, n_heads=4, head_dim=64, rope_dim=16, q_rank=48, o_rank=24, groups=2, window=8,
                    index_heads=4, index_hd=32, index_topk=8, cand_block=4, max_seq=256, max_tokens=40, max_batch=3)


@pytest.mark.parametrize("start,T,B,cand", [(0, 40, 2, True), (0, 40, 1, False), (77, 1, 3, True), (5, 1, 3, False)])
def test_small_ratio2_index_source_and_reuse(csa, orc, start, T, B, cand):
    g = _small_geom()
    gd = g.as_dict()
    L = 64
    w = weights(g, with_indexer=True, norm_ones=False)
    x = activations(g, B, T, seed_base=2000 + start)
    Z, KI = latent_cache(g, B, L, seed_base=3000)
    clen = min(L, (start + T) // 2 + 3)
    pos = positions(B, T, start)
    cm = candidate_mask(B * T, pos, 2, clen, g.cand_block, L // g.cand_block, 0.5, 99) if cand else None
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor)
    ring0 = orc.act_quant(ring_rows(g, B))[0] if start else np.zeros((B, g.window, g.head_dim), np.uint16)
    ring_o = ring0.copy()
    sel_o = np.full((B * T, g.index_topk), -7, np.int32)
    shared_o = dict(compress_kv=Z, index_k=KI, compress_len=clen, topk_idxs=sel_o)
    if cand:
        shared_o["candidates"] = cm
    role = dict(ratio=2, is_index_source=1, uses_candidates=int(cand))
    res = orc.attn_forward(gd, role, w, ring_o, x, start, tab, shared_o)

    ctx = csa.Context(gd)
    wd = _dev_weights(w)
    ring_d = to_dev(ring0)
    sel_d = torch.full((B * T, g.index_topk), -7, dtype=torch.int32, device="cuda")
    sh = csa.Shared(to_dev(Z), to_dev(KI), clen, sel_d, g.index_topk, None if cm is None else to_dev(cm))
    dbg = _dbg(B * T, g, L, g.window + g.index_topk)
    out = ctx.forward(wd, role, ring_d, to_dev(x), start, shared=sh, debug=dbg)
    torch.cuda.synchronize()
    assert sh.has_topk
    dbg["__out"] = out
    rows = np.arange(B * T)
    _compare_rows(res, dbg, rows, g, "ratio2")
    _compare_indexer_inputs(res, dbg, rows, rows, "ratio2")
    gi = to_np(dbg["idx"])
    assert np.array_equal(gi[:, :g.window], res["idx"][:, :g.window])
    # scores: inputs differ by the projections' bf16 rounding, so 1e-2 here (1e-3 at the kernel level)
    S_g = to_np(dbg["scores"])[:, :L]
    S_o = res["scores"]
    for r in rows:
        v = np.isfinite(S_o[r])
        if v.any():
            tol = 1e-2 * np.abs(S_o[r, v]).max()
            assert (np.abs(S_g[r, v] - S_o[r, v]) <= 1e-2 * np.abs(S_o[r, v]) + tol).all()
            _check_selection(gi[r, g.window:], S_o[r], g.index_topk, g.window if start else T, 2 * tol)
    assert np.array_equal(to_np(sel_d), gi[:, g.window:])
    # a reuse layer reads the published selection: same rows as the index source
    reuse = dict(ratio=2, is_index_source=0)
    ring_d2 = to_dev(ring0)
    out2 = ctx.forward(wd, reuse, ring_d2, to_dev(x), start, shared=sh)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(out2), to_np(out))
    assert ctx.status() == 0


@pytest.mark.parametrize("cand", [False, True])
def test_fused_indexer_topk_selection(csa, orc, cand):
    """Decode rows of at most 512 positions take scores and top-k in one kernel (tensor-core indexer
    shapes: 16 heads x 128); with K = 64 below the valid count the selection is a real cut.  The fast
    path (no debug buffers) must publish exactly the selection of the two-kernel path (debug scores
    requested), which must be the oracle's top-k of those very scores, bit for bit."""
    g = Geometry(dim=128, n_heads=4, head_dim=64, rope_dim=16, q_rank=64, o_rank=32, groups=2, window=8,
                 index_heads=16, index_hd=128, index_topk=64, cand_block=64, max_seq=1024, max_tokens=1, max_batch=4)
    gd = g.as_dict()
    B, T, start, L = 4, 1, 700, 384
    clen = 300  # limit min(701 // 2, 300) = 300 positions: three key tiles
    w = weights(g, with_indexer=True, norm_ones=False)
    x = activations(g, B, T, seed_base=2100 + int(cand))
    Z, KI = latent_cache(g, B, L, seed_base=3100)
    pos = positions(B, T, start)
    cm = candidate_mask(B * T, pos, 2, clen, g.cand_block, L // g.cand_block, 4, 98) if cand else None
    ring0 = orc.act_quant(ring_rows(g, B))[0]
    role = dict(ratio=2, is_index_source=1, uses_candidates=int(cand))
    ctx = csa.Context(gd)
    wd = _dev_weights(w)
    K = g.index_topk
    sel_d = torch.full((B * T, K), -7, dtype=torch.int32, device="cuda")
    sh = csa.Shared(to_dev(Z), to_dev(KI), clen, sel_d, K, None if cm is None else to_dev(cm))
    out_fast = ctx.forward(wd, role, to_dev(ring0), to_dev(x), start, shared=sh)
    sel_fast = sel_d.clone()
    dbg = _dbg(B * T, g, L, g.window + K)
    out = ctx.forward(wd, role, to_dev(ring0), to_dev(x), start, shared=sh, debug=dbg)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    assert torch.equal(sel_fast, sel_d)
    assert torch.equal(out_fast, out)
    S = to_np(dbg["scores"])[:, :L].astype(np.float32)
    S = np.where(np.isnan(S), -np.inf, S).astype(np.float32)
    want = orc.index_topk(S, K, pos, 2, clen, cm, g.cand_block, offset=g.window)
    assert_same_selection(to_np(sel_fast), want)
    n_valid = np.isfinite(S).sum(1)
    assert (n_valid > K).all()  # the cut is real on every row


@pytest.mark.parametrize("case", ["no latent rows yet", "masks keeping nothing"])
def test_ratio2_decode_degenerate_selection(csa, orc, case):
    """Degenerate selections of a ratio-2 index-source decode: before any latent row is published
    (compress_len 0) every selected entry is -1 and the attention runs over the window alone; with a
    candidate mask keeping no block for some queries, those queries select nothing either."""
    g = _small_geom()
    gd = g.as_dict()
    B, T, start, L = 3, 1, 40, 64
    w = weights(g, with_indexer=True, norm_ones=False)
    x = activations(g, B, T, seed_base=2200)
    Z, KI = latent_cache(g, B, L, seed_base=3200)
    clen = 0 if case == "no latent rows yet" else 20
    pos = positions(B, T, start)
    cm = None
    if case != "no latent rows yet":
        cm = candidate_mask(B * T, pos, 2, clen, g.cand_block, L // g.cand_block, 0.5, 97)
        cm[0, :] = 0
        cm[2, :] = 0
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor)
    ring0 = orc.act_quant(ring_rows(g, B))[0]
    ring_o = ring0.copy()
    sel_o = np.full((B * T, g.index_topk), -7, np.int32)
    shared_o = dict(compress_kv=Z, index_k=KI, compress_len=clen, topk_idxs=sel_o)
    if cm is not None:
        shared_o["candidates"] = cm
    role = dict(ratio=2, is_index_source=1, uses_candidates=int(cm is not None))
    res = orc.attn_forward(gd, role, w, ring_o, x, start, tab, shared_o)
    ctx = csa.Context(gd)
    sel_d = torch.full((B * T, g.index_topk), -7, dtype=torch.int32, device="cuda")
    sh = csa.Shared(to_dev(Z), to_dev(KI), clen, sel_d, g.index_topk, None if cm is None else to_dev(cm))
    dbg = _dbg(B * T, g, L, g.window + g.index_topk)
    out = ctx.forward(_dev_weights(w), role, to_dev(ring0), to_dev(x), start, shared=sh, debug=dbg)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    sel = to_np(sel_d)
    if case == "no latent rows yet":
        assert (sel == -1).all()
    else:
        assert (sel[0] == -1).all() and (sel[2] == -1).all() and (sel[1] >= 0).any()
    dbg["__out"] = out
    _compare_rows(res, dbg, np.arange(B * T), g, case)


def test_layer_refusals(csa):
    g = _small_geom()
    ctx = csa.Context(g.as_dict())
    w = _dev_weights(weights(g, with_indexer=True))
    ring = torch.zeros((3, g.window, g.head_dim), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((1, 2, g.dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=2, is_index_source=1), ring, x, 0)
    assert e.value.code == -3
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=0), ring, x, 5)
    assert e.value.code == -2
    sel = torch.zeros((2, g.index_topk), dtype=torch.int32, device="cuda")
    Z = torch.zeros((1, 16, g.head_dim), dtype=torch.bfloat16, device="cuda")
    sh = csa.Shared(Z, None, 4, sel, g.index_topk)
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=2, is_index_source=0), ring, x, 0, shared=sh)
    assert e.value.code == -4
    # a kv source without its compressor weights and state, a candidate source without a mask to
    # write or that would apply one: argument errors, nothing launched
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=2, is_kv_source=1), ring, x, 0, shared=sh)
    assert e.value.code == -1
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=2, is_index_source=1, is_candidate_source=1), ring, x, 0, shared=sh)
    assert e.value.code == -1
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=2, is_index_source=1, is_candidate_source=1, uses_candidates=1), ring, x, 0,
                    shared=sh)
    assert e.value.code == -1
    with pytest.raises(csa.CsaError) as e:
        ctx.forward(w, dict(ratio=0), ring, torch.zeros((1, 41, g.dim), dtype=torch.bfloat16, device="cuda"), 0)
    assert e.value.code == -2


# ------------------------------------------------------------------------------------- full width

def _full_case(orc, name, seqs, toks=None):
    wl = WORKLOADS[name]
    g = wl.geom
    B, T, start = wl.batch, wl.tokens, wl.start_pos
    w = weights(g, with_indexer=wl.is_index_source)
    x = activations(g, B, T)
    pos = positions(B, T, start)
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta if wl.ratio else g.rope_theta, g.orig_seq
                         if wl.ratio else 0, g.rope_factor, g.beta_fast, g.beta_slow)
    ring0 = orc.act_quant(ring_rows(g, B))[0] if start else np.zeros((B, g.window, g.head_dim), np.uint16)
    shared = None
    if wl.ratio:
        L = wl.compress_len
        Z, KI = latent_cache(g, B, L)
        shared = dict(compress_kv=Z, index_k=KI, compress_len=L, topk_idxs=None)
        if wl.uses_candidates:
            shared["candidates"] = candidate_mask(B * T, pos, wl.ratio, L, g.cand_block, -(-L // g.cand_block),
                                                  wl.cand_keep, 1015)
    return wl, g, w, x, tab, ring0, shared


@pytest.mark.parametrize("name,seqs,toks", [
    ("ratio0_decode", [0, 13, 31], None),
    ("reindex_decode_r2", [0, 7, 31], None),
    ("prefill_r4", [0], [0, 1, 127, 128, 1000, 2047, 2048, 3001, 4095]),
    ("longctx_decode_r4", [0, 63], None),
])
def test_full_width_sampled(csa, orc, name, seqs, toks):
    wl, g, w, x, tab, ring0, shared = _full_case(orc, name, seqs, toks)
    gd = g.as_dict()
    B, T, start = wl.batch, wl.tokens, wl.start_pos
    K = g.index_topk
    # GPU: the whole batch, as the benchmark runs it
    ctx = csa.Context(gd)
    wd = _dev_weights(w)
    ring_d = to_dev(ring0)
    role = dict(ratio=wl.ratio, is_index_source=int(wl.is_index_source), uses_candidates=int(wl.uses_candidates))
    sh = None
    if shared is not None:
        sel_d = torch.full((B * T, K), -7, dtype=torch.int32, device="cuda")
        sh = csa.Shared(to_dev(shared["compress_kv"]), to_dev(shared["index_k"]), shared["compress_len"], sel_d, K,
                        None if "candidates" not in shared else to_dev(shared["candidates"]))
    L = shared["compress_len"] if shared else 1
    xd = to_dev(x)
    # the benchmark's path first (no debug buffers: q's RoPE runs inside the attention kernel), then the
    # debug path (RoPE as its own pass, so the turned q can be read back); same inputs, same ring update
    out_fast = ctx.forward(wd, role, ring_d, xd, start, shared=sh)
    sel_fast = sel_d.clone() if shared is not None else None
    dbg = _dbg(B * T, g, L, g.window + (K if wl.ratio else 0))
    out = ctx.forward(wd, role, ring_d, xd, start, shared=sh, debug=dbg)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    # the fast path (q's RoPE inside the attention kernel; at short decode rows, scores and top-k in one
    # kernel) must give the debug path's selection and output bit for bit
    if sel_fast is not None and wl.is_index_source:
        assert torch.equal(sel_fast, sel_d), name + ": the fused indexer + top-k changes the selection"
    assert torch.equal(out_fast, out), name + ": the fast path changes the layer output"
    dbg["__out"] = out
    # oracle: only the sampled sequences (and, for the prefill chunk, the sampled tokens)
    for b in seqs:
        xb = x[b:b + 1]
        ring_o = ring0[b:b + 1].copy()
        sh_o = None
        if shared is not None:
            sh_o = dict(compress_kv=shared["compress_kv"][b:b + 1], index_k=shared["index_k"][b:b + 1],
                        compress_len=shared["compress_len"], topk_idxs=np.full((T, K), -7, np.int32))
            if "candidates" in shared:
                sh_o["candidates"] = shared["candidates"][b * T:(b + 1) * T]
        mask = None
        rows = np.arange(T)
        if toks is not None:
            mask = np.zeros(T, np.uint8)
            mask[toks] = 1
            rows = np.array(toks)
        res = orc.attn_forward(gd, role, w, ring_o, xb, start, tab, sh_o, tok_mask=mask)
        grows = b * T + rows
        assert_close_bf16(to_np(out).reshape(-1, g.dim)[grows], res["out"].reshape(-1, g.dim)[rows], what=name + " out")
        assert_close_bf16(to_np(dbg["o"])[grows], res["o"][rows], what=name + " o")
        _assert_fp8_rows_close(to_np(dbg["kv"])[grows], res["kv"][rows], name + " kv")
        if wl.ratio and wl.is_index_source:
            _compare_indexer_inputs(res, dbg, grows, rows, name)
        if toks is not None:  # every window row the oracle built: the sampled queries' windows and the ring's
            built = np.nonzero(np.abs(res["kv"].astype(np.int64)).sum(1))[0]
            _assert_fp8_rows_close(to_np(dbg["kv"])[b * T + built], res["kv"][built], name + " kv(all built)")
        gi = to_np(dbg["idx"])[grows]
        assert np.array_equal(gi[:, :g.window], res["idx"][rows, :g.window])
        _assert_fp8_rows_close(to_np(ring_d)[b], ring_o[0], name + " ring")
        if wl.ratio:
            S_o = res["scores"]
            for i, r in enumerate(rows):
                v = np.isfinite(S_o[r])
                if v.any():
                    tol = 1e-2 * np.abs(S_o[r, v]).max()
                    _check_selection(gi[i, g.window:], S_o[r], K, g.window if start else T, 2 * tol)


def test_fp8_wo_a_layer(csa, orc):
    """The Reindex decode layer (full width, 32 sequences at p = 1000) with the grouped wo_a kept in fp8
    (e4m3 codes and one scale per 128 x 128 tile): its output equals, bit for bit, the layer with the
    dequantised bf16 wo_a, and the oracle on those weights on sampled sequences.  The fp8 storage is the
    workload's bf16 wo_a encoded with the oracle's e4m3 rounding at scale amax / 448 per tile, so the
    layer keeps its usual magnitudes."""
    wl, g, w, x, tab, ring0, shared = _full_case(orc, "reindex_decode_r2", [0, 31])
    gd = g.as_dict()
    B, T, start, K = wl.batch, wl.tokens, wl.start_pos, g.index_topk
    gw = g.n_heads * g.head_dim // g.groups
    wf = bf(w["wo_a"]).reshape(g.groups * g.o_rank // 128, 128, gw // 128, 128)
    scales = (np.abs(wf).max(axis=(1, 3)) / 448.0).astype(np.float32)
    codes = orc.e4m3_encode((wf / scales[:, None, :, None]).astype(np.float32)).reshape(g.groups * g.o_rank, gw)
    w = dict(w)
    w["wo_a"] = orc.dequant_fp8_blocks(codes, scales)
    role = dict(ratio=wl.ratio, is_index_source=1, uses_candidates=1)
    ctx = csa.Context(gd)
    outs = []
    for fp8 in (True, False):
        wd = _dev_weights(w)
        if fp8:
            wd["wo_a"] = None
            wd["wo_a_fp8"] = to_dev(codes)
            wd["wo_a_scale"] = to_dev(scales)
        sel_d = torch.full((B * T, K), -7, dtype=torch.int32, device="cuda")
        sh = csa.Shared(to_dev(shared["compress_kv"]), to_dev(shared["index_k"]), shared["compress_len"], sel_d, K,
                        to_dev(shared["candidates"]))
        outs.append(ctx.forward(wd, role, to_dev(ring0), to_dev(x), start, shared=sh))
    torch.cuda.synchronize()
    assert ctx.status() == 0
    assert torch.equal(outs[0], outs[1]), "fp8 wo_a changes the layer output"
    got = to_np(outs[0]).reshape(-1, g.dim)
    for b in (0, 31):
        sh_o = dict(compress_kv=shared["compress_kv"][b:b + 1], index_k=shared["index_k"][b:b + 1],
                    compress_len=shared["compress_len"], topk_idxs=np.full((T, K), -7, np.int32),
                    candidates=shared["candidates"][b * T:(b + 1) * T])
        res = orc.attn_forward(gd, role, w, ring0[b:b + 1].copy(), x[b:b + 1], start, tab, sh_o)
        assert_close_bf16(got[b * T:(b + 1) * T], res["out"].reshape(-1, g.dim), what="fp8 wo_a layer out")


@pytest.mark.parametrize("B,keep", [(2, 256), (64, 64), (5, 100), (3, 7)])
def test_cluster_gather_topk_selection(csa, orc, B, keep):
    """Long decode rows under a candidate mask (16384 latent keys at p = 65535, ratio 4, blocks of 64)
    take the gathered scores and the top-k in one launch, a thread-block cluster selecting together.
    Its published selection must equal, bit for bit, the two-kernel path's (debug scores requested)
    and the oracle's top-k of those very scores -- from a mask keeping every block (the most keys a
    cluster holds) down to one keeping fewer keys than K."""
    g = Geometry(dim=128, n_heads=4, head_dim=64, rope_dim=16, q_rank=64, o_rank=32, groups=2, window=8,
                 index_heads=32, index_hd=128, index_topk=512, cand_block=64, max_seq=65536, max_tokens=1,
                 max_batch=B)
    gd = g.as_dict()
    T, start, L = 1, 65535, 16384
    w = weights(g, with_indexer=True, norm_ones=False, seed_base=1400)
    x = activations(g, B, T, seed_base=2500 + B)
    Z, KI = latent_cache(g, B, L, seed_base=3400)
    pos = positions(B, T, start)
    cm = candidate_mask(B * T, pos, 4, L, g.cand_block, L // g.cand_block, keep, 99 + B)
    ring0 = orc.act_quant(ring_rows(g, B))[0]
    role = dict(ratio=4, is_index_source=1, uses_candidates=1)
    ctx = csa.Context(gd)
    wd = _dev_weights(w)
    K = g.index_topk
    sel_d = torch.full((B * T, K), -7, dtype=torch.int32, device="cuda")
    sh = csa.Shared(to_dev(Z), to_dev(KI), L, sel_d, K, to_dev(cm))
    ctx.forward(wd, role, to_dev(ring0), to_dev(x), start, shared=sh)
    sel_fast = sel_d.clone()
    dbg = _dbg(B * T, g, L, g.window + K)
    ctx.forward(wd, role, to_dev(ring0), to_dev(x), start, shared=sh, debug=dbg)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    assert torch.equal(sel_fast, sel_d), "the cluster path changes the selection"
    S = to_np(dbg["scores"])[:, :L].astype(np.float32)
    S = np.where(np.isnan(S), -np.inf, S).astype(np.float32)
    want = orc.index_topk(S, K, pos, 4, L, cm, g.cand_block, offset=g.window)
    assert_same_selection(to_np(sel_fast), want)
    ctx.close()


def test_stage_tracing_eager(csa, orc):
    """Per-stage tracing outside a graph capture: each forward lists its stages (mode 1), or appends to
    one list over several forwards (mode 2), with positive times; the output is unchanged by tracing."""
    g = _small_geom()
    w = weights(g, with_indexer=False)
    x = activations(g, 1, 4)
    ctx = csa.Context(g.as_dict())
    wd = _dev_weights(w)
    ring = torch.zeros((1, g.window, g.head_dim), dtype=torch.bfloat16, device="cuda")
    ref = ctx.forward(wd, dict(ratio=0), ring.clone(), to_dev(x), 0)
    ctx.trace(True)
    out = ctx.forward(wd, dict(ratio=0), ring.clone(), to_dev(x), 0)
    st = ctx.trace_read()
    names = [n for n, _ in st]
    assert "proj x" in names and "sparse_attn" in names and "wo_b" in names
    assert all(ms > 0 for _, ms in st)
    assert torch.equal(out, ref)
    ctx.trace(True, append=True)
    for _ in range(3):
        ctx.forward(wd, dict(ratio=0), ring.clone(), to_dev(x), 0)
    assert len(ctx.trace_read()) == 3 * len(st)
    ctx.trace(False)
    assert ctx.status() == 0
    ctx.close()
