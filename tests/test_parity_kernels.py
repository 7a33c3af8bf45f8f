"""GPU parity of each step against the CPU oracle, through the C ABI.

Bit-exact where the pages make the result an integer or an exactly-rounded value fed identical
inputs: the fp8 codes, scales and values, the RoPE rotation, the ring slots, the window indices and
the top-k index sets.  Tolerances elsewhere: bf16 outputs atol/rtol 2e-2 (plus a relative error norm),
f32 indexer scores rtol 1e-3 with atol 1e-3 * max|S_row|.
"""
import math

import numpy as np
import pytest
import torch

from csa_inputs import WORKLOADS, Geometry, candidate_mask, latent_cache, positions, weights
from _helpers import assert_close_bf16, assert_same_selection, bf, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    import compressed_sparse_attention_attn_gb300 as m
    m.lib()
    return m


def _rng_bf16(orc, rng, shape, scale=1.0):
    return orc.f32_to_bf16((rng.standard_normal(shape) * scale).astype(np.float32))


def _ctx(csa, **kw):
    g = Geometry(**kw)
    return csa.Context(g.as_dict()), g


# ---------------------------------------------------------------------------------- fp8, RoPE

def test_act_quant_bit_exact(csa, orc):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 512)) * 10.0 ** rng.integers(-8, 8, (300, 1))).astype(np.float32)
    x[7, 32:64] = 0.0
    x[9, :32] = 448.0 * np.sign(rng.standard_normal(32))
    xb = orc.f32_to_bf16(x)
    want, codes, se = orc.act_quant(xb)
    xd = to_dev(xb)
    cd = torch.empty(xd.shape, dtype=torch.uint8, device="cuda")
    sd = torch.empty((300, 16), dtype=torch.int8, device="cuda")
    csa.act_quant(xd, cd, sd)
    assert np.array_equal(to_np(xd), want)
    assert np.array_equal(to_np(cd), codes)
    assert np.array_equal(to_np(sd), se)


@pytest.mark.parametrize("rd,hd,inverse", [(64, 512, False), (64, 512, True), (16, 64, False)])
def test_rope_bit_exact(csa, orc, rd, hd, inverse):
    rng = np.random.default_rng(2)
    rows, rpp = 96, 4
    x = _rng_bf16(orc, rng, (rows, hd))
    tab = orc.rope_table(rd, 2048, 10000.0)
    pos = rng.integers(0, 2048, rows // rpp).astype(np.int32)
    want = orc.apply_rotary(x, rd, pos, tab, inverse=inverse, rows_per_pos=rpp)
    xd = to_dev(x)
    csa.rope(xd, rd, to_dev(pos), to_dev(tab), inverse=inverse, rows_per_pos=rpp)
    assert np.array_equal(to_np(xd), want)


def test_rope_rounds_each_product(csa, orc):
    """A pair where rounding each product to f32 on its own and a fused multiply-add part at bf16:
    a = b = 1 + 2^-7, (c, s) = (1 + 2^-23, 1) gives re = 2^-23 exactly (0x3400), 2^-23 (1 + 2^-7) with
    the 2^-30 of a c kept."""
    rng = np.random.default_rng(12)
    rd, hd, rows = 16, 64, 4
    x = _rng_bf16(orc, rng, (rows, hd))
    x[:, hd - rd:hd - rd + 2] = orc.f32_to_bf16(np.full((rows, 2), 1 + 2.0 ** -7, np.float32))
    tab = np.zeros((1, rd // 2, 2), np.float32)
    tab[0, :, 0] = 1.0
    tab[0, 0] = (1 + 2.0 ** -23, 1.0)
    pos = np.zeros(rows, np.int32)
    want = orc.apply_rotary(x, rd, pos, tab)
    assert (want[:, hd - rd] == 0x3400).all()
    xd = to_dev(x)
    csa.rope(xd, rd, to_dev(pos), to_dev(tab))
    assert np.array_equal(to_np(xd), want)


def test_rope_tables_match_oracle(csa, orc):
    for g in (WORKLOADS["tiny_ratio0"].geom, Geometry(max_seq=70000, max_tokens=1, max_batch=1)):
        ctx = csa.Context(g.as_dict())
        plain = ctx.rope_table(0).numpy()
        comp = ctx.rope_table(1).numpy()
        want_p = orc.rope_table(g.rope_dim, g.max_seq, g.rope_theta)
        want_c = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta, g.orig_seq, g.rope_factor, g.beta_fast,
                                g.beta_slow)
        for a, b in ((plain, want_p), (comp, want_c)):
            ulp = np.abs(a.view(np.int32).astype(np.int64) - b.view(np.int32).astype(np.int64))
            close = np.abs(a - b) <= 1.2e-7
            assert ((ulp <= 1) | close).all()
        ctx.close()


# ---------------------------------------------------------------------------------- window rows

@pytest.mark.parametrize("hd,rd,W,T,start", [(64, 16, 8, 12, 0), (64, 16, 8, 1, 12), (64, 16, 8, 1, 13),
                                             (512, 64, 128, 200, 0), (512, 64, 128, 1, 1000), (512, 64, 128, 1, 5)])
def test_kv_finish_bit_exact(csa, orc, hd, rd, W, T, start):
    rng = np.random.default_rng(3 + T + start)
    B = 3
    kvn = _rng_bf16(orc, rng, (B * T, hd))
    tab = orc.rope_table(rd, 2048, 160000.0)
    ring0 = orc.act_quant(_rng_bf16(orc, rng, (B, W, hd)))[0]
    pos = positions(B, T, start)
    rot = orc.apply_rotary(kvn, rd, pos, tab)
    want_kv, want_codes, want_se = orc.act_quant(rot)
    want_ring = ring0.copy()
    for b in range(B):
        orc.ring_write(want_ring[b], want_kv[b * T:(b + 1) * T], start)
    if start == 0:
        want_idx = np.tile(orc.window_idx_prefill(T, W), (B, 1))
    else:
        want_idx = np.tile(orc.window_idx_decode(start, W)[None], (B, 1))
    ring = to_dev(ring0)
    kv_out = torch.empty((B * T, hd), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((B * T, W + 5), -9, dtype=torch.int32, device="cuda")
    codes = torch.empty((B * T, hd), dtype=torch.uint8, device="cuda")
    se = torch.empty((B * T, hd // 32), dtype=torch.int8, device="cuda")
    csa.kv_finish(to_dev(kvn), kv_out, B, T, start, rd, to_dev(tab), ring, idx, codes, se)
    assert np.array_equal(to_np(kv_out), want_kv)
    assert np.array_equal(to_np(codes), want_codes) and np.array_equal(to_np(se), want_se)
    assert np.array_equal(to_np(ring), want_ring)
    got_idx = to_np(idx)
    assert np.array_equal(got_idx[:, :W], want_idx) and (got_idx[:, W:] == -9).all()


# ---------------------------------------------------------------------------------- projections

@pytest.mark.parametrize("M,K,N,groups", [(12, 256, 64, 1), (32, 5120, 1280, 1), (33, 1280, 4096, 1),
                                          (32, 4096, 1024, 8), (200, 512, 96, 2), (1, 64, 32, 1),
                                          # many token tiles, activations that fit in L2: Stream-K
                                          (600, 512, 8192, 1), (520, 256, 1024, 8), (1030, 320, 4096, 2),
                                          # one token tile: a grid of whole tiles (144 x 1 tile, no fixup)
                                          (32, 1280, 18432, 1)])
def test_linear(csa, orc, M, K, N, groups):
    rng = np.random.default_rng(4 + M + N)
    x = _rng_bf16(orc, rng, (M, K * groups))
    W = _rng_bf16(orc, rng, (N * groups, K), 1.0 / math.sqrt(K))
    want = np.concatenate([orc.linear_bf16(x[:, g * K:(g + 1) * K], W[g * N:(g + 1) * N]) for g in range(groups)], 1)
    ctx, _ = _ctx(csa, dim=64, max_tokens=1, max_batch=1, max_seq=16)
    got = ctx.linear(to_dev(x), to_dev(W), groups=groups)
    assert_close_bf16(to_np(got), want, what="linear")
    # f32 accumulation (error at most K u sum|x W|, u = 2^-24) then one bf16 rounding (2^-8 relative)
    g, w = bf(to_np(got)).astype(np.float64), bf(want).astype(np.float64)
    xa, wa = np.abs(bf(x).astype(np.float64)), np.abs(bf(W).astype(np.float64))
    absdot = np.concatenate([xa[:, gi * K:(gi + 1) * K] @ wa[gi * N:(gi + 1) * N].T for gi in range(groups)], 1)
    assert (np.abs(g - w) <= np.abs(w) * 2 ** -7 + K * 2.0 ** -24 * absdot * 2 + 1e-30).all()


@pytest.mark.parametrize("M,K,N,groups", [(7680, 1024, 128, 8), (6200, 2048, 256, 8)])
def test_linear_waves(csa, orc, M, K, N, groups):
    """Activations above 96 MiB with many token tiles: whole tiles in waves, then Stream-K over the
    last partial wave.  The oracle computes sampled rows (every token tile, its edges and the ragged
    last one), all columns."""
    rng = np.random.default_rng(40 + M)
    x = _rng_bf16(orc, rng, (M, K * groups))
    W = _rng_bf16(orc, rng, (N * groups, K), 1.0 / math.sqrt(K))
    ctx, _ = _ctx(csa, dim=64, max_tokens=1, max_batch=1, max_seq=16)
    got = to_np(ctx.linear(to_dev(x), to_dev(W), groups=groups))
    rows = sorted(set([0, 1, 255, 256, 257, M - 1, M - 2] + list(range(100, M, 256)) +
                      list(rng.integers(0, M, 24))))
    want = np.concatenate([orc.linear_bf16(x[rows, g * K:(g + 1) * K], W[g * N:(g + 1) * N]) for g in range(groups)], 1)
    assert_close_bf16(got[rows], want, what="linear (waves)")


@pytest.mark.parametrize("M,K,N,groups", [(2100, 1280, 4096, 1), (3000, 640, 1024, 2), (2048, 96, 256, 1),
                                          (2304, 5120, 1280, 1), (4096, 1024, 1280, 1), (4096, 8192, 5120, 1)])
def test_linear_pairs(csa, orc, M, K, N, groups):
    """Many token tiles and an even number of weight tiles: clusters of two CTAs on adjacent weight
    tiles, each copying half of the shared token tile into both.  Ragged last token tile, a k-range
    that is not a whole number of 64-wide slices, two groups; more pair tiles than a wave of clusters
    (4096 x 1280: 80 pair tiles, the last four split by k-range and summed by a second kernel).  The
    oracle computes sampled rows (every token tile's edges and the ragged last one), all columns."""
    rng = np.random.default_rng(50 + M + N)
    x = _rng_bf16(orc, rng, (M, K * groups))
    W = _rng_bf16(orc, rng, (N * groups, K), 1.0 / math.sqrt(K))
    ctx, _ = _ctx(csa, dim=64, max_tokens=1, max_batch=1, max_seq=16)
    got = to_np(ctx.linear(to_dev(x), to_dev(W), groups=groups))
    assert ctx.status() == 0
    rows = sorted(set([0, 1, 127, 128, 255, 256, M - 1, M - 2] + list(range(130, M, 256)) +
                      list(rng.integers(0, M, 16)) + list(rng.integers(max(0, M - 1024), M, 8))))
    want = np.concatenate([orc.linear_bf16(x[rows, g * K:(g + 1) * K], W[g * N:(g + 1) * N]) for g in range(groups)], 1)
    assert_close_bf16(got[rows], want, what="linear (pairs)")


@pytest.mark.parametrize("M,K,N,groups", [(32, 4096, 1024, 8), (1, 4096, 1024, 8), (7, 256, 200, 1),
                                           (33, 1280, 384, 1), (20, 5120, 1280, 1), (5, 1040, 136, 1),
                                           (6200, 1024, 128, 8)])
def test_linear_fp8w(csa, orc, M, K, N, groups):
    """Projection with e4m3 weights and one f32 scale per 128 x 128 tile (the fp8 grouped wo_a): the
    oracle's linear_bf16 on the oracle's dequantised weights, within the linear tolerance, and against
    the bf16 product on those weights.  The kernel expands each tile to exactly those weights, so the
    two launches differ only where they split a tile's k-range at other points (an fp8 unit is 128
    wide, a bf16 one 64) and add the f32 partial sums in another order: at most one bf16 step of the
    result plus twice the f32 summation bound, 2 K 2^-24 sum_k |x_k w_k| (each product is exact in
    f32).  The grouped decode shapes of the layer's wo_a split at the same points and must agree bit
    for bit.  Ragged N and token tiles; the last case is a prefill-sized grouped launch (whole-tile
    waves, 128-token tiles), checked on sampled rows."""
    from csa_inputs import fp8_weight
    rng = np.random.default_rng(60 + M + N)
    x = _rng_bf16(orc, rng, (M, K * groups))
    codes, scales = fp8_weight((N * groups, K), 4000 + N)
    W = orc.dequant_fp8_blocks(codes, scales)
    ctx, _ = _ctx(csa, dim=64, max_tokens=1, max_batch=1, max_seq=16)
    xd = to_dev(x)
    got = to_np(ctx.linear_fp8w(xd, to_dev(codes), to_dev(scales), groups=groups))
    ref = to_np(ctx.linear(xd, to_dev(W), groups=groups))
    rows = np.arange(M) if M < 512 else np.array(sorted(set([0, 1, 255, 256, M - 1] + list(rng.integers(0, M, 12)))))
    want = np.concatenate([orc.linear_bf16(x[rows, g * K:(g + 1) * K], W[g * N:(g + 1) * N]) for g in range(groups)], 1)
    assert_close_bf16(got[rows], want, what="linear_fp8w")
    if groups == 8 and M <= 32:
        assert np.array_equal(got, ref), "fp8-weight product differs from the bf16 product on the dequantised weights"
    xa, wa = np.abs(bf(x[rows]).astype(np.float64)), np.abs(bf(W).astype(np.float64))
    s_abs = np.concatenate([xa[:, g * K:(g + 1) * K] @ wa[g * N:(g + 1) * N].T for g in range(groups)], 1)
    g64, r64 = bf(got[rows]).astype(np.float64), bf(ref[rows]).astype(np.float64)
    big = np.maximum(np.abs(g64), np.abs(r64))
    ulp = np.where(big > 0, np.exp2(np.floor(np.log2(np.where(big > 0, big, 1.0))) - 7), 0.0)
    bound = ulp + 2.0 * K * 2.0 ** -24 * s_abs
    assert (np.abs(g64 - r64) <= bound).all(), "fp8-weight product beyond the reordering bound of the bf16 product"
    assert ctx.status() == 0


def test_rmsnorm(csa, orc):
    rng = np.random.default_rng(5)
    x = _rng_bf16(orc, rng, (40, 1280), 3.0)
    w = (1 + 0.1 * rng.standard_normal(1280)).astype(np.float32)
    want = orc.rmsnorm(x, w, 1e-6)
    got = csa.rmsnorm(to_dev(x), to_dev(w), 1e-6)
    g, ww = bf(to_np(got)).astype(np.float64), bf(want).astype(np.float64)
    assert (np.abs(g - ww) <= np.abs(ww) * 2 ** -7 + 1e-30).all()


# ---------------------------------------------------------------------------------- indexer

def _index_case(orc, rng, B, T, start, Hi, dI, L, compress_len, ratio, cand_keep, cand_block):
    qI = _rng_bf16(orc, rng, (B * T, Hi, dI))
    wI = (rng.standard_normal((B * T, Hi)) / 64).astype(np.float32)
    KI = _rng_bf16(orc, rng, (B, L, dI))
    pos = positions(B, T, start)
    cand = None
    if cand_keep:
        cand = candidate_mask(B * T, pos, ratio, compress_len, cand_block, -(-L // cand_block), cand_keep, 77)
    S = np.concatenate([orc.index_scores(qI[b * T:(b + 1) * T], wI[b * T:(b + 1) * T], KI[b], pos[b * T:(b + 1) * T],
                                         ratio, compress_len, None if cand is None else cand[b * T:(b + 1) * T],
                                         cand_block) for b in range(B)])
    return qI, wI, KI, pos, cand, S


@pytest.mark.parametrize("B,T,start,L,clen,ratio,keep,cb", [
    (4, 1, 1000, 512, 500, 2, 0.5, 64),       # Reindex decode shape
    (1, 300, 0, 1024, 1024, 4, 0, 64),        # prefill, causal only
    (2, 1, 65535, 16384, 16384, 4, 64, 64),   # long context, 64 of 256 blocks
    (3, 1, 40, 64, 7, 1, 0, 8),               # short cache
])
def test_index_scores(csa, orc, B, T, start, L, clen, ratio, keep, cb):
    rng = np.random.default_rng(6 + T)
    qI, wI, KI, pos, cand, S = _index_case(orc, rng, B, T, start, 32, 128, L, clen, ratio, keep, cb)
    Sd = torch.full((B * T, L), float("nan"), device="cuda")
    csa.index_scores(to_dev(qI), to_dev(wI), to_dev(KI), B, T, start, clen, ratio, Sd,
                     None if cand is None else to_dev(cand), cb)
    got = to_np(Sd)
    valid = np.isfinite(S)
    assert np.isnan(got[~valid]).all()  # invalid positions are not written
    for r in range(B * T):
        v = valid[r]
        if not v.any():
            continue
        a, b = got[r, v].astype(np.float64), S[r, v].astype(np.float64)
        tol = 1e-3 * np.abs(b) + 1e-3 * np.abs(b).max()
        assert (np.abs(a - b) <= tol).all()


@pytest.mark.parametrize("Hi,B,T,start,L,clen,ratio,keep", [
    (64, 2, 7, 200, 256, 200, 2, 0), (16, 1, 20, 0, 300, 300, 1, 0),
    # many queries: Q^I resident, the key tiles looped over (ragged last group, a mask at prefill)
    (64, 2, 50, 600, 700, 700, 1, 0), (16, 1, 100, 300, 512, 400, 1, 0.5), (32, 1, 200, 800, 1024, 1000, 1, 0.3),
])
def test_index_scores_head_counts(csa, orc, Hi, B, T, start, L, clen, ratio, keep):
    """Other indexer head counts: the query groups of the tensor-core kernels hold 256 / Hi queries."""
    rng = np.random.default_rng(60 + Hi + T)
    qI, wI, KI, pos, cand, S = _index_case(orc, rng, B, T, start, Hi, 128, L, clen, ratio, keep, 64)
    Sd = torch.full((B * T, L), float("nan"), device="cuda")
    csa.index_scores(to_dev(qI), to_dev(wI), to_dev(KI), B, T, start, clen, ratio, Sd,
                     None if cand is None else to_dev(cand), 64)
    got = to_np(Sd)
    valid = np.isfinite(S)
    assert np.isnan(got[~valid]).all()
    tol = 1e-3 * np.abs(S[valid]) + 1e-3 * np.abs(S[valid]).max()
    assert (np.abs(got[valid].astype(np.float64) - S[valid]) <= tol).all()


@pytest.mark.parametrize("Hi,B,T,start,L,clen,ratio,keep", [
    (32, 1, 4096, 0, 1024, 1024, 4, 0),       # the prefill chunk: 512 groups of 8 queries
    (64, 2, 400, 100, 700, 650, 1, 0.5),      # 4-query groups, two sequences, a mask, ragged last tile
    (16, 1, 3000, 3, 1300, 1250, 2, 0),       # 16-query groups, ragged last group
])
def test_index_scores_many_groups(csa, orc, Hi, B, T, start, L, clen, ratio, keep):
    """More query groups than SMs: the persistent kernel that keeps a group's Q^I resident over its
    key tiles.  The oracle runs on sampled queries (first and last of every sequence, group edges,
    the ragged last group, random ones); every query's unwritten positions are checked."""
    rng = np.random.default_rng(120 + Hi + T)
    qI = _rng_bf16(orc, rng, (B * T, Hi, 128))
    wI = (rng.standard_normal((B * T, Hi)) / 64).astype(np.float32)
    KI = _rng_bf16(orc, rng, (B, L, 128))
    pos = positions(B, T, start)
    cand = None if not keep else candidate_mask(B * T, pos, ratio, clen, 64, -(-L // 64), keep, 79)
    Sd = torch.full((B * T, L), float("nan"), device="cuda")
    csa.index_scores(to_dev(qI), to_dev(wI), to_dev(KI), B, T, start, clen, ratio, Sd,
                     None if cand is None else to_dev(cand), 64)
    got = to_np(Sd)
    QG = 256 // Hi
    rows = set()
    for b in range(B):
        base = b * T
        rows.update([base, base + 1, base + T - 1, base + T - 2])
        rows.update(base + g * QG + d for g in (1, T // QG // 2, (T - 1) // QG) for d in (-1, 0, QG - 1) if 0 <= g * QG + d < T)
        rows.update(base + int(t) for t in rng.choice(T, 24, replace=False))
    rows = sorted(rows)
    for r in rows:
        b = r // T
        want = orc.index_scores(qI[r:r + 1], wI[r:r + 1], KI[b], pos[r:r + 1], ratio, clen,
                                None if cand is None else cand[r:r + 1], 64)[0]
        v = np.isfinite(want)
        assert np.isnan(got[r, ~v]).all()
        if v.any():
            a, w = got[r, v].astype(np.float64), want[v].astype(np.float64)
            assert (np.abs(a - w) <= 1e-3 * np.abs(w) + 1e-3 * np.abs(w).max()).all(), r
    # every query: the valid positions written, the others not
    t = np.arange(B * T) % T
    lim = np.minimum((start + t + 1) // ratio, clen)
    valid = np.arange(L)[None, :] < lim[:, None]
    if cand is not None:
        valid &= cand[:, np.arange(L) // 64] != 0
    assert np.isfinite(got[valid]).all() and np.isnan(got[~valid]).all()


@pytest.mark.parametrize("Hi,B,start,L,clen,ratio,keep,cb", [
    (32, 5, 4000, 2048, 2000, 2, 7, 64),        # odd number of kept units
    (32, 3, 3000, 2048, 1500, 2, 0.3, 128),     # blocks of two 64-key units, last one partial
    (64, 4, 20000, 8192, 5001, 4, 17, 64),      # 64 heads
    (16, 70, 8000, 4096, 2000, 4, 0.6, 64),     # many queries: a small CTA group per query
    (32, 2, 5000, 4096, 2500, 2, 1, 64),        # one kept block
    (32, 4, 1000, 512, 500, 2, 0.5, 64),        # short candidate span (the dense kernel)
])
def test_index_scores_gathered(csa, orc, Hi, B, start, L, clen, ratio, keep, cb):
    """One query per sequence with a candidate mask spanning more than 1024 keys: only the kept
    blocks' keys are read.  Row 0 of the mask keeps every causal block and row 1 (when there is one)
    none."""
    rng = np.random.default_rng(90 + Hi + B)
    T = 1
    qI = _rng_bf16(orc, rng, (B, Hi, 128))
    wI = (rng.standard_normal((B, Hi)) / 64).astype(np.float32)
    KI = _rng_bf16(orc, rng, (B, L, 128))
    pos = positions(B, T, start)
    width = -(-L // cb)
    cand = candidate_mask(B, pos, ratio, clen, cb, width, keep, 78)
    lim0 = min((start + 1) // ratio, clen)
    cand[0, :-(-lim0 // cb)] = 1
    if B > 1:
        cand[1, :] = 0
    S = np.concatenate([orc.index_scores(qI[b:b + 1], wI[b:b + 1], KI[b], pos[b:b + 1], ratio, clen,
                                         cand[b:b + 1], cb) for b in range(B)])
    Sd = torch.full((B, L), float("nan"), device="cuda")
    csa.index_scores(to_dev(qI), to_dev(wI), to_dev(KI), B, T, start, clen, ratio, Sd, to_dev(cand), cb)
    got = to_np(Sd)
    valid = np.isfinite(S)
    assert np.isnan(got[~valid]).all()
    for r in range(B):
        v = valid[r]
        if not v.any():
            continue
        a, b = got[r, v].astype(np.float64), S[r, v].astype(np.float64)
        tol = 1e-3 * np.abs(b) + 1e-3 * np.abs(b).max()
        assert (np.abs(a - b) <= tol).all()


@pytest.mark.parametrize("B,T,start,L,clen,ratio,keep,cb,K", [
    (4, 1, 1000, 512, 500, 2, 0.5, 64, 512),
    (1, 300, 0, 1024, 1024, 4, 0, 64, 512),
    (2, 1, 65535, 16384, 16384, 4, 64, 64, 512),
    (3, 1, 40, 64, 7, 1, 0, 8, 16),
    (1, 1, 65535, 16384, 16384, 4, 0, 64, 512),    # more valid positions than shared memory holds
    (1, 2, 8191, 4096, 4096, 2, 0, 64, 2048),      # K above the one-element-per-thread sort
    (1, 64, 4032, 1024, 1024, 4, 0, 64, 512),      # 1008..1024 valid, the selection a real cut
    (3, 1, 700, 512, 400, 2, 0.5, 64, 512),        # masked, fewer valid than K
    (1, 2, 100, 128, 128, 1, 0, 64, 600),          # K beyond the positions: -1 tail
    (2, 5, 250, 256, 256, 1, 0.25, 128, 64),       # blocks of 128, K below the valid count
    (1, 2, 8191, 4096, 4096, 2, 0, 64, 1000),      # a cut sorted over 1024 slots (three shared stages)
    (1, 1, 1300, 1024, 1024, 2, 0, 64, 700),       # 650 valid, all taken, sorted over 1024 slots
])
def test_index_topk_bit_exact(csa, orc, B, T, start, L, clen, ratio, keep, cb, K):
    rng = np.random.default_rng(7 + T)
    qI, wI, KI, pos, cand, S = _index_case(orc, rng, B, T, start, 32, 128, L, clen, ratio, keep, cb)
    S = np.where(np.isfinite(S), np.round(S * 4) / 4, S).astype(np.float32)  # many exact ties
    S[:, ::7] = np.where(np.isfinite(S[:, ::7]), -0.0, S[:, ::7])
    want = np.concatenate([orc.index_topk(S[b * T:(b + 1) * T], K, pos[b * T:(b + 1) * T], ratio, clen,
                                          None if cand is None else cand[b * T:(b + 1) * T], cb, offset=128)
                           for b in range(B)])
    out = torch.full((B * T, K), -5, dtype=torch.int32, device="cuda")
    csa.index_topk(to_dev(S), B, T, start, clen, ratio, K, out, offset=128,
                   cand=None if cand is None else to_dev(cand), cand_block=cb)
    assert_same_selection(to_np(out), want)


# ---------------------------------------------------------------------------------- attention

@pytest.mark.parametrize("H,hd,na,nb,a_len,b_len,B,T", [(4, 64, 8, 16, 12, 40, 1, 12), (64, 512, 128, 512, 128, 500, 3, 1),
                                                        (64, 512, 128, 512, 300, 1024, 1, 9),
                                                        (64, 512, 128, 512, 128, 700, 80, 1),
                                                        (64, 512, 7, 300, 7, 64, 2, 5),
                                                        (128, 512, 128, 256, 128, 300, 2, 1),
                                                        (64, 512, 64, 256, 64, 400, 2, 100),
                                                        # the widest list the tensor-core kernel takes: 6 tiles
                                                        (64, 512, 128, 640, 128, 900, 4, 1),
                                                        # more than two waves of queries
                                                        (64, 512, 128, 512, 128, 900, 2, 200),
                                                        (128, 512, 128, 256, 128, 300, 1, 200)])
def test_sparse_attn(csa, orc, H, hd, na, nb, a_len, b_len, B, T):
    rng = np.random.default_rng(8 + H)
    q = _rng_bf16(orc, rng, (B * T, H, hd))
    ra = _rng_bf16(orc, rng, (B, a_len, hd))
    rb = _rng_bf16(orc, rng, (B, b_len, hd))
    sink = rng.standard_normal(H).astype(np.float32)
    ia = rng.integers(-1, a_len, (B * T, na)).astype(np.int32)
    ib = np.where(rng.random((B * T, nb)) < 0.2, -1, rng.integers(0, b_len, (B * T, nb)) + a_len).astype(np.int32)
    ib[0, :] = -1
    ia[0, :] = -1  # a query with nothing selected: O = 0
    scale = 1 / math.sqrt(hd)
    rd, start = hd // 8, 0
    tab = orc.rope_table(rd, max(64, T), 10000.0)
    want = np.concatenate([orc.sparse_attn(q[b * T:(b + 1) * T], ra[b], rb[b],
                                           np.concatenate([ia[b * T:(b + 1) * T], ib[b * T:(b + 1) * T]], 1), sink, scale)
                           for b in range(B)])
    pos = positions(B, T, start)
    want_rot = orc.apply_rotary(want.reshape(-1, hd), rd, pos, tab, inverse=True, rows_per_pos=H).reshape(want.shape)
    ctx, _ = _ctx(csa, dim=64, max_tokens=1, max_batch=1, max_seq=16)
    o = torch.empty((B * T, H, hd), dtype=torch.bfloat16, device="cuda")
    o_rot = torch.empty_like(o)
    ctx.sparse_attn(to_dev(q), to_dev(ra), a_len, to_dev(ia), to_dev(sink), scale, rows_b=to_dev(rb), b_len=b_len,
                    idx_b=to_dev(ib), o=o, o_rot=o_rot, rd=rd, start_pos=start, tab=to_dev(tab), B=B, T=T)
    assert ctx.status() == 0
    got = to_np(o)
    assert (got[0] == 0).all()
    assert_close_bf16(got, want, what="sparse_attn")
    assert_close_bf16(to_np(o_rot), want_rot, what="sparse_attn o_rot")


@pytest.mark.parametrize("T,nb,b_len,keep", [(300, 512, 200, 0.8), (260, 256, 600, 0.5), (700, 512, 300, 0.6),
                                              (1000, 256, 900, 0.3)])
def test_sparse_attn_prefill_lists(csa, orc, T, nb, b_len, keep):
    """Prefill-shaped lists, one CTA a query over its whole list: the causal window of the chunk's own
    rows (its first entries -1 for early queries, so whole 64-entry halves are empty) and compressed
    entries with runs of -1 (some halves empty, some partial).  From a few hundred queries on, the
    queries run on the persistent kernel (a CTA an SM taking a sequence of them): there a query with
    nothing selected in the middle of a CTA's sequence writes zeros and the next one is unaffected."""
    rng = np.random.default_rng(31 + T)
    H, hd, W, B = 64, 512, 128, 1
    q = _rng_bf16(orc, rng, (T, H, hd))
    ra = _rng_bf16(orc, rng, (B, T, hd))
    rb = _rng_bf16(orc, rng, (B, b_len, hd))
    sink = rng.standard_normal(H).astype(np.float32)
    t = np.arange(T)[:, None]
    ia = (t - W + 1 + np.arange(W)[None, :]).astype(np.int32)
    ia[ia < 0] = -1
    ib = (rng.integers(0, b_len, (T, nb)) + T).astype(np.int32)
    ib[rng.random((T, nb)) > keep] = -1
    ib[:, 64:192] = -1            # two empty halves in the middle of the compressed part
    ib[5, :] = -1
    ia[7, :] = -1                 # a query with compressed rows only
    if T > 400:
        ia[T - 300, :] = -1       # nothing selected, between two queries of the same CTA
        ib[T - 300, :] = -1
    scale = 1 / math.sqrt(hd)
    rd = 64
    tab = orc.rope_table(rd, max(64, T), 10000.0)
    want = orc.sparse_attn(q, ra[0], rb[0], np.concatenate([ia, ib], 1), sink, scale)
    want_rot = orc.apply_rotary(want.reshape(-1, hd), rd, positions(B, T, 0), tab, inverse=True,
                                rows_per_pos=H).reshape(want.shape)
    ctx, _ = _ctx(csa, dim=64, max_tokens=1, max_batch=1, max_seq=16)
    o_rot = torch.empty((T, H, hd), dtype=torch.bfloat16, device="cuda")
    ctx.sparse_attn(to_dev(q), to_dev(ra), T, to_dev(ia), to_dev(sink), scale, rows_b=to_dev(rb), b_len=b_len,
                    idx_b=to_dev(ib), o_rot=o_rot, rd=rd, start_pos=0, tab=to_dev(tab), B=B, T=T)
    assert ctx.status() == 0
    got = to_np(o_rot)
    if T > 400:
        assert ((got[T - 300] & 0x7FFF) == 0).all()  # zeros (the inverse rotation may leave -0)
    assert_close_bf16(got, want_rot, what="sparse_attn o_rot (prefill lists)")
