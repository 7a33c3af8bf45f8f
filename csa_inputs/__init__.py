"""Seeded synthetic inputs for the compressed sparse attention layer core.

This module holds random-number draws and workload shapes only -- none of the method's arithmetic.
Both the CPU oracle (tests) and the GPU library (tests, benchmark) consume what it makes, so the
two sides always see bit-identical inputs.  Every tensor is drawn from its own ``torch.Generator``
seeded with ``seed_base + tensor_id``; bf16 tensors are returned as ``uint16`` numpy arrays of
their bit patterns (torch's float32 -> bfloat16 cast of the draw).

Distributions (the pages publish no data; these stand in for it):
  * x ~ N(0, 1) bf16 [B, T, dim]
  * projection weights ~ N(0, 1/in) bf16, [out, in] row-major
  * sink ~ N(0, 1) f32 [H]; q_norm, kv_norm = 1 (or bf16-valued 1 + 0.1 N(0,1) stored f32)
  * latent cache Z ~ N(0, 1) bf16 [B, L, hd]; index keys K^I ~ N(0, 1) bf16 [B, L, dI]
  * window ring rows ~ N(0, 1) bf16 [B, W, hd] (callers pass them through the fp8 round trip)
  * candidate block mask: per query, of the causal blocks of cand_block positions, a seeded
    permutation keeps exactly ``keep`` of them (a fraction or a count).
  * a kv source's compressor: kv and gate ~ N(0, 1/dim) f32 [hd, dim] (bf16 kv at ratio 1), index-key
    projection ~ N(0, 1/hd) bf16 [index_hd, hd]; norms as above.
"""
from dataclasses import dataclass, field, asdict
import math

import numpy as np
import torch


@dataclass
class Geometry:
    dim: int = 5120
    n_heads: int = 64
    head_dim: int = 512
    rope_dim: int = 64
    q_rank: int = 1280
    o_rank: int = 1024
    groups: int = 8
    window: int = 128
    eps: float = 1e-6
    index_heads: int = 32
    index_hd: int = 128
    index_topk: int = 512
    cand_block: int = 64
    cand_topk_blocks: int = 2048
    max_seq: int = 2048
    max_tokens: int = 64
    max_batch: int = 32
    rope_theta: float = 10000.0
    compress_rope_theta: float = 160000.0
    rope_factor: float = 16.0
    orig_seq: int = 65536
    beta_fast: float = 32.0
    beta_slow: float = 1.0

    def as_dict(self):
        return asdict(self)


@dataclass
class Workload:
    name: str
    geom: Geometry
    batch: int
    tokens: int          # T, tokens per call for each sequence
    start_pos: int
    ratio: int           # 0: window only
    is_index_source: bool = False
    uses_candidates: bool = False
    compress_len: int = 0  # latent rows published by the kv source
    cand_keep: float = 0.0  # fraction (< 1) or count (>= 1) of causal blocks kept per query
    layers: int = 1      # layers per step sharing one cache (reuse/Reindex chain)
    note: str = ""
    extra: dict = field(default_factory=dict)


def _full(**kw):
    g = Geometry()
    for k, v in kw.items():
        setattr(g, k, v)
    return g


WORKLOADS = {
    # tiny ratio-0 layer: prefill 12 at 0, then decode 12 and 13 through one ring
    "tiny_ratio0": Workload(
        "tiny_ratio0",
        _full(dim=256, n_heads=4, head_dim=64, rope_dim=16, q_rank=64, groups=2, o_rank=32, window=8,
              index_heads=4, index_hd=32, index_topk=16, cand_block=4, max_seq=64, max_tokens=16, max_batch=1),
        batch=1, tokens=12, start_pos=0, ratio=0, note="prefill 12 tokens at 0, then decode 12 and 13"),
    # full-width ratio-0 decode: batch 32 at context 1000, ring full
    "ratio0_decode": Workload(
        "ratio0_decode", _full(max_seq=1024, max_tokens=1, max_batch=32), batch=32, tokens=1, start_pos=1000,
        ratio=0),
    # Reindex compressed decode, ratio 2: 500 latent rows, index source, causal block mask keeping 50%
    "reindex_decode_r2": Workload(
        "reindex_decode_r2", _full(max_seq=1024, max_tokens=1, max_batch=32), batch=32, tokens=1, start_pos=1000,
        ratio=2, is_index_source=True, uses_candidates=True, compress_len=500, cand_keep=0.5),
    # compressed prefill chunk, ratio 4: 4096 tokens at 0, 1024 latent rows, no mask
    "prefill_r4": Workload(
        "prefill_r4", _full(max_seq=4096, max_tokens=4096, max_batch=1), batch=1, tokens=4096, start_pos=0, ratio=4,
        is_index_source=True, uses_candidates=False, compress_len=1024),
    # long-context compressed decode, ratio 4: 16384 latent rows, mask keeping 64 blocks, 4 Reindex layers
    "longctx_decode_r4": Workload(
        "longctx_decode_r4", _full(max_seq=65536, max_tokens=1, max_batch=64), batch=64, tokens=1,
        start_pos=65535, ratio=4, is_index_source=True, uses_candidates=True, compress_len=16384, cand_keep=64,
        layers=4),
}


def _gen(seed):
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, std, seed):
    """N(0, std^2) drawn in float32, cast to bf16; returned as uint16 bit patterns."""
    t = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * float(std)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def fp8_weight(shape, seed, block=128):
    """Random e4m3 weight storage: codes uint8 [N, K] drawn uniformly from the finite e4m3 codes (every
    byte but 0x7f and 0xff, the NaNs) and one positive f32 scale per block x block tile, 2^u with u
    uniform in [-12, -4).  Only random data: the dequantisation is the oracle's."""
    N, K = shape
    gen = _gen(seed)
    codes = torch.randint(0, 254, (N, K), generator=gen, dtype=torch.int32)
    codes = codes + (codes >= 0x7f).to(torch.int32)  # skip 0x7f; 0xff is above the drawn range
    u = torch.rand(-(-N // block), -(-K // block), generator=gen, dtype=torch.float64) * 8.0 - 12.0
    scales = torch.exp2(u).to(torch.float32)
    return codes.to(torch.uint8).numpy().copy(), scales.numpy().copy()


def f32_normal(shape, std, seed):
    return (torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * float(std)).numpy().copy()


# tensor ids for the seeds
_IDS = dict(x=1, wq_a=2, wq_b=3, wkv=4, wo_a=5, wo_b=6, idx_wq_b=7, idx_wproj=8, sink=9, q_norm=10, kv_norm=11,
            compress_kv=12, index_k=13, ring=14, cand=15, comp_wkv=16, comp_wgate=17, comp_norm=18, idx_wk=19,
            idx_k_norm=20)


def compressor_weights(g, ratio, seed_base=1000, with_index_keys=True, norm_ones=False):
    """A kv source's compressor weights: comp_wkv ~ N(0, 1/dim) [hd, dim] (f32 at ratio > 1, bf16 bits
    at ratio 1), comp_wgate ~ N(0, 1/dim) f32 (ratio > 1), comp_norm, and the index-key projection
    idx_wk ~ N(0, 1/hd) bf16 [index_hd, hd] with idx_k_norm.  Norm weights are 1, or bf16-valued
    1 + 0.1 N(0, 1) stored f32."""
    hd, dim = g.head_dim, g.dim
    w = {}
    if ratio > 1:
        w["comp_wkv"] = f32_normal((hd, dim), 1.0 / math.sqrt(dim), seed_base + _IDS["comp_wkv"])
        w["comp_wgate"] = f32_normal((hd, dim), 1.0 / math.sqrt(dim), seed_base + _IDS["comp_wgate"])
    else:
        w["comp_wkv"] = bf16_normal((hd, dim), 1.0 / math.sqrt(dim), seed_base + _IDS["comp_wkv"])

    def norm(name, n):
        if norm_ones:
            return np.ones(n, np.float32)
        t = 1.0 + 0.1 * torch.randn(n, generator=_gen(seed_base + _IDS[name]))
        return t.to(torch.bfloat16).to(torch.float32).numpy().copy()

    w["comp_norm"] = norm("comp_norm", hd)
    if with_index_keys:
        w["idx_wk"] = bf16_normal((g.index_hd, hd), 1.0 / math.sqrt(hd), seed_base + _IDS["idx_wk"])
        w["idx_k_norm"] = norm("idx_k_norm", g.index_hd)
    return w


def weights(g: Geometry, with_indexer=True, seed_base=1000, norm_ones=True):
    """Projection weights [out, in] ~ N(0, 1/in) bf16, sink ~ N(0,1) f32, norm weights."""
    H, hd, G = g.n_heads, g.head_dim, g.groups
    gw = H * hd // G

    def lin(name, out, inp):
        return bf16_normal((out, inp), 1.0 / math.sqrt(inp), seed_base + _IDS[name])

    w = dict(
        wq_a=lin("wq_a", g.q_rank, g.dim),
        wq_b=lin("wq_b", H * hd, g.q_rank),
        wkv=lin("wkv", hd, g.dim),
        wo_a=lin("wo_a", G * g.o_rank, gw),
        wo_b=lin("wo_b", g.dim, G * g.o_rank),
        sink=f32_normal((H,), 1.0, seed_base + _IDS["sink"]),
    )
    if norm_ones:
        w["q_norm"] = np.ones(g.q_rank, np.float32)
        w["kv_norm"] = np.ones(hd, np.float32)
    else:
        for name, n in (("q_norm", g.q_rank), ("kv_norm", hd)):
            t = 1.0 + 0.1 * torch.randn(n, generator=_gen(seed_base + _IDS[name]))
            w[name] = t.to(torch.bfloat16).to(torch.float32).numpy().copy()
    if with_indexer:
        w["idx_wq_b"] = lin("idx_wq_b", g.index_heads * g.index_hd, g.q_rank)
        w["idx_wproj"] = lin("idx_wproj", g.index_heads, g.dim)
    return w


def activations(g: Geometry, B, T, seed_base=1000):
    return bf16_normal((B, T, g.dim), 1.0, seed_base + _IDS["x"])


def ring_rows(g: Geometry, B, seed_base=1000):
    """Raw rows for a pre-filled ring [B, W, hd]; the caller rounds them through fp8."""
    return bf16_normal((B, g.window, g.head_dim), 1.0, seed_base + _IDS["ring"])


def latent_cache(g: Geometry, B, L, seed_base=1000):
    return (bf16_normal((B, L, g.head_dim), 1.0, seed_base + _IDS["compress_kv"]),
            bf16_normal((B, L, g.index_hd), 1.0, seed_base + _IDS["index_k"]))


def candidate_mask(n_queries, positions, ratio, compress_len, cand_block, width, keep, seed):
    """uint8 [n_queries, width]: for each query the causal blocks (those holding a valid compressed
    position j < min(floor((pos+1)/ratio), compress_len)) are permuted with a seeded generator and the
    first ``keep`` of them (a count, or a fraction rounded up) are set.  Non-causal blocks stay 0."""
    gen = _gen(seed)
    m = np.zeros((n_queries, width), np.uint8)
    for t in range(n_queries):
        limit = min((int(positions[t]) + 1) // ratio, compress_len) if ratio > 0 else 0
        nb = -(-limit // cand_block)
        if nb == 0:
            continue
        k = int(keep) if keep >= 1 else int(math.ceil(nb * keep))
        k = min(k, nb)
        perm = torch.randperm(nb, generator=gen).numpy()
        m[t, perm[:k]] = 1
    return m


def positions(B, T, start_pos):
    return np.array([start_pos + (r % T) for r in range(B * T)], np.int32)
