"""CPU oracle of the compressed sparse attention layer core -- TEST INFRASTRUCTURE ONLY.

``csa_oracle.c`` restates, step by step and in plain scalar C, what the pages define (the
``deepseek_v41_ref::attn`` rustdoc page, the DeepSeek V4.1 "Compressed sparse attention" and
"Join rows" atlas pages, the ``metrale_model_arch::attn_v41`` docs).  This module builds it with
gcc and exposes it to numpy through ctypes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` leg and reference arm may import it; the GPU library never does, and the
two share no code.  bf16 tensors travel as ``uint16`` arrays of their bit patterns.
:func:`dequant_fp8_blocks` (fp8 weight storage back to bf16) composes the C primitives in numpy.

Parity unpinned: :func:`compress` (the kv source's compressor).  Its pooling formula is a reading
(the pages give the weights, state and caches only); tests/test_oracle_compress.py pins what
mathematics fixes, not agreement with the real model.

The YaRN form of :func:`rope_table` follows the published method (the pages give its constants
only).  Pinned are its classes (pairs with at least beta_fast turns over the original length keep
their frequency, those with at most beta_slow turns run at frequency / factor, the others lie strictly
between) and every pair's blend weight inside the ramp, against ramp ends found by searching the
rotation counts rather than from the closed-form index.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_SO = os.path.join(_HERE, "liborc_csa.so")
_lib = None

I64, I32, F32, F64 = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no fused multiply-add, OpenMP) next to its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
                               "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        L.orc_bf16_to_f32.restype = F32
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_bf16.argtypes = [F32]
        L.orc_pow2_ceil.restype = F32
        L.orc_pow2_ceil.argtypes = [F32]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [F32]
        L.orc_e4m3_decode.restype = F32
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        for n in ("orc_f32_to_bf16_n", "orc_pow2_ceil_n", "orc_e4m3_encode_n", "orc_e4m3_decode_n"):
            getattr(L, n).argtypes = [P, P, I64]
            getattr(L, n).restype = None
        L.orc_linear_bf16.argtypes = [P, I64, I64, I64, P, I64, I64, P, I64]
        L.orc_linear_bf16.restype = None
        L.orc_rmsnorm.argtypes = [P, I64, I64, P, F32, P]
        L.orc_rmsnorm.restype = None
        L.orc_rope_table.argtypes = [I32, I64, F64, I64, F64, F64, F64, P]
        L.orc_rope_table.restype = I32
        L.orc_apply_rotary.argtypes = [P, I64, I32, I32, P, I32, P, I64, I32]
        L.orc_apply_rotary.restype = I32
        L.orc_act_quant.argtypes = [P, I64, P, P]
        L.orc_act_quant.restype = I32
        L.orc_window_idx_prefill.argtypes = [I64, I32, P]
        L.orc_window_idx_prefill.restype = None
        L.orc_window_idx_decode.argtypes = [I64, I32, P]
        L.orc_window_idx_decode.restype = None
        L.orc_ring_write.argtypes = [P, I32, I32, P, I64, I64]
        L.orc_ring_write.restype = None
        L.orc_index_scores.argtypes = [P, P, P, I64, I32, I32, I64, P, I32, I64, P, I32, I32, P]
        L.orc_index_scores.restype = None
        L.orc_index_topk.argtypes = [P, I64, I64, I32, P, I32, I64, P, I32, I32, ctypes.c_int32, P]
        L.orc_index_topk.restype = None
        L.orc_sparse_attn.argtypes = [P, I64, I32, I32, P, I64, P, I64, P, I32, P, F64, P]
        L.orc_sparse_attn.restype = I32
        L.orc_attn_forward.argtypes = [P, P, P, P, P, I32, I64, I64, P, P, I64, P, P, P]
        L.orc_attn_forward.restype = I32
        L.orc_candidate_blocks.argtypes = [P, I64, I64, P, I32, I64, I32, I32, I32, P]
        L.orc_candidate_blocks.restype = None
        L.orc_compress.argtypes = [P, I32, P, P, P, P, I32, I64, I64, P, I64, P, P, I64, P, P]
        L.orc_compress.restype = I32
        L.orc_compress_state_init.argtypes = [P, P, I64]
        L.orc_compress_state_init.restype = None
        L.orc_param_counts.argtypes = [P, I32, P]
        L.orc_param_counts.restype = None
        L.orc_n_idx.argtypes = [P, P]
        L.orc_n_idx.restype = I32
        L.orc_num_threads.restype = I32
        L.orc_set_num_threads.argtypes = [I32]
        L.orc_set_num_threads.restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(P)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------------------------
# numeric primitives
# ---------------------------------------------------------------------------------------------

def bf16_to_f32(u16):
    """bf16 bit patterns -> float32 (the bits are the top half of a binary32)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def f32_to_bf16(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_n(_p(x), _p(y), x.size)
    return y


def pow2_ceil(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.float32)
    lib().orc_pow2_ceil_n(_p(x), _p(y), x.size)
    return y


def e4m3_encode(x):
    x = _c(x, np.float32)
    y = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_n(_p(x), _p(y), x.size)
    return y


def e4m3_decode(c):
    c = _c(c, np.uint8)
    y = np.empty(c.shape, np.float32)
    lib().orc_e4m3_decode_n(_p(c), _p(y), c.size)
    return y


# ---------------------------------------------------------------------------------------------
# steps
# ---------------------------------------------------------------------------------------------

def linear_bf16(x, W):
    """y = bf16(x @ W.T) with W [out, in]; x [..., in] bf16 bits."""
    x = _c(x, np.uint16)
    W = _c(W, np.uint16)
    K = x.shape[-1]
    assert W.shape[1] == K
    M = x.size // K
    N = W.shape[0]
    y = np.empty(x.shape[:-1] + (N,), np.uint16)
    lib().orc_linear_bf16(_p(x), M, K, K, _p(W), N, K, _p(y), N)
    return y


def dequant_fp8_blocks(codes, scales, block=128):
    """Projection weights stored as e4m3 codes uint8 [N, K] with one f32 scale per block x block tile
    (scales [ceil(N/block), ceil(K/block)]), back to bf16 as the converter does before the bf16
    projections ([atlas] Attention excerpt: the grouped output projection is dequantised to bf16, and
    an fp8 grouped GEMM would halve its memory): w = bf16(f32(e4m3(code) * scale)).  The product of a
    4-bit significand and an f32 is exact in double, so one rounding to f32 gives the f32 product.
    The tile layout is a reading (the published fp8 weight format of DeepSeek-V3: 128 x 128 tiles);
    the pages print none."""
    codes = _c(codes, np.uint8)
    N, K = codes.shape
    s = _c(scales, np.float32)
    assert s.shape == (-(-N // block), -(-K // block)), (s.shape, N, K, block)
    full = np.repeat(np.repeat(s, block, 0), block, 1)[:N, :K].astype(np.float64)
    v = e4m3_decode(codes).astype(np.float64) * full
    return f32_to_bf16(v.astype(np.float32))


def rmsnorm(x, w, eps):
    x = _c(x, np.uint16)
    w = _c(w, np.float32)
    N = x.shape[-1]
    y = np.empty_like(x)
    lib().orc_rmsnorm(_p(x), x.size // N, N, _p(w), eps, _p(y))
    return y


def rope_table(rd, max_seq, theta, orig_seq=0, factor=1.0, beta_fast=32.0, beta_slow=1.0):
    """[max_seq, rd/2, 2] float32 of (cos, sin); YaRN only when max_seq > orig_seq > 0."""
    t = np.empty((max_seq, rd // 2, 2), np.float32)
    rc = lib().orc_rope_table(rd, max_seq, theta, orig_seq, factor, beta_fast, beta_slow, _p(t))
    assert rc == 0, rc
    return t


def apply_rotary(x, rd, pos, table, inverse=False, rows_per_pos=1):
    """Rotate the last rd elements of each row of x [rows, row_len]; returns a new array."""
    y = np.array(x, dtype=np.uint16, copy=True, order="C")
    row_len = y.shape[-1]
    rows = y.size // row_len
    pos = _c(pos, np.int32)
    table = _c(table, np.float32)
    rc = lib().orc_apply_rotary(_p(y), rows, row_len, rd, _p(pos), rows_per_pos, _p(table), table.shape[0],
                                int(inverse))
    assert rc == 0, rc
    return y


def act_quant(x):
    """fp8 round trip per block of 32 along the flattened array: (values, codes, scale exponents)."""
    y = np.array(x, dtype=np.uint16, copy=True, order="C")
    codes = np.empty(y.shape, np.uint8)
    se = np.empty(y.shape[:-1] + (y.shape[-1] // 32,), np.int8)
    rc = lib().orc_act_quant(_p(y), y.size, _p(codes), _p(se))
    assert rc == 0, rc
    return y, codes, se


def window_idx_prefill(T, W):
    idx = np.empty((T, W), np.int32)
    lib().orc_window_idx_prefill(T, W, _p(idx))
    return idx


def window_idx_decode(p, W):
    idx = np.empty((W,), np.int32)
    lib().orc_window_idx_decode(p, W, _p(idx))
    return idx


def ring_write(ring, rows, start_pos):
    """Write rows [T, hd] into ring [W, hd] (in place) at positions start_pos.."""
    assert ring.flags.c_contiguous and ring.dtype == np.uint16
    rows = _c(rows, np.uint16)
    lib().orc_ring_write(_p(ring), ring.shape[0], ring.shape[1], _p(rows), rows.shape[0], start_pos)
    return ring


def _cand(cand):
    if cand is None:
        return None, 0
    cand = _c(cand, np.uint8)
    return cand, cand.shape[-1]


def index_scores(qI, wI, KI, pos, ratio, compress_len, cand=None, cand_block=1):
    """qI [n, Hi, dI], wI [n, Hi] f32, KI [Lc, dI] -> S [n, Lc] f32 (-inf where not valid)."""
    qI = _c(qI, np.uint16)
    wI = _c(wI, np.float32)
    KI = _c(KI, np.uint16)
    pos = _c(pos, np.int32)
    n, Hi, dI = qI.shape
    Lc = KI.shape[0]
    cand, cw = _cand(cand)
    S = np.empty((n, Lc), np.float32)
    lib().orc_index_scores(_p(qI), _p(wI), _p(KI), n, Hi, dI, Lc, _p(pos), ratio, compress_len, _p(cand), cw,
                           cand_block, _p(S))
    return S


def index_topk(S, K, pos, ratio, compress_len, cand=None, cand_block=1, offset=0):
    S = _c(S, np.float32)
    pos = _c(pos, np.int32)
    n, Lc = S.shape
    cand, cw = _cand(cand)
    out = np.empty((n, K), np.int32)
    lib().orc_index_topk(_p(S), n, Lc, K, _p(pos), ratio, compress_len, _p(cand), cw, cand_block, offset, _p(out))
    return out


def candidate_blocks(S, pos, ratio, compress_len, cand_block, cand_topk, cand_width):
    """The candidate source's block mask (see orc_candidate_blocks): per query, the cand_topk blocks
    of cand_block positions whose largest valid score is highest (ties to the lower block), as uint8
    [n, cand_width].  S [n, L] f32 (invalid entries ignored by position)."""
    S = _c(S, np.float32)
    n, L = S.shape
    pos = _c(pos, np.int32)
    m = np.zeros((n, cand_width), np.uint8)
    lib().orc_candidate_blocks(_p(S), n, L, _p(pos), ratio, compress_len, cand_block, cand_topk, cand_width, _p(m))
    return m


def sparse_attn(q, rows_a, rows_b, idx, sink, scale):
    """q [n, H, hd], rows_a [Na, hd], rows_b [Nb, hd] or None, idx [n, n_idx], sink [H] -> o [n, H, hd]."""
    q = _c(q, np.uint16)
    rows_a = _c(rows_a, np.uint16)
    n, H, hd = q.shape
    if rows_b is None:
        rows_b = np.zeros((0, hd), np.uint16)
    rows_b = _c(rows_b, np.uint16)
    idx = _c(idx, np.int32)
    sink = _c(sink, np.float32)
    o = np.empty_like(q)
    rc = lib().orc_sparse_attn(_p(q), n, H, hd, _p(rows_a), rows_a.shape[0], _p(rows_b), rows_b.shape[0], _p(idx),
                               idx.shape[1], _p(sink), scale, _p(o))
    if rc != 0:
        raise ValueError("oracle sparse_attn: index out of range")
    return o


# ---------------------------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------------------------

class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("dim", "n_heads", "head_dim", "rope_dim", "q_rank", "o_rank",
                                            "groups", "window")] + \
               [("eps", ctypes.c_float)] + \
               [(n, ctypes.c_int) for n in ("index_heads", "index_hd", "index_topk", "cand_block")]


class _Role(ctypes.Structure):
    _fields_ = [("ratio", ctypes.c_int), ("is_index_source", ctypes.c_int), ("uses_candidates", ctypes.c_int)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, P) for n in ("sink", "q_norm", "kv_norm", "wq_a", "wq_b", "wkv", "wo_a", "wo_b", "idx_wq_b",
                                 "idx_wproj")]


class _Shared(ctypes.Structure):
    _fields_ = [("compress_kv", P), ("index_k", P), ("compress_len", I64), ("Lstride", I64), ("topk_idxs", P),
                ("candidates", P), ("cand_width", ctypes.c_int)]


class _Debug(ctypes.Structure):
    _fields_ = [(n, P) for n in ("q", "kv", "kv_codes", "kv_scale", "idx", "scores", "o", "og", "qr", "qI", "wI")]


def _cfg_struct(cfg):
    return _Cfg(cfg["dim"], cfg["n_heads"], cfg["head_dim"], cfg["rope_dim"], cfg["q_rank"], cfg["o_rank"],
                cfg["groups"], cfg["window"], cfg["eps"], cfg.get("index_heads", 0), cfg.get("index_hd", 0),
                cfg.get("index_topk", 0), cfg.get("cand_block", 1))


def param_counts(cfg, with_indexer=True):
    out = np.zeros(7, np.int64)
    c = _cfg_struct(cfg)
    lib().orc_param_counts(ctypes.byref(c), int(with_indexer), _p(out))
    return [int(v) for v in out]


def attn_forward(cfg, role, w, ring, x, start_pos, rope_tab, shared=None, tok_mask=None, debug=True):
    """One layer forward.  x [B, T, dim] bf16 bits; ring [B, W, hd] bf16 bits, updated in place.

    ``w`` maps sink, q_norm, kv_norm (f32) and wq_a, wq_b, wkv, wo_a, wo_b, idx_wq_b, idx_wproj (bf16
    bits, [out, in]).  ``shared`` (ratio > 0) maps compress_kv [B, L, hd], index_k [B, L, dI],
    compress_len, topk_idxs [B*T, K] int32 (read by reuse layers, written by index sources) and
    optionally candidates [B*T, cand_width] uint8.  Returns a dict with ``out`` [B, T, dim] and the
    intermediates (q, kv, kv_codes, kv_scale, idx, scores, o, og, qr, qI, wI) when ``debug``.
    """
    L = lib()
    assert ring.flags.c_contiguous and ring.dtype == np.uint16
    x = _c(x, np.uint16)
    B, T, dim = x.shape
    H, hd, G = cfg["n_heads"], cfg["head_dim"], cfg["groups"]
    NT = B * T
    c = _cfg_struct(cfg)
    r = _Role(role.get("ratio", 0), int(role.get("is_index_source", 0)), int(role.get("uses_candidates", 0)))
    keep = []

    def ptr(a, dtype):
        if a is None:
            return None
        a = _c(a, dtype)
        keep.append(a)
        return a.ctypes.data

    wt = _Weights(ptr(w["sink"], np.float32), ptr(w["q_norm"], np.float32), ptr(w["kv_norm"], np.float32),
                  ptr(w["wq_a"], np.uint16), ptr(w["wq_b"], np.uint16), ptr(w["wkv"], np.uint16),
                  ptr(w["wo_a"], np.uint16), ptr(w["wo_b"], np.uint16), ptr(w.get("idx_wq_b"), np.uint16),
                  ptr(w.get("idx_wproj"), np.uint16))
    sh_p = None
    L_stride = 1
    if shared is not None:
        ckv = shared.get("compress_kv")
        L_stride = ckv.shape[1] if ckv is not None else 1
        tk = shared.get("topk_idxs")
        if tk is not None:
            assert tk.flags.c_contiguous and tk.dtype == np.int32
            keep.append(tk)
        cand = shared.get("candidates")
        sh = _Shared(ptr(ckv, np.uint16), ptr(shared.get("index_k"), np.uint16), int(shared.get("compress_len", 0)),
                     L_stride, None if tk is None else tk.ctypes.data, ptr(cand, np.uint8),
                     0 if cand is None else cand.shape[-1])
        sh_p = ctypes.byref(sh)
    out = np.zeros((B, T, dim), np.uint16)
    dbg = {}
    dbg_p = None
    if debug:
        n_idx = L.orc_n_idx(ctypes.byref(c), ctypes.byref(r))
        Hi, dI = cfg.get("index_heads", 0), cfg.get("index_hd", 0)
        dbg = dict(q=np.zeros((NT, H, hd), np.uint16), kv=np.zeros((NT, hd), np.uint16),
                   kv_codes=np.zeros((NT, hd), np.uint8), kv_scale=np.zeros((NT, hd // 32), np.int8),
                   idx=np.zeros((NT, n_idx), np.int32), scores=np.full((NT, L_stride), np.nan, np.float32),
                   o=np.zeros((NT, H, hd), np.uint16), og=np.zeros((NT, G * cfg["o_rank"]), np.uint16),
                   qr=np.zeros((NT, cfg["q_rank"]), np.uint16), qI=np.zeros((NT, max(Hi * dI, 1)), np.uint16),
                   wI=np.zeros((NT, max(Hi, 1)), np.float32))
        d = _Debug(*[dbg[k].ctypes.data for k in ("q", "kv", "kv_codes", "kv_scale", "idx", "scores", "o", "og",
                                                  "qr", "qI", "wI")])
        dbg_p = ctypes.byref(d)
    tm = ptr(tok_mask, np.uint8)
    rope_tab = _c(rope_tab, np.float32)
    rc = L.orc_attn_forward(ctypes.byref(c), ctypes.byref(r), ctypes.byref(wt), _p(ring), _p(x), B, T, start_pos,
                            sh_p, _p(rope_tab), rope_tab.shape[0], tm, _p(out), dbg_p)
    if rc != 0:
        raise ValueError("oracle attn_forward refused the call (code %d)" % rc)
    res = dict(out=out)
    res.update(dbg)
    return res


class _CompWeights(ctypes.Structure):
    _fields_ = [(n, P) for n in ("wkv_f32", "wgate", "wkv_bf16", "norm", "wk", "k_norm")]


def compress_state(B, ratio, hd):
    """A kv source's empty partial group: kv [B, ratio, hd] = 0, score = -inf (f32)."""
    kv = np.empty((B, ratio, hd), np.float32)
    sc = np.empty((B, ratio, hd), np.float32)
    lib().orc_compress_state_init(_p(kv), _p(sc), kv.size)
    return kv, sc


def compress(cfg, ratio, w, st_kv, st_score, x, start_pos, rope_tab, Z, KI=None, compress_len=0, y_dbg=None):
    """The kv source's compressor over x [B, T, dim] bf16 bits at start_pos (see orc_compress): updates
    the partial group st_kv / st_score [B, ratio, hd] f32 and writes the closed groups' rows of the
    latent cache Z [B, L, hd] and (with w["wk"]) the index keys KI [B, L, dI], both bf16 bits, in
    place.  ``w`` maps wkv (f32 [hd, dim] at ratio > 1, bf16 bits at ratio 1), wgate (f32, ratio > 1),
    norm (f32 [hd]), and optionally wk (bf16 bits [dI, hd]) and k_norm (f32 [dI]).  y_dbg ([B, L, hd]
    bf16 bits, optional) receives the normed rows before RoPE and fp8.  Returns compress_len."""
    x = _c(x, np.uint16)
    B, T, dim = x.shape
    c = _cfg_struct(cfg)
    keep = []

    def ptr(a, dtype):
        if a is None:
            return None
        a = _c(a, dtype)
        keep.append(a)
        return a.ctypes.data

    for a, dt in ((st_kv, np.float32), (st_score, np.float32), (Z, np.uint16)):
        assert a.flags.c_contiguous and a.dtype == dt
    if KI is not None:
        assert KI.flags.c_contiguous and KI.dtype == np.uint16
    if y_dbg is not None:
        assert y_dbg.flags.c_contiguous and y_dbg.dtype == np.uint16
    cw = _CompWeights(ptr(w["wkv"], np.float32) if ratio > 1 else None, ptr(w.get("wgate"), np.float32),
                      ptr(w["wkv"], np.uint16) if ratio == 1 else None, ptr(w["norm"], np.float32),
                      ptr(w.get("wk"), np.uint16), ptr(w.get("k_norm"), np.float32))
    n = ctypes.c_int64(int(compress_len))
    rope_tab = _c(rope_tab, np.float32)
    rc = lib().orc_compress(ctypes.byref(c), int(ratio), ctypes.byref(cw), _p(st_kv), _p(st_score), _p(x), B, T,
                            int(start_pos), _p(rope_tab), rope_tab.shape[0], _p(Z),
                            None if KI is None else KI.ctypes.data, Z.shape[1], ctypes.byref(n),
                            None if y_dbg is None else y_dbg.ctypes.data)
    if rc != 0:
        raise ValueError("oracle compress refused the call (code %d)" % rc)
    return int(n.value)


def num_threads():
    return lib().orc_num_threads()


def set_num_threads(n):
    lib().orc_set_num_threads(n)
