"""GB300 (sm_103a) compressed sparse attention layer core of DeepSeek-V4.1.

Python face of the C ABI in ``include/csa.h``: every function here marshals torch CUDA tensors
(device pointers, the current stream) into one library call; all arithmetic runs in the library's
CUDA kernels.  bf16 tensors are ``torch.bfloat16``; int8/uint8/int32/f32 as the header states.
"""
import ctypes

import torch

from . import _abi

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _abi.load()
    return _lib


class CsaError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = lib().attn_v41_last_error().decode(errors="replace")
        super().__init__("%s: %s (%s)" % (where, _abi.ERRORS.get(code, code), msg))


def _check(rc, where):
    if rc != 0:
        raise CsaError(rc, where)


def _checked(t, dtype, cuda, what):
    if t.is_cuda != cuda:
        raise ValueError("%s: expected a %s tensor, got one on %s" % (what, "CUDA" if cuda else "host", t.device))
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s: expected %s, got %s" % (what, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s: expected a contiguous tensor (shape %s, strides %s)" % (what, tuple(t.shape), t.stride()))
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype=None, what="tensor"):
    """Device pointer of a contiguous CUDA tensor of the given dtype; None -> NULL.  The kernels read
    and write through raw pointers, so a host tensor, a strided view or a narrower dtype is refused
    here rather than read out of bounds on the GPU."""
    return None if t is None else _checked(t, dtype, True, what)


def _host(t, dtype=None, what="tensor"):
    """Host pointer of a contiguous CPU tensor of the given dtype (pinned for copies that overlap)."""
    return None if t is None else _checked(t, dtype, False, what)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


CFG_FIELDS = [f for f, _ in _abi.Cfg._fields_]


def make_cfg(geom):
    """csa_cfg from a mapping (or an object with the same attribute names)."""
    get = geom.get if isinstance(geom, dict) else (lambda k, d=None: getattr(geom, k, d))
    vals = {}
    for f, ty in _abi.Cfg._fields_:
        v = get(f, 0)
        vals[f] = float(v) if ty is _abi.F else int(v)
    return _abi.Cfg(**vals)


def make_role(role):
    return _abi.Role(int(role.get("ratio", 0)), int(role.get("is_kv_source", 0)), int(role.get("is_index_source", 0)),
                     int(role.get("is_candidate_source", 0)), int(role.get("uses_candidates", 0)))


class Shared:
    """What source layers publish (SharedV41 of the attn_v41 runtime) as device tensors."""

    def __init__(self, compress_kv, index_k, compress_len, topk_idxs, topk, candidates=None, has_topk=False):
        self.compress_kv = compress_kv
        self.index_k = index_k
        self.compress_len = int(compress_len)
        self.topk_idxs = topk_idxs
        self.topk = int(topk)
        self.candidates = candidates
        self.has_topk = bool(has_topk)
        self._c = None

    def struct(self):
        stride = self.compress_kv.shape[1] if self.compress_kv is not None else 0
        self._c = _abi.Shared(_dev(self.compress_kv, torch.bfloat16, "compress_kv"), _dev(self.index_k, torch.bfloat16, "index_k"),
                              self.compress_len, stride, _dev(self.topk_idxs, torch.int32, "topk_idxs"), self.topk,
                              int(self.has_topk), _dev(self.candidates, torch.uint8, "candidates"),
                              0 if self.candidates is None else self.candidates.shape[-1])
        return self._c

    def sync_back(self, kv_state=None, with_keys=False):
        """What the library published into the struct: the selection flag and, after a kv source (its
        kv_state), its caches and their length."""
        if self._c is not None:
            self.has_topk = bool(self._c.has_topk)
            self.compress_len = int(self._c.compress_len)
        if kv_state is not None:
            self.compress_kv = kv_state["latent"]
            if with_keys:
                self.index_k = kv_state["index_keys"]


DEBUG_FIELDS = ("q", "kv", "kv_codes", "kv_scale", "idx", "scores", "o", "og", "qr", "qI", "wI")
DEBUG_DTYPES = (torch.bfloat16, torch.bfloat16, torch.uint8, torch.int8, torch.int32, torch.float32, torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.float32)
WEIGHT_FIELDS = ("sink", "q_norm", "kv_norm", "wq_a", "wq_b", "wkv", "wo_a", "wo_b", "idx_wq_b", "idx_wproj",
                 "wo_a_fp8", "wo_a_scale", "comp_wkv", "comp_wgate", "comp_norm", "idx_wk", "idx_k_norm")
# (comp_wkv is f32 at ratio > 1 and bf16 at ratio 1: its dtype is checked against the role)
WEIGHT_DTYPES = (torch.float32, torch.float32, torch.float32, torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.bfloat16,
                 torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.uint8, torch.float32, None, torch.float32,
                 torch.float32, torch.bfloat16, torch.float32)


def make_state(ring, kv_state=None):
    """csa_layer_state: the window ring, and for a kv source the dict kv_state with comp_kv,
    comp_score (f32 [max_batch, ratio, hd]), latent (bf16 [max_batch, rows, hd]) and index_keys (bf16
    [max_batch, rows, index_hd], may be None)."""
    if kv_state is None:
        return _abi.LayerState(_dev(ring, torch.bfloat16, "ring"))
    kv, sc, lat = kv_state["comp_kv"], kv_state["comp_score"], kv_state["latent"]
    ik = kv_state.get("index_keys")
    return _abi.LayerState(_dev(ring, torch.bfloat16, "ring"), _dev(kv, torch.float32, "comp_kv"),
                           _dev(sc, torch.float32, "comp_score"), kv.shape[1], _dev(lat, torch.bfloat16, "latent"),
                           _dev(ik, torch.bfloat16, "index_keys"), lat.shape[1])


class Context:
    """A csa_ctx: workspaces and RoPE tables for one geometry, on the current CUDA device."""

    def __init__(self, geom):
        self.geom = geom
        self.cfg = make_cfg(geom)
        h = ctypes.c_void_p()
        _check(lib().csa_create(ctypes.byref(self.cfg), ctypes.byref(h)), "csa_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            lib().csa_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- layer ---------------------------------------------------------------------------------
    @staticmethod
    def layer_weights(w, role):
        wkv = w.get("comp_wkv")
        if wkv is not None:
            want = torch.float32 if int(role.get("ratio", 0)) > 1 else torch.bfloat16
            _dev(wkv, want, "comp_wkv")
        return _abi.LayerWeights(make_role(role), *[_dev(w.get(n), dt, n) for n, dt in zip(WEIGHT_FIELDS, WEIGHT_DTYPES)])

    def state_init(self, ring, batch, stream=None, kv_state=None):
        st = make_state(ring, kv_state)
        _check(lib().csa_state_init(self.h, ctypes.byref(st), batch, _stream(stream)), "csa_state_init")

    def compress(self, w, role, ring, kv_state, x, start_pos, shared=None, y_dbg=None, stream=None):
        """csa_compress: the kv source's compressor over x [B, T, dim]; publishes into shared."""
        B, T, _ = x.shape
        lw = self.layer_weights(w, role)
        st = make_state(ring, kv_state)
        sh = shared.struct() if shared is not None else None
        _check(lib().csa_compress(self.h, ctypes.byref(lw), ctypes.byref(st), _dev(x, torch.bfloat16, "x"), B, T,
                                  start_pos, ctypes.byref(sh) if sh is not None else None,
                                  _dev(y_dbg, torch.bfloat16, "y_dbg"), _stream(stream)), "csa_compress")
        if shared is not None:
            shared.sync_back(kv_state, w.get("idx_wk") is not None)

    def forward(self, w, role, ring, x, start_pos, shared=None, out=None, debug=None, stream=None, lw=None,
                kv_state=None):
        """attn_v41_forward.  x [B, T, dim] bf16 -> out [B, T, dim] bf16; ring [max_batch, W, hd] bf16.
        ``debug``: dict of preallocated device tensors named as in csa_debug.  ``lw``: a prebuilt
        LayerWeights struct (skips re-marshalling)."""
        B, T, _ = x.shape
        if out is None:
            out = torch.empty_like(x)
        if lw is None:
            lw = self.layer_weights(w, role)
        st = make_state(ring, kv_state)
        sh = shared.struct() if shared is not None else None
        dbg = None
        if debug:
            dbg = _abi.Debug(*[_dev(debug.get(n), dt, n) for n, dt in zip(DEBUG_FIELDS, DEBUG_DTYPES)])
        rc = lib().attn_v41_forward(self.h, ctypes.byref(lw), ctypes.byref(st), _dev(x, torch.bfloat16, "x"), B, T, start_pos,
                                    ctypes.byref(sh) if sh is not None else None, _dev(out, torch.bfloat16, "out"),
                                    ctypes.byref(dbg) if dbg is not None else None, _stream(stream))
        _check(rc, "attn_v41_forward")
        if shared is not None:
            shared.sync_back(kv_state if int(role.get("is_kv_source", 0)) else None, bool(lw.idx_wk))
        return out

    def forward_host(self, lw, ring, x_host, start_pos, shared, out_host, B, T, stream=None):
        """attn_v41_forward_host with host tensors (pinned for overlap)."""
        st = _abi.LayerState(_dev(ring, torch.bfloat16, "ring"))
        sh = shared.struct() if shared is not None else None
        rc = lib().attn_v41_forward_host(self.h, ctypes.byref(lw), ctypes.byref(st), _host(x_host, torch.bfloat16, "x_host"), B, T,
                                         start_pos, ctypes.byref(sh) if sh is not None else None,
                                         _host(out_host, torch.bfloat16, "out_host"), _stream(stream))
        _check(rc, "attn_v41_forward_host")
        if shared is not None:
            shared.sync_back()

    def rope_table(self, ratio_class):
        g = self.cfg
        t = torch.empty(g.max_seq, g.rope_dim // 2, 2, dtype=torch.float32)
        _check(lib().csa_rope_table_get(self.h, ratio_class, _host(t, torch.float32, "table")), "csa_rope_table_get")
        return t

    def status(self, clear=True):
        return lib().csa_status(self.h, int(clear))

    def workspace_bytes(self):
        return lib().csa_workspace_bytes(self.h)

    def trace(self, enable=True, append=False):
        """Stage tracing: enable (each forward lists its own stages) or, with append, every forward
        appends to one list that restarts here (several layers, or a captured and replayed step)."""
        _check(lib().csa_trace_enable(self.h, 2 if (enable and append) else int(bool(enable))), "csa_trace_enable")

    def trace_read(self):
        """[(stage name, milliseconds)] of the listed stages (waits for their events)."""
        names = (ctypes.c_char_p * 64)()
        ms = (ctypes.c_float * 64)()
        n = lib().csa_trace_read(self.h, 64, names, ms)
        if n < 0:
            _check(n, "csa_trace_read")
        return [(names[i].decode(), float(ms[i])) for i in range(min(n, 64))]

    def last_launches(self):
        return lib().csa_last_launches(self.h)

    # -- steps ---------------------------------------------------------------------------------
    def linear(self, x, W, out=None, groups=1, stream=None):
        """y = x W^T (bf16, f32 accumulation); groups > 1: block-diagonal W [groups*N, K]."""
        K = W.shape[1]
        N = W.shape[0] // groups
        M = x.numel() // x.shape[-1]
        if out is None:
            out = torch.empty(x.shape[:-1] + (N * groups,), dtype=torch.bfloat16, device=x.device)
        _check(lib().csa_linear(self.h, _dev(x, torch.bfloat16, "x"), M, K, x.shape[-1], _dev(W, torch.bfloat16, "W"), N, K, _dev(out, torch.bfloat16, "out"),
                                out.shape[-1], groups, _stream(stream)), "csa_linear")
        return out

    def linear_fp8w(self, x, W8, scale, out=None, groups=1, stream=None):
        """y = x w^T with w = bf16(e4m3(W8) * scale per 128 x 128 tile); W8 uint8 [groups*N, K] codes,
        scale f32 [ceil(groups*N/128), ceil(K/128)]."""
        K = W8.shape[1]
        N = W8.shape[0] // groups
        M = x.numel() // x.shape[-1]
        if out is None:
            out = torch.empty(x.shape[:-1] + (N * groups,), dtype=torch.bfloat16, device=x.device)
        _check(lib().csa_linear_fp8w(self.h, _dev(x, torch.bfloat16, "x"), M, K, x.shape[-1], _dev(W8, torch.uint8, "W8"),
                                     _dev(scale, torch.float32, "scale"), N, K, _dev(out, torch.bfloat16, "out"),
                                     out.shape[-1], groups, _stream(stream)), "csa_linear_fp8w")
        return out

    def sparse_attn(self, q, rows_a, a_len, idx_a, sink, scale, rows_b=None, b_len=0, idx_b=None, o=None, o_rot=None,
                    rd=0, start_pos=0, tab=None, B=1, T=None, stream=None):
        """q [B*T, H, hd]; rows_a [B, ., hd]; rows_b [B, ., hd]; idx_a [B*T, na]; idx_b [B*T, nb]."""
        n, H, hd = q.shape
        T = n // B if T is None else T
        _check(lib().csa_sparse_attn(self.h, _dev(q, torch.bfloat16, "q"), B, T, H, hd, _dev(rows_a, torch.bfloat16, "rows_a"),
                                     rows_a.shape[1] * hd, a_len, _dev(rows_b, torch.bfloat16, "rows_b"),
                                     0 if rows_b is None else rows_b.shape[1] * hd, b_len, _dev(idx_a, torch.int32, "idx_a"),
                                     idx_a.shape[1], _dev(idx_b, torch.int32, "idx_b"), 0 if idx_b is None else idx_b.shape[1],
                                     _dev(sink, torch.float32, "sink"), scale, _dev(o, torch.bfloat16, "o"), _dev(o_rot, torch.bfloat16, "o_rot"), rd,
                                     start_pos, _dev(tab, torch.float32, "tab"), 0 if tab is None else tab.shape[0],
                                     _stream(stream)), "csa_sparse_attn")


def rmsnorm(x, w, eps, out=None, stream=None):
    N = x.shape[-1]
    out = torch.empty_like(x) if out is None else out
    _check(lib().csa_rmsnorm(_dev(x, torch.bfloat16, "x"), x.numel() // N, N, _dev(w, torch.float32, "w"), eps, _dev(out, torch.bfloat16, "out"),
                             _stream(stream)), "csa_rmsnorm")
    return out


def rope(x, rd, pos, tab, inverse=False, rows_per_pos=1, stream=None):
    """In place on x [rows, row_len]."""
    row_len = x.shape[-1]
    _check(lib().csa_rope(_dev(x, torch.bfloat16, "x"), x.numel() // row_len, row_len, rd, _dev(pos, torch.int32, "pos"), rows_per_pos,
                          _dev(tab, torch.float32, "tab"), tab.shape[0], int(inverse), _stream(stream)), "csa_rope")
    return x


def act_quant(x, codes=None, scale_exp=None, stream=None):
    """In place on x; codes uint8 like x, scale_exp int8 [n/32]."""
    _check(lib().csa_act_quant(_dev(x, torch.bfloat16, "x"), x.numel(), _dev(codes, torch.uint8, "codes"), _dev(scale_exp, torch.int8, "scale_exp"),
                               _stream(stream)), "csa_act_quant")
    return x


def kv_finish(kv_in, kv_out, B, T, start_pos, rd, tab, ring, win_idx=None, codes=None, scales=None, stream=None):
    hd = kv_in.shape[-1]
    W = ring.shape[1]
    _check(lib().csa_kv_finish(_dev(kv_in, torch.bfloat16, "kv_in"), _dev(kv_out, torch.bfloat16, "kv_out"), B, T, start_pos, hd, rd,
                               _dev(tab, torch.float32, "tab"), tab.shape[0], _dev(ring, torch.bfloat16, "ring"), W, _dev(win_idx, torch.int32, "win_idx"),
                               0 if win_idx is None else win_idx.shape[-1], _dev(codes, torch.uint8, "codes"),
                               _dev(scales, torch.int8, "scales"), _stream(stream)), "csa_kv_finish")


def index_scores(qI, wI, KI, B, T, start_pos, compress_len, ratio, S, cand=None, cand_block=1, stream=None):
    n, Hi, dI = qI.shape
    _check(lib().csa_index_scores(_dev(qI, torch.bfloat16, "qI"), _dev(wI, torch.float32, "wI"), _dev(KI, torch.bfloat16, "KI"), B, T, start_pos, Hi, dI,
                                  KI.shape[1], compress_len, ratio, _dev(cand, torch.uint8, "cand"),
                                  0 if cand is None else cand.shape[-1], cand_block, _dev(S, torch.float32, "S"), _stream(stream)),
           "csa_index_scores")
    return S


def candidate_blocks(S, B, T, start_pos, compress_len, ratio, cand_block, K, mask, stream=None):
    """csa_candidate_blocks: mask uint8 [B*T, cand_width] from the scores S f32 [B*T, L]."""
    _check(lib().csa_candidate_blocks(_dev(S, torch.float32, "S"), B, T, start_pos, S.shape[-1], compress_len, ratio,
                                      cand_block, K, _dev(mask, torch.uint8, "mask"), mask.shape[-1], _stream(stream)),
           "csa_candidate_blocks")
    return mask


def index_topk(S, B, T, start_pos, compress_len, ratio, K, out, offset=0, cand=None, cand_block=1, stream=None):
    _check(lib().csa_index_topk(_dev(S, torch.float32, "S"), B, T, start_pos, S.shape[-1], compress_len, ratio,
                                _dev(cand, torch.uint8, "cand"), 0 if cand is None else cand.shape[-1], cand_block, K, offset,
                                _dev(out, torch.int32, "out"), _stream(stream)), "csa_index_topk")
    return out
