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


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


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
        self._c = _abi.Shared(_ptr(self.compress_kv), _ptr(self.index_k), self.compress_len, stride,
                              _ptr(self.topk_idxs), self.topk, int(self.has_topk), _ptr(self.candidates),
                              0 if self.candidates is None else self.candidates.shape[-1])
        return self._c

    def sync_back(self):
        if self._c is not None:
            self.has_topk = bool(self._c.has_topk)


DEBUG_FIELDS = ("q", "kv", "kv_codes", "kv_scale", "idx", "scores", "o", "og", "qr", "qI", "wI")


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
        return _abi.LayerWeights(make_role(role), *[_ptr(w.get(n)) for n in (
            "sink", "q_norm", "kv_norm", "wq_a", "wq_b", "wkv", "wo_a", "wo_b", "idx_wq_b", "idx_wproj")])

    def state_init(self, ring, batch, stream=None):
        st = _abi.LayerState(_ptr(ring))
        _check(lib().csa_state_init(self.h, ctypes.byref(st), batch, _stream(stream)), "csa_state_init")

    def forward(self, w, role, ring, x, start_pos, shared=None, out=None, debug=None, stream=None, lw=None):
        """attn_v41_forward.  x [B, T, dim] bf16 -> out [B, T, dim] bf16; ring [max_batch, W, hd] bf16.
        ``debug``: dict of preallocated device tensors named as in csa_debug.  ``lw``: a prebuilt
        LayerWeights struct (skips re-marshalling)."""
        B, T, _ = x.shape
        if out is None:
            out = torch.empty_like(x)
        if lw is None:
            lw = self.layer_weights(w, role)
        st = _abi.LayerState(_ptr(ring))
        sh = shared.struct() if shared is not None else None
        dbg = None
        if debug:
            dbg = _abi.Debug(*[_ptr(debug.get(n)) for n in DEBUG_FIELDS])
        rc = lib().attn_v41_forward(self.h, ctypes.byref(lw), ctypes.byref(st), _ptr(x), B, T, start_pos,
                                    ctypes.byref(sh) if sh is not None else None, _ptr(out),
                                    ctypes.byref(dbg) if dbg is not None else None, _stream(stream))
        _check(rc, "attn_v41_forward")
        if shared is not None:
            shared.sync_back()
        return out

    def forward_host(self, lw, ring, x_host, start_pos, shared, out_host, B, T, stream=None):
        """attn_v41_forward_host with host tensors (pinned for overlap)."""
        st = _abi.LayerState(_ptr(ring))
        sh = shared.struct() if shared is not None else None
        rc = lib().attn_v41_forward_host(self.h, ctypes.byref(lw), ctypes.byref(st), _ptr(x_host), B, T, start_pos,
                                         ctypes.byref(sh) if sh is not None else None, _ptr(out_host), _stream(stream))
        _check(rc, "attn_v41_forward_host")
        if shared is not None:
            shared.sync_back()

    def rope_table(self, ratio_class):
        g = self.cfg
        t = torch.empty(g.max_seq, g.rope_dim // 2, 2, dtype=torch.float32)
        _check(lib().csa_rope_table_get(self.h, ratio_class, _ptr(t)), "csa_rope_table_get")
        return t

    def status(self, clear=True):
        return lib().csa_status(self.h, int(clear))

    def workspace_bytes(self):
        return lib().csa_workspace_bytes(self.h)

    def trace(self, enable=True):
        _check(lib().csa_trace_enable(self.h, int(enable)), "csa_trace_enable")

    def trace_read(self):
        """[(stage name, milliseconds)] of the last traced forward (waits for its events)."""
        names = (ctypes.c_char_p * 32)()
        ms = (ctypes.c_float * 32)()
        n = lib().csa_trace_read(self.h, 32, names, ms)
        if n < 0:
            _check(n, "csa_trace_read")
        return [(names[i].decode(), float(ms[i])) for i in range(min(n, 32))]

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
        _check(lib().csa_linear(self.h, _ptr(x), M, K, x.shape[-1], _ptr(W), N, K, _ptr(out), out.shape[-1], groups,
                                _stream(stream)), "csa_linear")
        return out

    def sparse_attn(self, q, rows_a, a_len, idx_a, sink, scale, rows_b=None, b_len=0, idx_b=None, o=None, o_rot=None,
                    rd=0, start_pos=0, tab=None, B=1, T=None, stream=None):
        """q [B*T, H, hd]; rows_a [B, ., hd]; rows_b [B, ., hd]; idx_a [B*T, na]; idx_b [B*T, nb]."""
        n, H, hd = q.shape
        T = n // B if T is None else T
        _check(lib().csa_sparse_attn(self.h, _ptr(q), B, T, H, hd, _ptr(rows_a), rows_a.shape[1] * hd, a_len,
                                     _ptr(rows_b), 0 if rows_b is None else rows_b.shape[1] * hd, b_len, _ptr(idx_a),
                                     idx_a.shape[1], _ptr(idx_b), 0 if idx_b is None else idx_b.shape[1], _ptr(sink),
                                     scale, _ptr(o), _ptr(o_rot), rd, start_pos, _ptr(tab),
                                     0 if tab is None else tab.shape[0], _stream(stream)), "csa_sparse_attn")


def rmsnorm(x, w, eps, out=None, stream=None):
    N = x.shape[-1]
    out = torch.empty_like(x) if out is None else out
    _check(lib().csa_rmsnorm(_ptr(x), x.numel() // N, N, _ptr(w), eps, _ptr(out), _stream(stream)), "csa_rmsnorm")
    return out


def rope(x, rd, pos, tab, inverse=False, rows_per_pos=1, stream=None):
    """In place on x [rows, row_len]."""
    row_len = x.shape[-1]
    _check(lib().csa_rope(_ptr(x), x.numel() // row_len, row_len, rd, _ptr(pos), rows_per_pos, _ptr(tab), tab.shape[0],
                          int(inverse), _stream(stream)), "csa_rope")
    return x


def act_quant(x, codes=None, scale_exp=None, stream=None):
    """In place on x; codes uint8 like x, scale_exp int8 [n/32]."""
    _check(lib().csa_act_quant(_ptr(x), x.numel(), _ptr(codes), _ptr(scale_exp), _stream(stream)), "csa_act_quant")
    return x


def kv_finish(kv_in, kv_out, B, T, start_pos, rd, tab, ring, win_idx=None, codes=None, scales=None, stream=None):
    hd = kv_in.shape[-1]
    W = ring.shape[1]
    _check(lib().csa_kv_finish(_ptr(kv_in), _ptr(kv_out), B, T, start_pos, hd, rd, _ptr(tab), tab.shape[0], _ptr(ring), W,
                               _ptr(win_idx), 0 if win_idx is None else win_idx.shape[-1], _ptr(codes), _ptr(scales),
                               _stream(stream)), "csa_kv_finish")


def index_scores(qI, wI, KI, B, T, start_pos, compress_len, ratio, S, cand=None, cand_block=1, stream=None):
    n, Hi, dI = qI.shape
    _check(lib().csa_index_scores(_ptr(qI), _ptr(wI), _ptr(KI), B, T, start_pos, Hi, dI, KI.shape[1], compress_len,
                                  ratio, _ptr(cand), 0 if cand is None else cand.shape[-1], cand_block, _ptr(S),
                                  _stream(stream)), "csa_index_scores")
    return S


def index_topk(S, B, T, start_pos, compress_len, ratio, K, out, offset=0, cand=None, cand_block=1, stream=None):
    _check(lib().csa_index_topk(_ptr(S), B, T, start_pos, S.shape[-1], compress_len, ratio, _ptr(cand),
                                0 if cand is None else cand.shape[-1], cand_block, K, offset, _ptr(out),
                                _stream(stream)), "csa_index_topk")
    return out
