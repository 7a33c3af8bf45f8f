"""ctypes declarations of ``include/csa.h`` (argument marshalling only).

Loads the in-tree ``libcsa.so``; raises ImportError if it has not been built -- there is no other
implementation to fall back on.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

CSA_OK = 0
ERRORS = {
    -1: "CSA_ERR_ARG", -2: "CSA_ERR_SHAPE", -3: "CSA_ERR_NO_KV_SOURCE", -4: "CSA_ERR_NO_SELECTION",
    -5: "CSA_ERR_TOO_WIDE", -6: "CSA_ERR_UNSUPPORTED", -7: "CSA_ERR_CUDA", -8: "CSA_ERR_DEVICE_TIMEOUT",
    -9: "CSA_ERR_NOMEM",
}

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
F = ctypes.c_float


class Cfg(ctypes.Structure):
    _fields_ = [(n, I) for n in ("dim", "n_heads", "head_dim", "rope_dim", "q_rank", "o_rank", "groups", "window")] + \
               [("eps", F)] + \
               [(n, I) for n in ("index_heads", "index_hd", "index_topk", "cand_block", "cand_topk_blocks",
                                 "max_seq", "max_tokens", "max_batch")] + \
               [("rope_theta", F), ("compress_rope_theta", F), ("rope_factor", F), ("orig_seq", I),
                ("beta_fast", F), ("beta_slow", F)]


class Role(ctypes.Structure):
    _fields_ = [(n, I) for n in ("ratio", "is_kv_source", "is_index_source", "is_candidate_source",
                                 "uses_candidates")]


class LayerWeights(ctypes.Structure):
    _fields_ = [("role", Role)] + [(n, P) for n in ("sink", "q_norm", "kv_norm", "wq_a", "wq_b", "wkv", "wo_a",
                                                      "wo_b", "idx_wq_b", "idx_wproj", "wo_a_fp8", "wo_a_scale",
                                                      "comp_wkv", "comp_wgate", "comp_norm", "idx_wk",
                                                      "idx_k_norm")]


class LayerState(ctypes.Structure):
    _fields_ = [("window", P), ("comp_kv", P), ("comp_score", P), ("comp_ratio", I), ("latent", P),
                ("index_keys", P), ("cache_rows", I)]


class Shared(ctypes.Structure):
    _fields_ = [("compress_kv", P), ("index_k", P), ("compress_len", I), ("compress_stride", I), ("topk_idxs", P),
                ("topk", I), ("has_topk", I), ("candidates", P), ("cand_width", I)]


class Debug(ctypes.Structure):
    _fields_ = [(n, P) for n in ("q", "kv", "kv_codes", "kv_scale", "idx", "scores", "o", "og", "qr", "qI", "wI")]


# name -> (restype, argtypes); mirrors include/csa.h
SIGNATURES = {
    "csa_create": (I, [ctypes.POINTER(Cfg), ctypes.POINTER(P)]),
    "csa_destroy": (I, [P]),
    "csa_state_init": (I, [P, ctypes.POINTER(LayerState), I, P]),
    "attn_v41_forward": (I, [P, ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerState), P, I, I, I,
                             ctypes.POINTER(Shared), P, ctypes.POINTER(Debug), P]),
    "attn_v41_forward_host": (I, [P, ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerState), P, I, I, I,
                                  ctypes.POINTER(Shared), P, P]),
    "attn_v41_last_error": (ctypes.c_char_p, []),
    "csa_rope_table_get": (I, [P, I, P]),
    "csa_status": (I, [P, I]),
    "csa_workspace_bytes": (ctypes.c_size_t, [P]),
    "csa_trace_enable": (I, [P, I]),
    "csa_trace_read": (I, [P, I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(F)]),
    "csa_last_launches": (I, [P]),
    "csa_linear": (I, [P, P, I, I, I, P, I, I, P, I, I, P]),
    "csa_linear_noalloc": (I, [P, I, I, I, P, I, I, P, I, I, P]),
    "csa_linear_noalloc_status": (I, [I]),
    "csa_debug_stall": (I, [ctypes.c_ulonglong]),
    "csa_linear_fp8w": (I, [P, P, I, I, I, P, P, I, I, P, I, I, P]),
    "csa_compress": (I, [P, ctypes.POINTER(LayerWeights), ctypes.POINTER(LayerState), P, I, I, I,
                         ctypes.POINTER(Shared), P, P]),
    "csa_rmsnorm": (I, [P, I, I, P, F, P, P]),
    "csa_rope": (I, [P, I64, I, I, P, I, P, I, I, P]),
    "csa_act_quant": (I, [P, I64, P, P, P]),
    "csa_kv_finish": (I, [P, P, I, I, I, I, I, P, I, P, I, P, I, P, P, P]),
    "csa_index_scores": (I, [P, P, P, I, I, I, I, I, I, I, I, P, I, I, P, P]),
    "csa_index_topk": (I, [P, I, I, I, I, I, I, P, I, I, I, I, P, P]),
    "csa_candidate_blocks": (I, [P, I, I, I, I, I, I, I, I, P, I, P]),
    "csa_sparse_attn": (I, [P, P, I, I, I, I, P, I64, I, P, I64, I, P, I, P, I, P, F, P, P, I, I, P, I, P]),
}


def load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libcsa.so is not built (run __graft_entry__.build() or "
                          "python -m compressed_sparse_attention_attn_gb300._build)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib
