"""csa_linear_noalloc, the allocation-free projection, against csa_linear.

Some callers cannot allocate device memory: an embedding runtime that owns a fixed device-memory
budget, or code that runs without a csa_ctx (creating one allocates workspaces).  For them the
library exports one projection entry point whose scratch is a static device array inside the
library.  This file checks, through the C ABI, that it gives the same result as csa_linear (within
the bf16 tolerance used by the other tests) on two calls in a row -- the second call finds the
array holding the first call's contents -- and that it refuses sizes beyond its fixed scratch.
It is collected last, so a run that stops at the first failure has run every other test before it.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from _helpers import assert_close_bf16, to_np

pytestmark = pytest.mark.gpu


def _noalloc(L, x, W, y, groups):
    K = W.shape[1]
    N = W.shape[0] // groups
    return L.csa_linear_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], K, x.shape[1],
                                ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(y.data_ptr()), y.shape[1], groups,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,K,N,groups", [(32, 5120, 1280, 1), (32, 4096, 1024, 8), (7, 1280, 4224, 1)])
def test_noalloc_matches_linear_on_two_calls(M, K, N, groups):
    import compressed_sparse_attention_attn_gb300 as csa
    from csa_inputs import Geometry
    L = csa.lib()
    gen = torch.Generator().manual_seed(11 + M + N)
    x = torch.randn(M, K * groups, generator=gen).to(torch.bfloat16).cuda()
    W = (torch.randn(N * groups, K, generator=gen) / math.sqrt(K)).to(torch.bfloat16).cuda()
    ctx = csa.Context(Geometry(dim=64, max_tokens=1, max_batch=1, max_seq=16).as_dict())
    want = to_np(ctx.linear(x, W, groups=groups))
    for _ in range(2):
        y = torch.full((M, N * groups), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(L, x, W, y, groups)
        assert rc == 0, L.attn_v41_last_error()
        torch.cuda.synchronize()
        assert_close_bf16(to_np(y), want, what="csa_linear_noalloc")
    ctx.close()


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import compressed_sparse_attention_attn_gb300 as csa
    L = csa.lib()
    x = torch.zeros(33, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    y = torch.full((33, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(L, x, W, y, 1) == -2  # CSA_ERR_SHAPE: more tokens than the static scratch holds
    torch.cuda.synchronize()
    assert (y == 7.0).all()  # nothing was launched
