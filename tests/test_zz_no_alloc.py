"""csa_linear_noalloc, the allocation-free projection, against the oracle and against csa_linear.

Some callers cannot allocate device memory: an embedding runtime that owns a fixed device-memory
budget and forbids allocations outside it, or code that runs without a csa_ctx (creating one
allocates workspaces).  For them the library exports one projection entry point whose scratch is a
static device array inside the library.  This file checks, through the C ABI, that it gives the
oracle's linear_bf16 and the same result as csa_linear (within the bf16 tolerance used by the other
tests) on two calls in a row -- the second call finds the array holding the first call's contents --
that its status word reads clean afterwards, that a call changes no device-memory count, and that
it refuses sizes beyond its fixed scratch.  It is collected last, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from _helpers import assert_close_bf16, to_dev, to_np

pytestmark = pytest.mark.gpu


def _noalloc(L, x, W, y, groups):
    K = W.shape[1]
    N = W.shape[0] // groups
    return L.csa_linear_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], K, x.shape[1],
                                ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(y.data_ptr()), y.shape[1], groups,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,K,N,groups", [(32, 5120, 1280, 1), (32, 4096, 1024, 8), (7, 1280, 4224, 1)])
def test_noalloc_matches_oracle_and_linear_on_two_calls(M, K, N, groups):
    import compressed_sparse_attention_attn_gb300 as csa
    import oracle as orc
    from csa_inputs import Geometry
    L = csa.lib()
    rng = np.random.default_rng(11 + M + N)
    x_np = orc.f32_to_bf16(rng.standard_normal((M, K * groups)).astype(np.float32))
    W_np = orc.f32_to_bf16((rng.standard_normal((N * groups, K)) / math.sqrt(K)).astype(np.float32))
    oracle = np.concatenate([orc.linear_bf16(x_np[:, g * K:(g + 1) * K], W_np[g * N:(g + 1) * N])
                             for g in range(groups)], 1)
    x, W = to_dev(x_np), to_dev(W_np)
    ctx = csa.Context(Geometry(dim=64, max_tokens=1, max_batch=1, max_seq=16).as_dict())
    existing = to_np(ctx.linear(x, W, groups=groups))
    ctx.close()
    for _ in range(2):
        y = torch.full((M, N * groups), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(L, x, W, y, groups)
        assert rc == 0, L.attn_v41_last_error()
        torch.cuda.synchronize()
        assert_close_bf16(to_np(y), oracle, what="csa_linear_noalloc vs the oracle")
        assert_close_bf16(to_np(y), existing, what="csa_linear_noalloc vs csa_linear")
    assert L.csa_linear_noalloc_status(1) == 0, L.attn_v41_last_error()


def test_noalloc_changes_no_device_memory_count():
    import compressed_sparse_attention_attn_gb300 as csa
    L = csa.lib()
    gen = torch.Generator().manual_seed(5)
    x = torch.randn(16, 1024, generator=gen).to(torch.bfloat16).cuda()
    W = (torch.randn(512, 1024, generator=gen) / 32).to(torch.bfloat16).cuda()
    y = torch.empty(16, 512, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(L, x, W, y, 1) == 0  # warm-up: the first call on a device looks the array up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(L, x, W, y, 1) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import compressed_sparse_attention_attn_gb300 as csa
    L = csa.lib()
    x = torch.zeros(33, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    y = torch.full((33, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(L, x, W, y, 1) == -2  # CSA_ERR_SHAPE: more tokens than the static scratch holds
    torch.cuda.synchronize()
    assert (y == 7.0).all()  # nothing was launched
