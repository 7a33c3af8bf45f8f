"""The C ABI library loads and exports every function include/csa.h declares, and the Python
binding declares each of them (no GPU needed: no compute call is made)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^CSA_API\s+[\w\s\*]*?\b(\w+)\s*\(", txt, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libpath():
    from compressed_sparse_attention_attn_gb300 import _build
    return _build.build()


def test_header_declares_the_layer_call():
    names = _declared()
    assert "attn_v41_forward" in names and "csa_create" in names and len(names) >= 15


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    for n in _declared():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(_declared()) <= exported


def test_binding_covers_every_declared_symbol(libpath):
    from compressed_sparse_attention_attn_gb300 import _abi
    assert set(_declared()) == set(_abi.SIGNATURES)
    _abi.load()


def test_binding_refuses_tensors_the_kernels_cannot_take():
    """The kernels read and write through raw pointers, so the binding refuses, before any call, a
    host tensor where a device pointer is declared, a strided view and a dtype other than the one
    declared (a narrower one would be read past its end)."""
    import torch
    import compressed_sparse_attention_attn_gb300 as csa
    with pytest.raises(ValueError, match="CUDA"):
        csa._dev(torch.zeros(4, dtype=torch.float32), torch.float32, "S")
    with pytest.raises(ValueError, match="contiguous"):
        csa._host(torch.zeros(4, 6, dtype=torch.float32).t(), torch.float32, "table")
    with pytest.raises(ValueError, match="bfloat16"):
        csa._host(torch.zeros(8, dtype=torch.float32), torch.bfloat16, "x_host")
    t = torch.zeros(8, dtype=torch.bfloat16)
    assert csa._host(t, torch.bfloat16, "x_host").value == t.data_ptr()
    assert csa._dev(None, torch.float32, "cand") is None and csa._host(None) is None
    # the declared dtypes line up with the structs' fields
    assert len(csa.DEBUG_DTYPES) == len(csa.DEBUG_FIELDS) == len(csa._abi.Debug._fields_)
    assert len(csa.WEIGHT_DTYPES) == len(csa.WEIGHT_FIELDS) == len(csa._abi.LayerWeights._fields_) - 1
    assert [f for f, _ in csa._abi.Debug._fields_] == list(csa.DEBUG_FIELDS)
    assert [f for f, _ in csa._abi.LayerWeights._fields_][1:] == list(csa.WEIGHT_FIELDS)
