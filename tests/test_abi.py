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
