"""The C-ABI library on the CPU: it builds, loads, exports every entry point
include/csa.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from sparse_compressed_kv_gb300 import build as B
from sparse_compressed_kv_gb300 import csa

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "csa.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return csa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for fn in ("csa_workspace_size", "csa_indexer_scores", "csa_topk", "csa_gather_mixed",
               "csa_sparse_mqa_decode", "csa_decode", "csa_status_string", "csa_abi_version"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for fn in declared_functions():
        assert hasattr(lib, fn), fn
    assert csa.abi_version() == 1


def test_checked_build_exports_the_same_symbols():
    # libcsa_checks.so: the same sources with CSA_CHECKS defined (internal
    # bounds checks report CSA_DEV_CHECK); loaded on its own, not through csa
    path = B.build(checks=True)
    chk = ctypes.CDLL(path)
    for fn in declared_functions():
        assert hasattr(chk, fn), fn
    chk.csa_abi_version.restype = ctypes.c_int
    assert chk.csa_abi_version() == 1


def test_status_strings(lib):
    assert csa.status_string(0) == "CSA_OK"
    assert csa.status_string(7) == "CSA_ERR_WORKSPACE"


def _layout(T=1, B=1, R=256, maxr=256, swa_cap=128):
    return csa.csa_layout_t(B, T, R, maxr, None, None, None, None, swa_cap, None)


def test_workspace_size_is_host_only(lib):
    n = ctypes.c_size_t(0)
    L = _layout()
    P = csa.params(16, 64)
    assert lib.csa_workspace_size(ctypes.byref(L), ctypes.byref(P), ctypes.byref(n)) == 0
    assert n.value > 0
    # grows with the number of blocks (score row) and with the number of tokens
    L2 = _layout(R=262144, maxr=262144)
    n2 = ctypes.c_size_t(0)
    lib.csa_workspace_size(ctypes.byref(L2), ctypes.byref(P), ctypes.byref(n2))
    assert n2.value >= n.value + 4 * (262144 - 256)


@pytest.mark.parametrize("field,value,code", [
    ("hd", 256, 2), ("ihd", 64, 2), ("n_ih", 32, 2), ("n_heads", 24, 2), ("n_heads", 256, 2),
    ("top_k", 0, 1), ("top_k", 4096, 2), ("window", 0, 1), ("ratio", 0, 1),
])
def test_bad_params_rejected_before_launch(lib, field, value, code):
    P = csa.params(16, 64)
    setattr(P, field, value)
    L = _layout()
    n = ctypes.c_size_t(0)
    assert lib.csa_workspace_size(ctypes.byref(L), ctypes.byref(P), ctypes.byref(n)) == code
    assert lib.csa_indexer_scores(ctypes.byref(L), ctypes.byref(P), None, None, None, None, 256,
                                  None, None) == code


def test_bad_layout_and_null_pointers_rejected(lib):
    P = csa.params(16, 64)
    assert lib.csa_decode(None, ctypes.byref(P), *([None] * 10), 0, None) == 1
    L = _layout()
    # tokens but no layout arrays
    assert lib.csa_indexer_scores(ctypes.byref(L), ctypes.byref(P), None, None, None, None, 256,
                                  None, None) == 1
    # max rows above total rows
    L = _layout(R=10, maxr=20)
    assert lib.csa_topk(ctypes.byref(L), ctypes.byref(P), None, 20, None, None, None, None, 0,
                        None) == 1
    # the ring smaller than the window
    L = _layout(swa_cap=64)
    dummy = ctypes.c_void_p(16)
    L.tok_seq = L.tok_pos = L.comp_off = L.swa_kv = L.swa_first_pos = dummy
    assert lib.csa_gather_mixed(ctypes.byref(L), ctypes.byref(P), dummy, dummy, dummy, dummy,
                                dummy, dummy, None) == 3
    # no tokens: nothing to do, nothing launched
    L = _layout(T=0)
    assert lib.csa_decode(ctypes.byref(L), ctypes.byref(P), *([None] * 10), 0, None) == 0


def test_binding_refuses_host_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        csa._p(torch.zeros(4))


def _noalloc(lib):
    fn = lib.csa_topk_noalloc
    fn.argtypes = [ctypes.POINTER(csa.csa_layout_t), ctypes.POINTER(csa.csa_params_t),
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


@pytest.mark.parametrize("case", ["n_heads", "scale", "top_k0", "top_k2049", "rows2g",
                                  "no_tok_seq", "ld", "maxr", "null_idx"])
def test_noalloc_rejects_what_topk_rejects(lib, case):
    """csa_topk_noalloc returns the code csa_topk returns for the same bad
    input (both decide before any device call)."""
    dummy = ctypes.c_void_p(256)
    P = csa.params(16, 64)
    L = _layout(R=1000, maxr=1000)
    L.tok_seq = L.tok_pos = L.comp_off = dummy
    ld = 1000
    idx = dummy
    if case == "n_heads":
        P.n_heads = 24
    elif case == "scale":
        P.scale = float("nan")
    elif case == "top_k0":
        P.top_k = 0
    elif case == "top_k2049":
        P.top_k = 2049
    elif case == "rows2g":
        L = _layout(R=1 << 31, maxr=1000)
        L.tok_seq = L.tok_pos = L.comp_off = dummy
    elif case == "no_tok_seq":
        L.tok_seq = None
    elif case == "ld":
        ld = 999
    elif case == "maxr":
        L = _layout(R=10, maxr=20)
        L.tok_seq = L.tok_pos = L.comp_off = dummy
    elif case == "null_idx":
        idx = None
    want = lib.csa_topk(ctypes.byref(L), ctypes.byref(P), dummy, ld, idx, dummy, dummy, None, 0,
                        None)
    got = _noalloc(lib)(ctypes.byref(L), ctypes.byref(P), dummy, ld, idx, dummy, dummy, None)
    assert want != 0 and want != 7      # decided before the workspace check
    assert got == want


def test_noalloc_token_limit_is_a_capacity_error(lib):
    dummy = ctypes.c_void_p(256)
    P = csa.params(16, 64)
    L = _layout(T=17, R=1000, maxr=1000)
    L.tok_seq = L.tok_pos = L.comp_off = dummy
    assert _noalloc(lib)(ctypes.byref(L), ctypes.byref(P), dummy, 1000, dummy, dummy, dummy,
                         None) == 3
