"""csa_topk_noalloc: the top-k for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc at all -- an inference engine whose memory
planner owns every byte of the device, or a plug-in that is not allowed to
touch the allocator -- so they cannot provide the workspace csa_topk needs.
csa_topk_noalloc keeps its scratch in a fixed array inside the library
instead.  This test drives it through the C ABI and requires the same
selection as csa_topk, bit for bit, on two calls in a row (the second call
must not be confused by what the first left in the shared array).

It lives in its own file, collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import csa_workloads as W
from sparse_compressed_kv_gb300 import csa
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _noalloc_topk(run, scores, idx, n_sel):
    lib = csa.load()
    fn = lib.csa_topk_noalloc
    fn.argtypes = [ctypes.POINTER(csa.csa_layout_t), ctypes.POINTER(csa.csa_params_t),
                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    lc = run.layout.c()
    code = fn(ctypes.byref(lc), ctypes.byref(run.prm), csa._p(scores), int(scores.shape[1]),
              csa._p(idx), csa._p(n_sel), csa._p(run.status), csa._stream())
    return code


@pytest.mark.parametrize("wl_fn", [
    lambda: W.make("noalloc-a", seed=41, seq_lens=[4 * 20000 + 3, 4 * 900], tokens=[1, 1],
                   n_comp=[20000, 900], top_k=1024, n_heads=16),
    lambda: W.make("noalloc-b", seed=42, seq_lens=[4 * 5000], tokens=[3], top_k=256,
                   n_heads=16),
], ids=["two-sequences", "three-tokens"])
def test_noalloc_topk_matches_workspace_topk_twice(cuda_device, wl_fn):
    run = H.Run(wl_fn(), cuda_device)
    _check_twice(run, run.scores())


def _check_twice(run, scores):
    """Two calls in a row: each equal to csa_topk with a workspace, bit for
    bit, and to the oracle's selection on the same scores."""
    ref_idx, ref_n = run.topk(scores)
    torch.cuda.synchronize()
    H.check_topk_exact(run.wl, scores, ref_idx, ref_n)
    for _ in range(2):
        idx = torch.full_like(ref_idx, -9)
        n_sel = torch.full_like(ref_n, -9)
        assert _noalloc_topk(run, scores, idx, n_sel) == 0
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.equal(n_sel, ref_n)
        H.check_topk_exact(run.wl, scores, idx, n_sel)
    assert run.dev_status() == 0


def test_noalloc_topk_sixteen_tokens(cuda_device):
    # the largest call the fixed scratch takes: every token's state in use
    run = H.Run(W.make("noalloc-16", seed=44, seq_lens=[4 * 3000], tokens=[16], top_k=512,
                       n_heads=16), cuda_device)
    _check_twice(run, run.scores())


def test_noalloc_topk_all_equal_row(cuda_device):
    # w = 0: every score is 0, so every entry shares the threshold digit and
    # the per-warp staging overflows; the one-block path then re-reads the row
    wl = W.make("noalloc-flat", seed=45, seq_lens=[4 * 20000, 4 * 700], tokens=[1, 1],
                n_comp=[20000, 700], top_k=1000, n_heads=16)
    wl.w_idx[0].zero_()
    run = H.Run(wl, cuda_device)
    scores = run.scores()
    torch.cuda.synchronize()
    assert (scores.cpu()[0, :20000] == 0).all()
    _check_twice(run, scores)


def test_noalloc_topk_rejects_too_many_tokens(cuda_device):
    run = H.Run(W.make("noalloc-c", seed=43, seq_lens=[4 * 600], tokens=[17], top_k=64,
                       n_heads=16), cuda_device)
    scores = run.scores()
    idx = torch.empty(17, 64, dtype=torch.int32, device=cuda_device)
    n_sel = torch.empty(17, dtype=torch.int32, device=cuda_device)
    assert _noalloc_topk(run, scores, idx, n_sel) == 3   # CSA_ERR_CAPACITY


def test_noalloc_topk_rejects_top_k_above_2048(cuda_device):
    # the same code as csa_topk: the selection size is unsupported, not a
    # capacity limit of the fixed scratch
    run = H.Run(W.make("noalloc-d", seed=46, seq_lens=[4 * 3000], tokens=[1], top_k=64,
                       n_heads=16), cuda_device)
    scores = run.scores()
    run.prm.top_k = 2049
    idx = torch.empty(1, 2049, dtype=torch.int32, device=cuda_device)
    n_sel = torch.empty(1, dtype=torch.int32, device=cuda_device)
    assert _noalloc_topk(run, scores, idx, n_sel) == 2   # CSA_ERR_UNSUPPORTED
