"""GPU parity of HCA decode (dense attention over every visible compressed
row plus the window) against the oracle's HCA step."""
import numpy as np
import pytest
import torch

import csa_workloads as W
import oracle
from sparse_compressed_kv_gb300 import csa
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def run_hca(wl, device, sinks=None):
    d = wl.to(device)
    layout = csa.Layout(d.tok_seq, d.tok_pos, d.comp_off, d.swa_kv, d.swa_first_pos,
                        max_comp_rows=max(1, wl.max_comp_rows),
                        total_comp_rows=int(wl.comp_kv.shape[0]), swa_cap=wl.swa_cap)
    prm = csa.params(wl.n_heads, 1, wl.window, wl.ratio, wl.scale)
    ws = csa.hca_workspace(layout, prm)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    out = torch.full((wl.num_tokens, wl.n_heads, wl.hd), float("nan"), device=device)
    csa.csa_hca_decode(layout, prm, d.comp_kv, d.q, out, st, ws, sinks=sinks)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


def oracle_hca(wl, sinks=None):
    return oracle.hca_decode(W.bits(wl.comp_kv), W.bits(wl.swa_kv), W.bits(wl.q),
                             wl.tok_seq.numpy(), wl.tok_pos.numpy(), wl.comp_off.numpy(),
                             wl.swa_first_pos.numpy(), window=wl.window, ratio=wl.ratio,
                             scale=wl.scale, sinks=sinks)


def test_hca_ragged_small(cuda_device):
    wl = W.make("hca", seed=31, seq_lens=[128 * 300 + 5, 128 * 3 + 127, 60], tokens=[1, 2, 1],
                n_comp=[300, 4, 0], ratio=128, n_heads=32, swa_cap=160, top_k=1)
    out = run_hca(wl, cuda_device)
    ref, _ = oracle_hca(wl)
    err = np.abs(out.cpu().numpy() - ref).max()
    assert err <= H.ATTN_ATOL, err


def test_hca_1m_context(cuda_device):
    wl = W.hca1m()
    out = run_hca(wl, cuda_device)
    ref, kv_len = oracle_hca(wl)
    assert kv_len[0] == 8192 + 128
    err = np.abs(out.cpu().numpy() - ref).max()
    assert err <= H.ATTN_ATOL, err


def test_hca_with_sinks(cuda_device):
    wl = W.make("hcas", seed=32, seq_lens=[128 * 64 + 9], n_comp=[64], ratio=128, n_heads=16,
                top_k=1)
    sinks = torch.randn(16, generator=torch.Generator().manual_seed(2))
    out = run_hca(wl, cuda_device, sinks=sinks.to(cuda_device))
    ref, _ = oracle_hca(wl, sinks=sinks.numpy())
    assert np.abs(out.cpu().numpy() - ref).max() <= H.ATTN_ATOL
