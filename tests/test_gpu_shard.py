"""Sharded single-sequence decode on one GPU (shards run one after another).

The merged selection must equal csa_topk on the whole sequence's scores, bit
for bit, and the combined output must match the f64 oracle on the rows the
selection names (and csa_decode's output) -- for one to several shards,
shards with no visible block, several query tokens, ties across shards and
sinks.
"""
import numpy as np
import pytest
import torch

import csa_workloads as W
from sparse_compressed_kv_gb300 import csa, shard
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def run_sharded(run: H.Run, G: int, rows: int = None, sinks=None):
    wl = run.wl
    n = int(wl.k_idx.shape[0]) if rows is None else rows
    bounds = shard.shard_bounds(n, G)
    shards = [shard.make_shard(run.layout, run.prm, bounds[g], bounds[g + 1], run.d.k_idx,
                               run.d.comp_kv) for g in range(G)]
    out, idx, n_sel = shard.decode_local(shards, run.layout, run.prm, run.d.q_idx, run.d.w_idx,
                                         run.d.q, run.status, sinks=sinks)
    torch.cuda.synchronize()
    return out, idx, n_sel


def check(run: H.Run, out, idx, n_sel, sinks=None):
    wl = run.wl
    sc = run.scores()
    ref_idx, ref_n = run.topk(sc)
    torch.cuda.synchronize()
    assert torch.equal(n_sel, ref_n)
    assert torch.equal(idx, ref_idx)
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    H.check_attention(wl, kv_buf, kv_len, out, sinks=sinks)
    fout, fidx = run.decode(sinks=sinks)
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    np.testing.assert_allclose(out.cpu().numpy(), fout.cpu().numpy(), rtol=0, atol=1e-5)
    assert run.dev_status() == 0


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8])
def test_sharded_decode_equals_single_device(cuda_device, G):
    wl = W.make("shard", seed=40 + G, seq_lens=[4 * 5000], n_comp=[5000], top_k=256, n_heads=64)
    run = H.Run(wl, cuda_device)
    out, idx, n_sel = run_sharded(run, G)
    check(run, out, idx, n_sel)


def test_shards_without_visible_blocks(cuda_device):
    # 3000 valid blocks in a 6000-row cache cut into 4 shards: the last two
    # hold no visible block (their candidate lists are empty)
    wl = W.make("shardcap", seed=50, seq_lens=[4 * 3000], n_comp=[3000], comp_capacity=[6000],
                top_k=512, n_heads=64)
    run = H.Run(wl, cuda_device, max_comp_rows=6000)
    out, idx, n_sel = run_sharded(run, 4, rows=6000)
    check(run, out, idx, n_sel)


def test_sharded_prefill_tokens(cuda_device):
    # 37 query tokens of one sequence, each seeing a different number of blocks
    wl = W.make("shardchunk", seed=51, seq_lens=[4 * 700], tokens=[37], top_k=128, n_heads=16)
    run = H.Run(wl, cuda_device)
    out, idx, n_sel = run_sharded(run, 3)
    check(run, out, idx, n_sel)


def test_sharded_ties_across_shards(cuda_device):
    # every key equal: every score ties, and the lowest block indices must win
    # wherever they sit
    wl = W.make("shardties", seed=52, seq_lens=[4 * 2000], n_comp=[2000], top_k=100, n_heads=16)
    wl.k_idx[:] = wl.k_idx[0]
    run = H.Run(wl, cuda_device)
    out, idx, n_sel = run_sharded(run, 4)
    assert idx[0].tolist() == list(range(100))
    check(run, out, idx, n_sel)


def test_sharded_with_sinks(cuda_device):
    wl = W.make("shardsink", seed=53, seq_lens=[4 * 4000], n_comp=[4000], top_k=512, n_heads=64)
    run = H.Run(wl, cuda_device)
    sinks = torch.randn(wl.n_heads, generator=torch.Generator().manual_seed(9)).to(cuda_device)
    out, idx, n_sel = run_sharded(run, 3, sinks=sinks)
    check(run, out, idx, n_sel, sinks=sinks)


def test_sharded_decode_1m(cuda_device):
    wl = W.ctx1m(seed=11)
    run = H.Run(wl, cuda_device)
    out, idx, n_sel = run_sharded(run, 4)
    sc = run.scores()
    ref_idx, ref_n = run.topk(sc)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx) and torch.equal(n_sel, ref_n)
    assert set(wl.planted.numpy().tolist()) <= set(idx.cpu().numpy()[0].tolist())
    fout, fidx = run.decode()
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    np.testing.assert_allclose(out.cpu().numpy(), fout.cpu().numpy(), rtol=0, atol=1e-5)
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    H.check_attention(wl, kv_buf, kv_len, out)
    assert run.dev_status() == 0


def test_merge_rejects_bad_arguments(cuda_device):
    dev = cuda_device
    z = torch.zeros(2, 1, 8, dtype=torch.int32, device=dev)
    f = torch.zeros(2, 1, 8, dtype=torch.float32, device=dev)
    n = torch.zeros(2, 1, dtype=torch.int32, device=dev)
    o = torch.zeros(1, 8, dtype=torch.int32, device=dev)
    o1 = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(csa.CsaError) as e:
        csa.csa_shard_merge([0, 10, 5], f, z, n, o, o1, z.clone(), n.clone(), st)   # bounds go down
    assert e.value.code == 1
    nine = torch.zeros(9, 1, 8, dtype=torch.int32, device=dev)
    with pytest.raises(csa.CsaError) as e:
        csa.csa_shard_merge(list(range(10)), nine.float(), nine, torch.zeros(9, 1, dtype=torch.int32,
                            device=dev), o, o1, nine.clone(), torch.zeros(9, 1, dtype=torch.int32,
                            device=dev), st)
    assert e.value.code == 2   # more than 8 shards
