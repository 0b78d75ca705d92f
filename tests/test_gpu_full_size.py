"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: sampled outputs checked one by one against the oracle, and
properties that hold at any size."""
import numpy as np
import pytest
import torch

import csa_workloads as W
import oracle
from sparse_compressed_kv_gb300 import csa
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def sub_run(run: H.Run, tokens):
    """The same caches with only `tokens` as queries (for gathering a sample)."""
    wl = run.wl
    sub = W.Workload(**{**wl.__dict__})
    sub.tok_seq = wl.tok_seq[tokens].clone()
    sub.tok_pos = wl.tok_pos[tokens].clone()
    sub.q_idx = wl.q_idx[tokens].clone()
    sub.w_idx = wl.w_idx[tokens].clone()
    sub.q = wl.q[tokens].clone()
    return H.Run(sub, run.dev)


def test_1m_context_decode(cuda_device):
    wl = W.ctx1m()
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    nv = 262144
    # sampled scores, plus every planted block
    H.check_scores(wl, sc, blocks_per_token=3000)
    planted = wl.planted.numpy()
    ref = np.array([oracle.block_score(W.bits(wl.q_idx[0]), wl.w_idx[0].numpy(),
                                       W.bits(wl.k_idx[s])) for s in planted])
    assert np.all(np.abs(sc.cpu().numpy()[0, planted] - ref) <=
                  H.score_tolerance(wl, 0, planted))
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    assert set(planted.tolist()) <= set(idx.cpu().numpy()[0].tolist())
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    assert int(kv_len[0]) == 1024 + 128
    out = run.attention(kv_buf, kv_len)
    err, cos = H.check_attention(wl, kv_buf, kv_len, out)
    fout, fidx = run.decode()
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    H.check_attention(wl, kv_buf, kv_len, fout)
    np.testing.assert_allclose(fout.cpu().numpy(), out.cpu().numpy(), rtol=0, atol=1e-5)
    rec = H.recall_vs_oracle(wl, idx, n_sel)
    assert rec >= 0.99, rec
    assert run.dev_status() == 0


def test_batch32_decode(cuda_device):
    wl = W.batch32()
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    H.check_scores(wl, sc, blocks_per_token=300)
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    out = run.attention(kv_buf, kv_len)
    H.check_attention(wl, kv_buf, kv_len, out)
    fout, fidx = run.decode()
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    H.check_attention(wl, kv_buf, kv_len, fout)
    np.testing.assert_allclose(fout.cpu().numpy(), out.cpu().numpy(), rtol=0, atol=1e-5)
    rec = H.recall_vs_oracle(wl, idx, n_sel, tokens=[0, 7, 31])
    assert rec >= 0.99, rec
    assert run.dev_status() == 0


def test_prefill_chunk(cuda_device):
    wl = W.prefill()
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    sample = [0, 1, 2, 3, 1001, 2046, 4093, 4095]
    H.check_scores(wl, sc, tokens=sample, blocks_per_token=400)
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel, tokens=sample)
    fout, fidx = run.decode()
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    # attention for the sampled tokens, from their own gathered rows
    sr = sub_run(run, sample)
    kv_buf, kv_len = H.gpu_rows(sr, idx[sample].contiguous(), n_sel[sample].contiguous())
    H.check_attention(sr.wl, kv_buf, kv_len, fout[sample])
    # every token sees exactly min(top_k, n_vis) blocks, all strictly preceding
    ns = n_sel.cpu().numpy()
    nvis = 65536 + np.arange(4096) // 4
    assert (ns == np.minimum(1024, nvis)).all()
    last = idx.cpu().numpy()[np.arange(4096), ns - 1]
    assert (last < nvis).all()
    assert run.dev_status() == 0


def test_64k_decode_loop(cuda_device):
    wl = W.ctx64k()
    gen = torch.Generator().manual_seed(1234)
    # max_comp_rows is the cache capacity: one workspace serves the whole loop
    run = H.Run(wl, cuda_device, max_comp_rows=int(wl.k_idx.shape[0]))
    for i in range(100):
        if i:
            W.ctx64k_step(wl, i, gen)
            # the step's new state goes to the device buffers in place
            run.d.tok_pos.copy_(wl.tok_pos)
            run.d.comp_off.copy_(wl.comp_off)
            run.d.swa_kv.copy_(wl.swa_kv)
            run.d.swa_first_pos.copy_(wl.swa_first_pos)
            run.d.q_idx.copy_(wl.q_idx)
            run.d.w_idx.copy_(wl.w_idx)
            run.d.q.copy_(wl.q)
        out, fidx = run.decode()
        if i == 1:
            # after one full round of calls every buffer size has been seen:
            # from here on nothing may allocate device memory ("1M-context
            # viability", falsifiable gate A4: memory_reserved flat across
            # decode steps); the library itself never allocates at all
            torch.cuda.synchronize()
            reserved0 = torch.cuda.memory_reserved()
            free0 = torch.cuda.mem_get_info()[0]
        if i % 9 == 0 or i == 99:
            sc = run.scores()
            idx, n_sel = run.topk(sc)
            H.check_topk_exact(wl, sc, idx, n_sel)
            assert torch.equal(fidx, idx)
            kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
            H.check_attention(wl, kv_buf, kv_len, out)
    assert run.dev_status() == 0
    # the pages' gate: reserved memory flat within 50 MB over the loop; and the
    # device's free memory moved by no more than what torch itself reserved
    grown = torch.cuda.memory_reserved() - reserved0
    assert abs(grown) <= 50 << 20
    assert abs((free0 - torch.cuda.mem_get_info()[0]) - grown) <= 2 << 20
