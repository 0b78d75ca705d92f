"""FP4 indexer keys on the GPU (through the C ABI).

The quantizer must match the oracle's MXFP4 bytes exactly; the FP4 scoring
path must equal the bf16 indexer on the dequantized keys, within the same
tolerance as the bf16 path (the oracle scores the dequantized keys in f64);
csa_decode_fp4 must select exactly what csa_topk selects on those scores.
"""
import dataclasses

import numpy as np
import pytest
import torch

import csa_workloads as W
import oracle
from sparse_compressed_kv_gb300 import csa
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def gpu_rows(k_idx_dev: torch.Tensor) -> torch.Tensor:
    rows = torch.full((k_idx_dev.shape[0], csa.FP4_ROW), 0xAB, dtype=torch.uint8,
                      device=k_idx_dev.device)
    csa.csa_fp4_quantize_keys(k_idx_dev, rows)
    return rows


def dequantized(wl: W.Workload) -> W.Workload:
    """The workload with its keys replaced by their MXFP4 round trip."""
    kd = oracle.fp4_dequantize(oracle.fp4_quantize(W.bits(wl.k_idx)))
    return dataclasses.replace(wl, k_idx=torch.from_numpy(kd.view(np.int16)).view(torch.bfloat16))


def fp4_scores(run: H.Run, rows: torch.Tensor) -> torch.Tensor:
    sc = torch.full((run.T, run.ld), float("nan"), dtype=torch.float32, device=run.dev)
    csa.csa_indexer_scores_fp4(run.layout, run.prm, run.d.q_idx, run.d.w_idx, rows, sc,
                               run.status)
    return sc


def fp4_decode(run: H.Run, rows: torch.Tensor):
    out = torch.full((run.T, run.wl.n_heads, run.wl.hd), float("nan"), dtype=torch.float32,
                     device=run.dev)
    idx = torch.full((run.T, run.wl.top_k), -7, dtype=torch.int32, device=run.dev)
    csa.csa_decode_fp4(run.layout, run.prm, run.d.q_idx, run.d.w_idx, rows, run.d.comp_kv,
                       run.d.q, out, run.status, run.ws, idx_out=idx)
    return out, idx


def test_fp4_quantizer_bit_exact(cuda_device):
    # N(0,1) keys at scales from 2^-40 to 2^40, bf16 subnormals, zero and
    # signed-zero blocks, exact grid midpoints, and the largest bf16 values
    rng = np.random.default_rng(21)
    R = 20000
    x = rng.standard_normal((R, 128)) * np.exp2(rng.uniform(-40, 40, (R, 1)))
    x[0] = 0.0
    x[1, :64] = -0.0
    x[2] = rng.standard_normal(128) * 2.0 ** -130            # bf16 subnormals
    x[3, :] = 4.0
    x[3, 1:8] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]     # midpoints: ties to even
    x[4] = rng.choice([-1.0, 1.0], 128) * 3.0e38             # near the largest bf16
    kb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    want = oracle.fp4_quantize(W.bits(kb))
    got = gpu_rows(kb.to(cuda_device)).cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:4].tolist()}"


@pytest.mark.parametrize("name", ["tiny", "64k"])
def test_fp4_indexer_matches_oracle_on_dequantized_keys(cuda_device, name):
    wl = W.tiny(seed=5) if name == "tiny" else W.ctx64k(seed=5)
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    sc = fp4_scores(run, rows)
    H.check_scores(dequantized(wl), sc, blocks_per_token=None if name == "tiny" else 500)
    assert run.dev_status() == 0


def test_fp4_decode_selects_exactly_topk_of_its_scores(cuda_device):
    wl = W.tiny(seed=6)
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    sc = fp4_scores(run, rows)
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    out, fidx = fp4_decode(run, rows)
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    H.check_attention(wl, kv_buf, kv_len, out)
    assert run.dev_status() == 0


def test_fp4_decode_1m(cuda_device):
    wl = W.ctx1m(seed=7)
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    # the cache itself: a sample of rows against the oracle's bytes
    sample = np.random.default_rng(7).choice(wl.k_idx.shape[0], 2048, replace=False)
    want = oracle.fp4_quantize(W.bits(wl.k_idx[torch.from_numpy(sample)]))
    assert np.array_equal(rows[torch.from_numpy(sample).to(cuda_device)].cpu().numpy(), want)
    sc = fp4_scores(run, rows)
    wd = dequantized(wl)
    H.check_scores(wd, sc, blocks_per_token=300)
    out, fidx = fp4_decode(run, rows)
    idx, n_sel = run.topk(sc)
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    H.check_topk_exact(wd, sc, idx, n_sel)
    planted = set(wl.planted.numpy().tolist())
    assert planted <= set(fidx.cpu().numpy()[0].tolist())
    # how much of the bf16 selection survives FP4 keys (reported, not a parity bar)
    _, bidx = run.decode()
    torch.cuda.synchronize()
    common = len(set(bidx.cpu().numpy()[0].tolist()) & set(fidx.cpu().numpy()[0].tolist()))
    print(f"fp4 vs bf16 selection overlap at 1M: {common}/{wl.top_k}")
    assert run.dev_status() == 0


@pytest.mark.parametrize("top_k", [8, 16])
def test_fp4_many_tokens_per_cta(cuda_device, top_k):
    # ~500 short sequences of 1..3 key units each: every CTA's range crosses
    # several token boundaries, so each token's queries are loaded and
    # converted ahead into alternating buffers (first, second and reused
    # buffers); tokens with no more visible blocks than top_k take the
    # select-everything path between them
    rng = np.random.default_rng(17)
    B = 480
    n_comp = rng.integers(5, 97, B).tolist()
    seq_lens = [4 * n + int(rng.integers(0, 4)) for n in n_comp]
    wl = W.make("fp4_many", seed=18, seq_lens=seq_lens, tokens=[1] * B, n_comp=n_comp,
                top_k=top_k, n_heads=16, swa_cap=128)
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    sc = fp4_scores(run, rows)
    H.check_scores(dequantized(wl), sc)
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    out, fidx = fp4_decode(run, rows)
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    toks = list(range(0, B, 37))
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    H.check_attention(wl, kv_buf, kv_len, out, tokens=toks)
    assert run.dev_status() == 0


@pytest.mark.parametrize("q_exp", [-20, 20])
def test_fp4_scores_query_scale(cuda_device, q_exp):
    # the query scaled by an exact power of two far from 1: the f16 queries
    # of the FP4 path must keep their precision (no f16 subnormals, no
    # overflow), so the scores stay within the bound against the oracle
    wl = W.tiny(seed=9)
    scaled = (wl.q_idx.float() * 2.0 ** q_exp).to(torch.bfloat16)
    assert torch.equal(scaled.float(), wl.q_idx.float() * 2.0 ** q_exp)   # exact in bf16
    wl = dataclasses.replace(wl, q_idx=scaled)
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    sc = fp4_scores(run, rows)
    H.check_scores(dequantized(wl), sc)
    assert run.dev_status() == 0


@pytest.mark.parametrize("q_exp", [0, -20])
def test_fp4_prefill_chunk(cuda_device, q_exp):
    # 16 query tokens of one sequence (a prefill chunk): FP4 keys go through
    # the chunk indexer (converter warps, bf16 expansion) and the separate
    # top-k instead of the decode kernel
    wl = W.make("fp4_chunk", seed=23, seq_lens=[8192], tokens=[16], n_comp=[2051], top_k=64,
                n_heads=16, swa_cap=144)
    if q_exp:
        wl = dataclasses.replace(wl, q_idx=(wl.q_idx.float() * 2.0 ** q_exp).to(torch.bfloat16))
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    sc = fp4_scores(run, rows)
    H.check_scores(dequantized(wl), sc, blocks_per_token=300)
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    out, fidx = fp4_decode(run, rows)
    torch.cuda.synchronize()
    assert torch.equal(fidx, idx)
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    H.check_attention(wl, kv_buf, kv_len, out, tokens=[0, 7, 15])
    assert run.dev_status() == 0


def test_fp4_selection_recall_against_the_bf16_oracle(cuda_device):
    # Recall is the measure of the FP4 cache ("parity is recall vs the bf16
    # oracle"): the FP4 step's selection against the oracle's f64 selection
    # on the bf16 keys.  On the synthetic 1M layer (Gaussian keys, whose top
    # 1,024 of 262,144 sit in a dense tail) MXFP4's rounding moves about 15%
    # of the cut; the 32 planted blocks, far above it, are always kept.  The
    # bound below pins that behaviour (a broken expansion or scale drops far
    # lower and loses planted blocks).
    wl = W.ctx1m(seed=5)
    run = H.Run(wl, cuda_device)
    rows = gpu_rows(run.d.k_idx)
    _, idx = fp4_decode(run, rows)
    torch.cuda.synchronize()
    assert run.dev_status() == 0
    got = set(idx[0].cpu().numpy().tolist()) - {-1}
    ref_sc = H._scores_full(wl, 0)
    nv = oracle.n_vis(int(wl.comp_off[1] - wl.comp_off[0]), int(wl.tok_pos[0]), wl.ratio)
    ref_idx, ref_n = oracle.topk(ref_sc[:nv], wl.top_k)
    ref = set(ref_idx[:ref_n].tolist())
    recall = len(ref & got) / len(ref)
    assert len(got) == wl.top_k
    assert recall >= 0.80, recall
    assert set(wl.planted.tolist()) <= got
