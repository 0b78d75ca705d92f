"""GPU parity: every C-ABI entry point against the CPU oracle on seeded inputs.

Bars: indexer scores within relative 1e-4 of sum_h |w_h| ReLU(q_h.k) (plus an
f32 floor); top-k bit-exact against the oracle's selection on the GPU's own
scores; gather bit-exact; attention max-abs 2e-3 against the f64 oracle on the
rows the GPU attended; the fused step bit-identical to the unfused chain's
selection.
"""
import numpy as np
import pytest
import torch

import csa_workloads as W
import oracle
from sparse_compressed_kv_gb300 import csa
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def full_chain(run: H.Run, check_recall=True):
    """Unfused chain with a parity check at every step, then the fused step."""
    wl = run.wl
    sc = run.scores()
    H.check_scores(wl, sc)
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
    out = run.attention(kv_buf, kv_len)
    err, cos = H.check_attention(wl, kv_buf, kv_len, out)
    fout, fidx = run.decode()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(fidx.cpu().numpy(), idx.cpu().numpy())
    # the same rows: the fused output against the oracle on them, and against
    # the unfused one (the fused path starts the window rows at a multiple of
    # four slots, so chunk boundaries, and f32 rounding, may differ slightly)
    H.check_attention(wl, kv_buf, kv_len, fout)
    np.testing.assert_allclose(fout.cpu().numpy(), out.cpu().numpy(), rtol=0, atol=1e-5)
    assert run.dev_status() == 0
    rec = H.recall_vs_oracle(wl, idx, n_sel) if check_recall else None
    return err, cos, rec


def test_tiny(cuda_device):
    err, cos, rec = full_chain(H.Run(W.tiny(), cuda_device))
    assert cos > 0.9999 and rec >= 0.95


def test_ragged_multi_sequence(cuda_device):
    # three sequences, 1-2 tokens each; one short context (window clipped at 0),
    # n_comp not a multiple of the 128-key tile
    wl = W.make("ragged", seed=21, seq_lens=[4 * 300 + 3, 90, 4 * 1000 + 1], tokens=[1, 2, 1],
                n_comp=[300, 22, 1000], top_k=64, n_heads=32, swa_cap=160)
    full_chain(H.Run(wl, cuda_device))


def test_grouped_tokens_single_sequence(cuda_device):
    # one sequence, 37 tokens: the indexer groups 4 tokens per MMA (N = 256),
    # the last group is partial; every token has its own causal cut
    wl = W.make("chunk", seed=22, seq_lens=[4 * 700], tokens=[37], top_k=128, n_heads=16,
                swa_cap=256)
    full_chain(H.Run(wl, cuda_device))


SHAPE_CASES = {
    # the largest top_k the library takes, two sequences
    "topk2048": lambda: W.make("k2048", seed=41, seq_lens=[4 * 20000, 4 * 9000],
                               n_comp=[20000, 9000], top_k=2048, n_heads=64),
    # another compression ratio and a shorter window (visibility and window
    # arithmetic away from ratio 4 / window 128)
    "ratio8_window64": lambda: W.make("r8w64", seed=42, seq_lens=[8 * 3000 + 5, 8 * 700],
                                      tokens=[1, 2], n_comp=[3000, 700], top_k=256, n_heads=32,
                                      ratio=8, window=64, swa_cap=96),
    # two head groups per token
    "heads128": lambda: W.make("h128", seed=43, seq_lens=[4 * 6000, 4 * 2500],
                               n_comp=[6000, 2500], top_k=512, n_heads=128),
}


@pytest.mark.parametrize("name", list(SHAPE_CASES))
def test_other_shapes(cuda_device, name):
    full_chain(H.Run(SHAPE_CASES[name](), cuda_device))


def test_topk_covers_everything_and_empty(cuda_device):
    # token 0: position 2 -> no visible block (window only)
    # token 1: top_k >= n_vis -> every visible block, attention is dense
    wl = W.make("edges", seed=23, seq_lens=[2, 4 * 50 + 2], tokens=[1, 1], n_comp=[0, 50],
                top_k=64, n_heads=16, swa_cap=128)
    run = H.Run(wl, cuda_device)
    full_chain(run, check_recall=False)
    _, idx = run.decode()
    idx = idx.cpu().numpy()
    assert (idx[0] == -1).all()
    assert list(idx[1, :50]) == list(range(50)) and (idx[1, 50:] == -1).all()


def test_ties_resolve_to_lowest_index(cuda_device):
    # duplicated keys give bit-identical scores: the cut falls inside a tie
    wl = W.make("ties", seed=24, seq_lens=[4 * 2000], n_comp=[2000], top_k=100, n_heads=16)
    base = wl.k_idx[:40].clone()
    for rep in range(50):
        wl.k_idx[40 * rep:40 * rep + 40] = base
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)
    assert run.dev_status() == 0


def test_all_equal_scores_overflow_path(cuda_device):
    # w = 0: every score is 0, every block ties, and the candidate list
    # overflows its capacity: the resolver falls back to scanning the row
    wl = W.make("flat", seed=25, seq_lens=[4 * 20000], n_comp=[20000], top_k=1000, n_heads=16)
    wl.w_idx.zero_()
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    assert (sc.cpu()[0, :20000] == 0).all()
    idx, n_sel = run.topk(sc)
    assert list(idx.cpu().numpy()[0]) == list(range(1000))
    H.check_topk_exact(wl, sc, idx, n_sel)


def test_negative_and_signed_zero_scores(cuda_device):
    wl = W.make("signs", seed=26, seq_lens=[4 * 3000], n_comp=[3000], top_k=300, n_heads=16)
    wl.w_idx.copy_(-wl.w_idx.abs())        # every score <= 0, many exactly -0.0 or 0.0
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    idx, n_sel = run.topk(sc)
    H.check_topk_exact(wl, sc, idx, n_sel)


def test_determinism_and_workspace_reuse(cuda_device):
    run = H.Run(W.make("det", seed=27, seq_lens=[4 * 5000], n_comp=[5000], top_k=256,
                       n_heads=64), cuda_device)
    o1, i1 = run.decode()
    for _ in range(3):
        o2, i2 = run.decode()
    torch.cuda.synchronize()
    assert torch.equal(i1, i2)
    assert torch.equal(o1, o2)
    assert run.dev_status() == 0


def test_causality_perturbation(cuda_device):
    wl = W.make("causal", seed=28, seq_lens=[4 * 600 + 1], n_comp=[600], comp_capacity=[700],
                top_k=64, n_heads=16, swa_cap=256)
    run = H.Run(wl, cuda_device)
    o1, i1 = run.decode()
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(5)
    wl.k_idx[600:] = W.bf16_normal(g, 100, wl.ihd) * 100
    wl.comp_kv[600:] = W.bf16_normal(g, 100, wl.hd) * 100
    p = int(wl.tok_pos[0])
    inside = {x % wl.swa_cap for x in range(p - wl.window + 1, p + 1)}
    for slot in range(wl.swa_cap):
        if slot not in inside:
            wl.swa_kv[0, slot] = W.bf16_normal(g, wl.hd) * 100
    wl.comp_off[1] = 700       # the extra rows exist in the cache but are not visible
    run2 = H.Run(wl, cuda_device)
    o2, i2 = run2.decode()
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(o1, o2)


def test_device_status_bits(cuda_device):
    wl = W.make("status", seed=29, seq_lens=[4 * 100], n_comp=[100], top_k=8, n_heads=16)
    run = H.Run(wl, cuda_device)
    idx = torch.tensor([[0, 5, 150, -1, -1, -1, -1, -1]], dtype=torch.int32, device=cuda_device)
    n_sel = torch.tensor([3], dtype=torch.int32, device=cuda_device)
    kv_buf, kv_len = run.gather(idx, n_sel)
    st = run.dev_status()
    assert st & csa.DEV_BAD_INDEX
    assert (kv_buf[0, 2].float() == 0).all()            # the bad row is zeroed, not clamped
    np.testing.assert_array_equal(W.bits(kv_buf[0, 1]), W.bits(wl.comp_kv[5]))
    # a window row the ring no longer holds
    run.status.zero_()
    run.d.swa_first_pos[0] = int(wl.tok_pos[0])          # only the current position resident
    run.gather(torch.tensor([[0] + [-1] * 7], dtype=torch.int32, device=cuda_device),
               torch.tensor([1], dtype=torch.int32, device=cuda_device))
    assert run.dev_status() & csa.DEV_MISSING_SWA


SINK_CASES = {
    # 3 splits of 64 rows per token, merged by the combine kernel (the sink
    # in its denominator)
    "tiny": lambda: W.tiny(seed=3),
    # 18 splits
    "wide": lambda: W.make("sinkwide", seed=5, seq_lens=[4 * 5000], n_comp=[5000], top_k=1024,
                           n_heads=16),
    # 160 tokens of 64 heads: one split each, normalised (sink included) in
    # the attention kernel itself
    "onesplit": lambda: W.make("sinkone", seed=6, seq_lens=[4 * 600], tokens=[160], top_k=128,
                               n_heads=64),
    # a full and a partial head group (64 + 16 heads)
    "heads80": lambda: W.make("sink80", seed=7, seq_lens=[4 * 900, 4 * 300], tokens=[2, 1],
                              top_k=256, n_heads=80),
    # two full head groups
    "heads128": lambda: W.make("sink128", seed=8, seq_lens=[4 * 1500], top_k=512, n_heads=128),
}


@pytest.mark.parametrize("name", list(SINK_CASES))
def test_sink_attention(cuda_device, name):
    wl = SINK_CASES[name]()
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    idx, n_sel = run.topk(sc)
    kv_buf, kv_len = run.gather(idx, n_sel)
    sinks = torch.randn(wl.n_heads, generator=torch.Generator().manual_seed(4)).to(cuda_device)
    out = run.attention(kv_buf, kv_len, sinks=sinks)
    H.check_attention(wl, kv_buf, kv_len, out, sinks=sinks)
    fout, _ = run.decode(sinks=sinks)
    H.check_attention(wl, kv_buf, kv_len, fout, sinks=sinks)
    np.testing.assert_allclose(fout.cpu().numpy(), out.cpu().numpy(), rtol=0, atol=1e-5)


def test_host_errors_on_gpu(cuda_device):
    run = H.Run(W.tiny(), cuda_device)
    small = torch.zeros(16, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(csa.CsaError) as e:
        csa.csa_decode(run.layout, run.prm, run.d.q_idx, run.d.w_idx, run.d.k_idx,
                       run.d.comp_kv, run.d.q, torch.empty(1, 16, 512, device=cuda_device),
                       run.status, small)
    assert e.value.code == 7   # CSA_ERR_WORKSPACE
    bad = csa.params(16, 64, hd=256)
    with pytest.raises(csa.CsaError) as e:
        csa.csa_indexer_scores(run.layout, bad, run.d.q_idx, run.d.w_idx, run.d.k_idx,
                               torch.empty(1, 256, device=cuda_device), run.status)
    assert e.value.code == 2   # CSA_ERR_UNSUPPORTED


def _monotone():
    # every head's query is one direction v and block s's key is 2^(s/256) v:
    # scores grow with the block index, so the whole selection sits in the
    # last key range and the candidates of the other ranges cannot prove it
    # (the selection then comes from the whole score row)
    wl = W.make("monotone", seed=30, seq_lens=[4 * 2000], n_comp=[2000], top_k=100, n_heads=16)
    g = torch.Generator().manual_seed(7)
    v = torch.randn(wl.ihd, generator=g)
    v = v / v.norm()
    wl.q_idx[0] = v.to(torch.bfloat16)[None, :].expand(wl.n_ih, -1)
    wl.w_idx.fill_(1.0 / 64)
    c = torch.pow(2.0, torch.arange(2000, dtype=torch.float32) / 256.0)
    wl.k_idx[:2000] = (c[:, None] * v[None, :]).to(torch.bfloat16)
    return wl


def _ties():
    wl = W.make("ties2", seed=31, seq_lens=[4 * 2000], n_comp=[2000], top_k=100, n_heads=16)
    base = wl.k_idx[:40].clone()
    for rep in range(50):
        wl.k_idx[40 * rep:40 * rep + 40] = base
    return wl


def _flat():
    wl = W.make("flat2", seed=32, seq_lens=[4 * 20000], n_comp=[20000], top_k=1000, n_heads=16)
    wl.w_idx.zero_()
    return wl


def _one_bin(name, seed, n, k):
    # every score in [1.27, 1.47], inside one first-level radix bin (a quarter
    # octave): the threshold bin holds all n candidates, so the cut is
    # settled entirely by the digits below the first
    wl = W.make(name, seed=seed, seq_lens=[4 * n], n_comp=[n], top_k=k, n_heads=16)
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(wl.ihd, generator=g)
    v = v / v.norm()
    wl.q_idx[0] = v.to(torch.bfloat16)[None, :].expand(wl.n_ih, -1)
    wl.w_idx.fill_(1.0 / wl.n_ih)
    a = 1.27 + 0.2 * torch.rand(n, generator=g)
    wl.k_idx[:n] = (a[:, None] * v[None, :]).to(torch.bfloat16)
    return wl


def _signs():
    wl = W.make("signs2", seed=33, seq_lens=[4 * 3000], n_comp=[3000], top_k=300, n_heads=16)
    wl.w_idx.copy_(-wl.w_idx.abs())
    return wl


INDEXER_TOPK_CASES = {
    "tiny": lambda: W.tiny(seed=9),
    "ragged": lambda: W.make("ragged2", seed=34, seq_lens=[4 * 300 + 3, 90, 4 * 1000 + 1],
                             tokens=[1, 2, 1], n_comp=[300, 22, 1000], top_k=64, n_heads=16,
                             swa_cap=160),
    "batch": lambda: W.make("batch6", seed=35, seq_lens=[4 * n for n in
                                                         [5000, 12000, 800, 30000, 2500, 64]],
                            n_comp=[5000, 12000, 800, 30000, 2500, 64], top_k=512, n_heads=16),
    "chunk": lambda: W.make("chunk2", seed=36, seq_lens=[4 * 700], tokens=[37], top_k=128,
                            n_heads=16, swa_cap=256),
    "ties": _ties, "flat": _flat, "signs": _signs, "monotone": _monotone,
    "one_bin_2k": lambda: _one_bin("onebin1", 37, 2040, 1000),
    "one_bin_10k": lambda: _one_bin("onebin2", 38, 10000, 1024),
}


@pytest.mark.parametrize("name", list(INDEXER_TOPK_CASES))
def test_indexer_topk_equals_topk_on_the_scores(cuda_device, name):
    """csa_indexer_topk (the selection folded into the indexer for decode
    batches) selects exactly what csa_topk selects on csa_indexer_scores'
    scores, which is the oracle's selection on those scores, and again on a
    second call with the same workspace."""
    wl = INDEXER_TOPK_CASES[name]()
    run = H.Run(wl, cuda_device)
    sc = run.scores()
    ref_idx, ref_n = run.topk(sc)
    H.check_topk_exact(wl, sc, ref_idx, ref_n)
    for _ in range(2):
        idx, n_sel = run.indexer_topk()
        torch.cuda.synchronize()
        assert torch.equal(n_sel, ref_n)
        assert torch.equal(idx, ref_idx)
    if name.startswith("one_bin"):
        s = sc.cpu()[0, :wl.total_comp_rows]
        assert float(s.min()) > 1.25 and float(s.max()) < 1.5
    if name == "monotone":
        # the selection is the tail of the cache (rounding may swap neighbours)
        assert idx.cpu().numpy()[0].min() >= 1800
    assert run.dev_status() == 0


@pytest.mark.parametrize("B", [480, 700, 1100])
def test_many_short_sequences(cuda_device, B):
    # B sequences of 20..60 blocks, one token each: 480 keeps the selection
    # folded into the decode indexer with several tokens per CTA, 700 is past
    # the folded selection's token limit (decode indexer + separate top-k),
    # 1100 past the decode indexer's (the chunk indexer, one token per tile)
    rng = np.random.default_rng(B)
    n_comp = rng.integers(20, 61, B).tolist()
    seq_lens = [4 * n + int(rng.integers(0, 4)) for n in n_comp]
    wl = W.make(f"many{B}", seed=B, seq_lens=seq_lens, tokens=[1] * B, n_comp=n_comp, top_k=16,
                n_heads=16)
    full_chain(H.Run(wl, cuda_device), check_recall=False)


def test_layout_rewritten_by_a_kernel_right_before(cuda_device):
    # the layout is read as a kernel starts; a torch kernel that rewrites it
    # just before the call (same stream, no synchronisation, no programmatic
    # launch) has finished by then: each call must see the shrunken cache
    wl = W.make("devlayout", seed=44, seq_lens=[4 * 3000], n_comp=[3000], top_k=256, n_heads=16)
    run = H.Run(wl, cuda_device)
    for k in range(1, 5):
        run.d.comp_off[1:].sub_(37)          # a device kernel on the current stream
        out, fidx = run.decode()
        wl.comp_off[1:] -= 37                # the oracle's view of the same layout
        sc = run.scores()
        idx, n_sel = run.topk(sc)
        H.check_topk_exact(wl, sc, idx, n_sel)
        torch.cuda.synchronize()
        assert int(n_sel[0]) == 256 and torch.equal(fidx, idx)
        assert int(idx[0].max()) < 3000 - 37 * k
        kv_buf, kv_len = H.gpu_rows(run, idx, n_sel)
        H.check_attention(wl, kv_buf, kv_len, out)
    assert run.dev_status() == 0
