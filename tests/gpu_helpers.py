"""Shared pieces of the GPU parity tests: run each C-ABI entry point on a
seeded workload and compare with the CPU oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import csa_workloads as W
import oracle
from sparse_compressed_kv_gb300 import csa

# Attention: max-abs error against the f64 oracle on identical rows, for N(0,1)
# inputs with f32 accumulation (the stated correctness criterion).
ATTN_ATOL = 2e-3
# Indexer: relative 1e-4 of sum_h |w_h| ReLU(q_h.k) (the stated criterion), plus
# an f32 rounding floor that only matters when every ReLU term vanishes:
# 2^-22 of sum_h |w_h| sum_d |q_hd k_d| (an f32 dot of 128 exact products).
SCORE_RTOL = 1e-4
SCORE_FLOOR = 2.0 ** -22


def bits_to_f64(b):
    return (np.asarray(b).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# Canary guard bands: every buffer a library call writes is allocated with
# GUARD bytes of a known pattern on each side, checked after the call.  A
# write just past (or before) an output, the workspace included, fails the
# test even when the values inside the buffer are right.
GUARD = 4096
GUARD_BYTE = 0xA5


class Guarded:
    """A device tensor of `shape` with guard bands on both sides (offsets keep
    the 256-byte alignment of the allocation)."""

    def __init__(self, shape, dtype, device, fill=None):
        elem = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        g = GUARD // elem
        self.raw = torch.empty(n + 2 * g, dtype=dtype, device=device)
        self.raw.view(torch.uint8).fill_(GUARD_BYTE)
        self.t = self.raw[g:g + n].view(*shape)
        if fill is not None:
            self.t.fill_(fill)

    def intact(self) -> bool:
        b = self.raw.view(torch.uint8)
        return bool((b[:GUARD] == GUARD_BYTE).all()) and bool((b[-GUARD:] == GUARD_BYTE).all())


class Run:
    """One workload on the GPU, with its layout, params and workspace."""

    def __init__(self, wl: W.Workload, device, max_comp_rows=None):
        self.wl = wl
        self.dev = device
        d = wl.to(device)
        self.d = d
        mcr = max(1, wl.max_comp_rows if max_comp_rows is None else max_comp_rows)
        self.layout = csa.Layout(d.tok_seq, d.tok_pos, d.comp_off, d.swa_kv, d.swa_first_pos,
                                 max_comp_rows=mcr,
                                 total_comp_rows=int(wl.k_idx.shape[0]), swa_cap=wl.swa_cap)
        self.prm = csa.params(wl.n_heads, wl.top_k, wl.window, wl.ratio, wl.scale)
        self.guards = []
        self.ws = self.buf((csa.csa_workspace_size(self.layout, self.prm),), torch.uint8, 0)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.T = wl.num_tokens
        self.ld = mcr

    def buf(self, shape, dtype, fill):
        g = Guarded(shape, dtype, self.dev, fill)
        self.guards.append(g)
        return g.t

    def check_guards(self):
        torch.cuda.synchronize()
        bad = [i for i, g in enumerate(self.guards) if not g.intact()]
        assert not bad, f"guard band overwritten around buffer(s) {bad}"
        # forget output buffers (keep the workspace): memory stays bounded
        self.guards = self.guards[:1]

    # -- oracle-side views
    def n_vis(self):
        out = []
        for t in range(self.T):
            b = int(self.wl.tok_seq[t])
            n_comp = int(self.wl.comp_off[b + 1] - self.wl.comp_off[b])
            out.append(oracle.n_vis(n_comp, int(self.wl.tok_pos[t]), self.wl.ratio))
        return out

    # -- GPU calls (each checks the guard bands of what it wrote)
    def scores(self):
        sc = self.buf((self.T, self.ld), torch.float32, float("nan"))
        csa.csa_indexer_scores(self.layout, self.prm, self.d.q_idx, self.d.w_idx, self.d.k_idx,
                               sc, self.status)
        self.check_guards()
        return sc

    def topk(self, scores):
        idx = self.buf((self.T, self.wl.top_k), torch.int32, -7)
        n_sel = self.buf((self.T,), torch.int32, -7)
        csa.csa_topk(self.layout, self.prm, scores, idx, n_sel, self.status, self.ws)
        self.check_guards()
        return idx, n_sel

    def indexer_topk(self):
        idx = self.buf((self.T, self.wl.top_k), torch.int32, -7)
        n_sel = self.buf((self.T,), torch.int32, -7)
        csa.csa_indexer_topk(self.layout, self.prm, self.d.q_idx, self.d.w_idx, self.d.k_idx, idx,
                             n_sel, self.status, self.ws)
        self.check_guards()
        return idx, n_sel

    def gather(self, idx, n_sel):
        rows = self.wl.top_k + self.wl.window
        kv_buf = self.buf((self.T, rows, self.wl.hd), torch.bfloat16, 0)
        kv_len = self.buf((self.T,), torch.int32, -7)
        csa.csa_gather_mixed(self.layout, self.prm, idx, n_sel, self.d.comp_kv, kv_buf, kv_len,
                             self.status)
        self.check_guards()
        return kv_buf, kv_len

    def attention(self, kv_buf, kv_len, sinks=None):
        out = self.buf((self.T, self.wl.n_heads, self.wl.hd), torch.float32, float("nan"))
        csa.csa_sparse_mqa_decode(self.prm, self.d.q, kv_buf, kv_len, out, self.status, self.ws,
                                  sinks=sinks)
        self.check_guards()
        return out

    def decode(self, sinks=None):
        out = self.buf((self.T, self.wl.n_heads, self.wl.hd), torch.float32, float("nan"))
        idx = self.buf((self.T, self.wl.top_k), torch.int32, -7)
        csa.csa_decode(self.layout, self.prm, self.d.q_idx, self.d.w_idx, self.d.k_idx,
                       self.d.comp_kv, self.d.q, out, self.status, self.ws, idx_out=idx,
                       sinks=sinks)
        self.check_guards()
        return out, idx

    def dev_status(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def score_tolerance(wl: W.Workload, t: int, blocks: np.ndarray) -> np.ndarray:
    """Per-block tolerance of the indexer score of token t (see SCORE_RTOL)."""
    b = int(wl.tok_seq[t])
    off = int(wl.comp_off[b])
    q = bits_to_f64(W.bits(wl.q_idx[t]))                        # [64, 128]
    k = bits_to_f64(W.bits(wl.k_idx[off + blocks]))             # [n, 128]
    w = np.abs(wl.w_idx[t].numpy().astype(np.float64))         # [64]
    dots = k @ q.T                                              # [n, 64]
    rel = (np.maximum(dots, 0.0) * w).sum(1)
    absd = (np.abs(k) @ np.abs(q).T * w).sum(1)
    return SCORE_RTOL * rel + SCORE_FLOOR * absd


def check_scores(wl, gpu_scores: torch.Tensor, tokens=None, blocks_per_token=None, seed=0):
    """Compare GPU scores with the oracle on every (or a sample of) visible block."""
    sc = gpu_scores.cpu().numpy()
    rng = np.random.default_rng(seed)
    tokens = range(wl.num_tokens) if tokens is None else tokens
    worst = 0.0
    for t in tokens:
        b = int(wl.tok_seq[t])
        n_comp = int(wl.comp_off[b + 1] - wl.comp_off[b])
        nv = oracle.n_vis(n_comp, int(wl.tok_pos[t]), wl.ratio)
        if nv == 0:
            continue
        if blocks_per_token is None or blocks_per_token >= nv:
            blocks = np.arange(nv)
        else:
            blocks = np.unique(np.concatenate([
                rng.choice(nv, blocks_per_token, replace=False), [0, nv - 1]]))
        off = int(wl.comp_off[b])
        qb = W.bits(wl.q_idx[t])
        w = wl.w_idx[t].numpy()
        kb = W.bits(wl.k_idx)
        ref = np.array([oracle.block_score(qb, w, kb[off + s]) for s in blocks]) \
            if len(blocks) < 4096 else _scores_full(wl, t)[blocks]
        tol = score_tolerance(wl, t, blocks)
        err = np.abs(sc[t, blocks].astype(np.float64) - ref)
        bad = err > tol
        assert not bad.any(), (f"token {t}: {bad.sum()} blocks off, worst err {err.max():.3e} "
                               f"tol {tol[np.argmax(err)]:.3e}")
        worst = max(worst, float((err / np.maximum(tol, 1e-300)).max()))
    return worst


def _scores_full(wl, t):
    s, nv = oracle.indexer_scores(W.bits(wl.q_idx[t:t + 1]), wl.w_idx[t:t + 1].numpy(),
                                  W.bits(wl.k_idx), wl.tok_seq[t:t + 1].numpy(),
                                  wl.tok_pos[t:t + 1].numpy(), wl.comp_off.numpy())
    return s[0]


def check_topk_exact(wl, gpu_scores: torch.Tensor, idx: torch.Tensor, n_sel: torch.Tensor,
                     tokens=None):
    """idx must equal, bit for bit, the oracle's selection on the GPU's own scores."""
    sc = gpu_scores.cpu().numpy().astype(np.float64)
    idx = idx.cpu().numpy()
    n_sel = n_sel.cpu().numpy()
    tokens = range(wl.num_tokens) if tokens is None else tokens
    for t in tokens:
        b = int(wl.tok_seq[t])
        nv = oracle.n_vis(int(wl.comp_off[b + 1] - wl.comp_off[b]), int(wl.tok_pos[t]), wl.ratio)
        ref_idx, ref_n = oracle.topk(sc[t, :nv], wl.top_k)
        assert n_sel[t] == ref_n, (t, n_sel[t], ref_n)
        np.testing.assert_array_equal(idx[t], ref_idx, err_msg=f"token {t}")


def check_attention(wl, kv_buf: torch.Tensor, kv_len: torch.Tensor, out: torch.Tensor,
                    tokens=None, sinks=None):
    """GPU attention vs the f64 oracle on the very rows the GPU attended."""
    tokens = list(range(wl.num_tokens)) if tokens is None else list(tokens)
    kb = W.bits(kv_buf[tokens])
    kl = kv_len[tokens].cpu().numpy()
    ref = oracle.attention(W.bits(wl.q[tokens]), kb, kl, wl.scale,
                           sinks=None if sinks is None else sinks.cpu().numpy())
    got = out[tokens].cpu().numpy().astype(np.float64)
    err = np.abs(got - ref).max() if got.size else 0.0
    assert err <= ATTN_ATOL, f"attention max-abs error {err:.3e}"
    num = (got * ref).sum()
    den = np.sqrt((got * got).sum() * (ref * ref).sum())
    cos = float(num / den) if den > 0 else 1.0
    return float(err), cos


def gpu_rows(run: Run, idx: torch.Tensor, n_sel: torch.Tensor):
    """Gather on the GPU, and check it bit-exactly against the oracle's gather."""
    kv_buf, kv_len = run.gather(idx, n_sel)
    wl = run.wl
    ref_buf, ref_len = oracle.gather(idx.cpu().numpy(), n_sel.cpu().numpy(), W.bits(wl.comp_kv),
                                     W.bits(wl.swa_kv), wl.tok_seq.numpy(), wl.tok_pos.numpy(),
                                     wl.comp_off.numpy(), wl.swa_first_pos.numpy(),
                                     top_k=wl.top_k, window=wl.window, ratio=wl.ratio)
    np.testing.assert_array_equal(kv_len.cpu().numpy(), ref_len)
    got = W.bits(kv_buf)
    for t in range(wl.num_tokens):
        L = int(ref_len[t])
        np.testing.assert_array_equal(got[t, :L], ref_buf[t, :L], err_msg=f"token {t}")
    return kv_buf, kv_len


def recall_vs_oracle(wl, idx: torch.Tensor, n_sel: torch.Tensor, tokens=None):
    """Recall of the GPU selection against the oracle's own f64 selection, and
    a check that every disagreement sits within score tolerance of the cut."""
    idx = idx.cpu().numpy()
    n_sel = n_sel.cpu().numpy()
    tokens = range(wl.num_tokens) if tokens is None else tokens
    hit = tot = 0
    for t in tokens:
        ref_sc = _scores_full(wl, t)
        b = int(wl.tok_seq[t])
        nv = oracle.n_vis(int(wl.comp_off[b + 1] - wl.comp_off[b]), int(wl.tok_pos[t]), wl.ratio)
        ref_idx, ref_n = oracle.topk(ref_sc[:nv], wl.top_k)
        a = set(ref_idx[:ref_n].tolist())
        g = set(idx[t, :n_sel[t]].tolist())
        hit += len(a & g)
        tot += len(a)
        diff = np.array(sorted(a ^ g), dtype=np.int64)
        if diff.size:
            kth = np.sort(ref_sc[:nv])[::-1][ref_n - 1]
            tol = score_tolerance(wl, t, diff)
            assert (np.abs(ref_sc[diff] - kth) <= 2 * tol).all(), f"token {t}: far disagreement"
    return hit / max(tot, 1)
