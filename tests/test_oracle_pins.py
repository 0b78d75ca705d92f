"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Each group names the failure it is there to catch (a dropped ReLU, a wrong
sign, a transposed operand, the per-head key algebra, an off-by-one in the
causal rule, a wrong tie-break, a wrong window order ...).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import csa_workloads as W
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(a) -> np.ndarray:
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- visibility

def test_visibility_golden_table():
    rows = read_golden("visibility_cases.txt")
    assert len(rows) >= 15
    for pos, n_comp, ratio, expect in rows:
        assert oracle.n_vis(int(n_comp), int(pos), int(ratio)) == int(expect), (pos, n_comp)


def test_visibility_brute_force_block_membership():
    # Block j = positions [r*j, r*j + r); visible iff every position of block j
    # is < pos (strictly preceding) and j < n_comp.  Enumerate positions.
    for ratio in (1, 2, 4, 8):
        for n_comp in range(0, 7):
            for pos in range(0, 40):
                vis = sum(1 for j in range(n_comp)
                          if all(x < pos for x in range(ratio * j, ratio * j + ratio))
                          and not (ratio * j <= pos < ratio * j + ratio))
                assert oracle.n_vis(n_comp, pos, ratio) == vis


# ------------------------------------------------------------------- indexer

def _closed_form_case(n_ih=64, ihd=128, n_blocks=300):
    # q[h, d] = (h+1) * (-1)^d, k_s = e_{s mod ihd}  =>  q_h . k_s = (h+1)(-1)^s
    q = np.array([[(h + 1) * (-1) ** d for d in range(ihd)] for h in range(n_ih)], np.float32)
    k = np.zeros((n_blocks, ihd), np.float32)
    for s in range(n_blocks):
        k[s, s % ihd] = 1.0
    return bf16_bits(q), bf16_bits(k)


def test_indexer_closed_form_alternating_sign():
    """w = 1: score = sum_h ReLU((h+1)(-1)^s) = 2080 (even s) and 0 (odd s).
    A dropped ReLU gives -2080 on odd blocks; a dropped head gives < 2080."""
    qb, kb = _closed_form_case()
    n_blocks = kb.shape[0]
    w = np.ones((1, 64), np.float32)
    sc, nv = oracle.indexer_scores(qb[None], w, kb, [0], [4 * n_blocks], [0, n_blocks])
    assert nv[0] == n_blocks
    expect = np.array([2080.0 if (s % 128) % 2 == 0 else 0.0 for s in range(n_blocks)])
    np.testing.assert_array_equal(sc[0, :n_blocks], expect)


def test_indexer_closed_form_signed_weights():
    """w_h = (-1)^h: even s -> sum_h (-1)^h (h+1) = -32 exactly; odd s -> 0."""
    qb, kb = _closed_form_case(n_blocks=8)
    w = np.array([[(-1.0) ** h for h in range(64)]], np.float32)
    sc, _ = oracle.indexer_scores(qb[None], w, kb, [0], [32], [0, 8])
    np.testing.assert_array_equal(sc[0, :8], [-32.0, 0.0] * 4)


def test_indexer_closed_form_triangular():
    """q_h = first h+1 ones, k_s = first s+1 ones => q_h . k_s = min(h, s) + 1.
    Transposing q (d <-> h) or summing over the wrong axis breaks this."""
    n_ih, ihd, n = 64, 128, 128
    q = np.zeros((n_ih, ihd), np.float32)
    for h in range(n_ih):
        q[h, : h + 1] = 1.0
    k = np.zeros((n, ihd), np.float32)
    for s in range(n):
        k[s, : s + 1] = 1.0
    w = (np.arange(n_ih, dtype=np.float32) + 1.0)[None] / 64.0   # exact in bf16/f32
    sc, _ = oracle.indexer_scores(bf16_bits(q)[None], w, bf16_bits(k), [0], [4 * n], [0, n])
    expect = [sum((h + 1) / 64.0 * (min(h, s) + 1) for h in range(n_ih)) for s in range(n)]
    np.testing.assert_allclose(sc[0, :n], expect, rtol=0, atol=1e-12)


def test_indexer_one_hot_weights_is_relu_gemv():
    """w = e_h reduces the score to ReLU(K q_h): a plain matrix-vector product."""
    wl = W.make(seed=3, seq_lens=[4 * 200], n_comp=[200], n_heads=4)
    qb = W.bits(wl.q_idx)
    kb = W.bits(wl.k_idx)
    K = bits_to_f64(kb)
    for h in (0, 17, 63):
        w = np.zeros((1, 64), np.float32)
        w[0, h] = 1.0
        sc, nv = oracle.indexer_scores(qb, w, kb, [0], [800], [0, 200])
        ref = np.maximum(K @ bits_to_f64(qb[0, h]), 0.0)
        np.testing.assert_allclose(sc[0, :200], ref, rtol=1e-13, atol=1e-12)


def test_indexer_nonnegative_terms_and_homogeneity():
    wl = W.make(seed=4, seq_lens=[4 * 256], n_comp=[256], n_heads=4)
    qb, kb = W.bits(wl.q_idx), W.bits(wl.k_idx)
    w = np.abs(wl.w_idx.numpy())
    sc, _ = oracle.indexer_scores(qb, w, kb, [0], [1024], [0, 256])
    assert (sc[0, :256] >= 0).all() and (sc[0, :256] > 0).any()
    sc2, _ = oracle.indexer_scores(qb, 2.0 * wl.w_idx.numpy(), kb, [0], [1024], [0, 256])
    sc1, _ = oracle.indexer_scores(qb, wl.w_idx.numpy(), kb, [0], [1024], [0, 256])
    np.testing.assert_array_equal(sc2[0, :256], 2.0 * sc1[0, :256])


def test_indexer_mqa_einsum_cross_check():
    """The pages' corrected einsum 'tnd,cd->tnc' -> ReLU -> x w -> sum over heads,
    evaluated with numpy in float64 on a multi-token, multi-sequence layout."""
    wl = W.make(seed=5, seq_lens=[40, 100], tokens=[3, 2], n_comp=[10, 25], n_heads=2)
    qb, kb = W.bits(wl.q_idx), W.bits(wl.k_idx)
    sc, nv = oracle.indexer_scores(qb, wl.w_idx.numpy(), kb, wl.tok_seq.numpy(),
                                   wl.tok_pos.numpy(), wl.comp_off.numpy())
    Q, K, Wt = bits_to_f64(qb), bits_to_f64(kb), wl.w_idx.numpy().astype(np.float64)
    for t in range(wl.num_tokens):
        b = int(wl.tok_seq[t])
        off = int(wl.comp_off[b])
        n = int(nv[t])
        assert n == min(int(wl.comp_off[b + 1]) - off, int(wl.tok_pos[t]) // 4)
        raw = np.einsum("nd,cd->nc", Q[t], K[off:off + n])
        ref = (np.maximum(raw, 0.0) * Wt[t][:, None]).sum(0)
        np.testing.assert_allclose(sc[t, :n], ref, rtol=1e-12, atol=1e-10)


def test_per_head_key_algebra_is_rejected():
    """Negative control (Post-probe rewrite, F3): widening the 128-wide key
    buffer to n_ih*ihd and giving every head its own slice changes the scores.
    The closed-form pin above would catch an oracle that did this."""
    qb, kb = _closed_form_case(n_blocks=4)
    q = bits_to_f64(qb)
    k = bits_to_f64(kb)
    wide = np.zeros((4, 64, 128))
    wide[:, 0, :] = k              # the real key lands in head 0's slice only
    wrong = np.einsum("nd,cnd->nc", q, wide)
    wrong = np.maximum(wrong, 0).sum(0)
    sc, _ = oracle.indexer_scores(qb[None], np.ones((1, 64), np.float32), kb, [0], [16], [0, 4])
    assert not np.allclose(wrong, sc[0, :4])
    np.testing.assert_array_equal(sc[0, :4], [2080.0, 0.0, 2080.0, 0.0])


# --------------------------------------------------------------------- top-k

def _dominance_subsets(scores, k):
    """Every k-subset S with: for i in S, j not in S, i ranks before j under
    (score desc, index asc).  Exactly one exists."""
    n = len(scores)
    out = []
    for S in itertools.combinations(range(n), k):
        rest = [j for j in range(n) if j not in S]
        if all(scores[i] > scores[j] or (scores[i] == scores[j] and i < j)
               for i in S for j in rest):
            out.append(list(S))
    return out


def test_topk_brute_force_tiny_with_ties():
    rng = np.random.default_rng(0)
    for trial in range(300):
        n = int(rng.integers(0, 11))
        k = int(rng.integers(1, 6))
        scores = rng.integers(-3, 4, size=n).astype(np.float64)   # many ties
        idx, n_sel = oracle.topk(scores, k)
        kk = min(k, n)
        subs = _dominance_subsets(list(scores), kk)
        assert len(subs) == 1, (scores, k)
        assert n_sel == kk
        assert list(idx[:kk]) == subs[0]
        assert (idx[kk:] == -1).all()


def test_topk_matches_lexsort():
    """A library routine: numpy lexsort on (index, -score)."""
    rng = np.random.default_rng(1)
    for n, k in [(1000, 64), (5000, 1024), (300, 300), (17, 1024)]:
        scores = np.round(rng.normal(size=n), 2)
        idx, n_sel = oracle.topk(scores, k)
        order = np.lexsort((np.arange(n), -scores))[: min(k, n)]
        assert n_sel == min(k, n)
        np.testing.assert_array_equal(idx[:n_sel], np.sort(order))


def test_topk_signed_zero_ties_and_padding():
    scores = np.array([0.0, -0.0, 0.0, -1.0, -0.0])
    idx, n_sel = oracle.topk(scores, 2)
    assert n_sel == 2 and list(idx) == [0, 1]
    idx, n_sel = oracle.topk(np.array([5.0, -0.0, 0.0]), 2)
    assert list(idx) == [0, 1]
    idx, n_sel = oracle.topk(np.zeros(0), 4)
    assert n_sel == 0 and list(idx) == [-1] * 4
    idx, n_sel = oracle.topk(np.array([1.0, 3.0, 2.0]), 8)
    assert n_sel == 3 and list(idx) == [0, 1, 2] + [-1] * 5


def test_topk_rejects_nan():
    with pytest.raises(oracle.OracleError):
        oracle.topk(np.array([1.0, np.nan]), 1)


# -------------------------------------------------------------------- gather

def test_gather_rows_and_window_order():
    wl = W.make(seed=6, seq_lens=[50, 300], tokens=[1, 2], n_comp=[12, 75], top_k=8,
                window=16, swa_cap=32, hd=8, n_heads=2)
    idx = np.full((3, 8), -1, np.int32)
    n_sel = np.array([3, 8, 0], np.int32)
    idx[0, :3] = [0, 5, 11]
    idx[1, :8] = [1, 2, 3, 10, 20, 40, 74, 0]
    comp_kv, swa = W.bits(wl.comp_kv), W.bits(wl.swa_kv)
    buf, kv_len = oracle.gather(idx, n_sel, comp_kv, swa, wl.tok_seq.numpy(),
                                wl.tok_pos.numpy(), wl.comp_off.numpy(),
                                wl.swa_first_pos.numpy(), top_k=8, window=16)
    assert list(kv_len) == [3 + 16, 8 + 16, 0 + 16]
    for t in range(3):
        b = int(wl.tok_seq[t])
        p = int(wl.tok_pos[t])
        off = int(wl.comp_off[b])
        for i in range(n_sel[t]):
            np.testing.assert_array_equal(buf[t, i], comp_kv[off + idx[t, i]])
        for j, x in enumerate(range(p - 15, p + 1)):          # oldest -> newest
            np.testing.assert_array_equal(buf[t, n_sel[t] + j], swa[b, x % 32])


def test_gather_short_sequence_window_and_errors():
    wl = W.make(seed=7, seq_lens=[5], tokens=[1], n_comp=[1], top_k=4, window=16, hd=8,
                n_heads=1)
    buf, kv_len = oracle.gather(np.array([[0, -1, -1, -1]]), np.array([1]), W.bits(wl.comp_kv),
                                W.bits(wl.swa_kv), [0], [5], [0, 1], [0], top_k=4, window=16)
    assert kv_len[0] == 1 + 6           # positions 0..5
    with pytest.raises(oracle.OracleError) as e:      # block 1 is not visible at pos 5
        oracle.gather(np.array([[1, -1, -1, -1]]), np.array([1]), W.bits(wl.comp_kv),
                      W.bits(wl.swa_kv), [0], [5], [0, 2], [0], top_k=4, window=16)
    assert e.value.code == oracle.EINDEX
    with pytest.raises(oracle.OracleError) as e:      # ring no longer holds position 0
        oracle.gather(np.array([[0, -1, -1, -1]]), np.array([1]), W.bits(wl.comp_kv),
                      W.bits(wl.swa_kv), [0], [5], [0, 1], [1], top_k=4, window=16)
    assert e.value.code == oracle.ESWA


# ----------------------------------------------------------------- attention

def _sdpa_f64(q_bits, rows_bits, scale):
    q = torch.from_numpy(bits_to_f64(q_bits))[None]            # [1, H, hd]
    kv = torch.from_numpy(bits_to_f64(rows_bits))[None, None]  # [1, 1, L, hd]
    kv = kv.expand(1, q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q[:, :, None, :].transpose(0, 0), kv,
                                                         kv, scale=scale)
    return o[0, :, 0, :].numpy()


def test_attention_matches_sdpa_f64():
    rng = np.random.default_rng(8)
    H, hd, L = 4, 64, 37
    q = bf16_bits(rng.normal(size=(1, H, hd)))
    rows = bf16_bits(rng.normal(size=(1, 50, hd)))
    out = oracle.attention(q, rows, [L], scale=1 / math.sqrt(hd))
    q4 = torch.from_numpy(bits_to_f64(q))[:, :, None, :]             # [1, H, 1, hd]
    kv = torch.from_numpy(bits_to_f64(rows[:, :L]))[:, None].expand(1, H, L, hd)
    ref = torch.nn.functional.scaled_dot_product_attention(q4, kv, kv, scale=1 / math.sqrt(hd))
    np.testing.assert_allclose(out[0], ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    H, hd = 3, 32
    q = bf16_bits(rng.normal(size=(1, H, hd)))
    rows = bf16_bits(rng.normal(size=(1, 20, hd)))
    # a single row returns that row exactly
    out = oracle.attention(q, rows, [1], scale=0.3)
    for h in range(H):
        np.testing.assert_array_equal(out[0, h], bits_to_f64(rows[0, 0]))
    # identical rows return that row
    same = np.repeat(rows[:, :1], 20, axis=1)
    out = oracle.attention(q, same, [20], scale=0.3)
    np.testing.assert_allclose(out[0], np.repeat(bits_to_f64(rows[0, :1]), H, 0), rtol=1e-14)
    # q = 0 gives the mean of the rows
    out = oracle.attention(np.zeros_like(q), rows, [20], scale=0.3)
    np.testing.assert_allclose(out[0, 1], bits_to_f64(rows[0]).mean(0), rtol=1e-13, atol=1e-15)
    # permuting the rows changes nothing beyond rounding
    perm = rng.permutation(20)
    a = oracle.attention(q, rows, [20], scale=0.3)
    b = oracle.attention(q, rows[:, perm], [20], scale=0.3)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    # outputs are convex combinations of the rows
    r = bits_to_f64(rows[0])
    assert (a[0] <= r.max(0) + 1e-12).all() and (a[0] >= r.min(0) - 1e-12).all()


def test_attention_sink_identity():
    """With a sink logit s_h: out_sink = out * sigmoid(logsumexp(l) - s_h)."""
    rng = np.random.default_rng(10)
    H, hd, L = 4, 16, 9
    q = bf16_bits(rng.normal(size=(1, H, hd)))
    rows = bf16_bits(rng.normal(size=(1, L, hd)))
    sinks = rng.normal(size=H).astype(np.float32) * 2
    base = oracle.attention(q, rows, [L], scale=0.25)
    withs = oracle.attention(q, rows, [L], scale=0.25, sinks=sinks)
    logits = torch.from_numpy(0.25 * bits_to_f64(q[0]) @ bits_to_f64(rows[0]).T)
    lse = torch.logsumexp(logits, dim=1).numpy()
    factor = 1.0 / (1.0 + np.exp(sinks.astype(np.float64) - lse))
    np.testing.assert_allclose(withs[0], base[0] * factor[:, None], rtol=1e-12, atol=1e-14)


# ----------------------------------------------- partial attention and merge

def test_partials_merge_to_the_whole_attention():
    """Cut a token's rows into random parts: the log-sum-exp merge of the
    parts' partials equals the attention over all rows (the C oracle), with
    and without a sink; an empty part changes nothing."""
    rng = np.random.default_rng(12)
    H, hd, L = 5, 64, 90
    q = bf16_bits(rng.normal(size=(1, H, hd)) * 2)
    rows = bf16_bits(rng.normal(size=(1, L, hd)))
    sinks = (rng.normal(size=H) * 3).astype(np.float32)
    full = oracle.attention(q, rows, [L], scale=0.2)
    full_s = oracle.attention(q, rows, [L], scale=0.2, sinks=sinks)
    for trial in range(4):
        cuts = np.sort(rng.choice(np.arange(1, L), size=trial + 1, replace=False))
        parts = np.split(np.arange(L), cuts)
        parts.append(np.arange(0))                     # an empty part
        got = [oracle.attention_partial(q[0], rows[0, p], 0.2) for p in parts]
        O = np.stack([g[0] for g in got])
        m = np.stack([g[1] for g in got])
        lv = np.stack([g[2] for g in got])
        np.testing.assert_allclose(oracle.combine_partials(O, m, lv), full[0], rtol=1e-12,
                                   atol=1e-13)
        np.testing.assert_allclose(oracle.combine_partials(O, m, lv, sinks=sinks), full_s[0],
                                   rtol=1e-12, atol=1e-13)


def test_partial_attention_closed_forms():
    rng = np.random.default_rng(13)
    H, hd = 3, 16
    q = bf16_bits(rng.normal(size=(H, hd)))
    rows = bf16_bits(rng.normal(size=(4, hd)))
    # one row: O = the row, m = its logit, l = 1
    O, m, lv = oracle.attention_partial(q, rows[:1], 0.5)
    r = bits_to_f64(rows[0])
    np.testing.assert_array_equal(lv, np.ones(H))
    np.testing.assert_allclose(m, 0.5 * bits_to_f64(q) @ r, rtol=1e-15)
    np.testing.assert_array_equal(O, np.repeat(r[None], H, 0))
    # q = 0: m = 0, l = n, O = the row sum
    O, m, lv = oracle.attention_partial(np.zeros_like(q), rows, 0.5)
    np.testing.assert_array_equal(m, np.zeros(H))
    np.testing.assert_array_equal(lv, np.full(H, 4.0))
    np.testing.assert_allclose(O[1], bits_to_f64(rows).sum(0), rtol=1e-15)
    # no rows: (0, -inf, 0), and a merge of nothing but empty parts is zero
    O, m, lv = oracle.attention_partial(q, rows[:0], 0.5)
    assert (m == -np.inf).all() and (lv == 0).all() and (O == 0).all()
    np.testing.assert_array_equal(oracle.combine_partials(O[None], m[None], lv[None]),
                                  np.zeros((H, hd)))


# ----------------------------------------------------------- the whole step

def _visible_rows(wl, t, nv):
    b = int(wl.tok_seq[t])
    p = int(wl.tok_pos[t])
    off = int(wl.comp_off[b])
    comp = W.bits(wl.comp_kv)[off:off + nv]
    first = max(0, p - wl.window + 1)
    swa = np.stack([W.bits(wl.swa_kv)[b, x % wl.swa_cap] for x in range(first, p + 1)])
    return np.concatenate([comp, swa])


def test_decode_reduces_to_dense_attention_when_topk_covers_all():
    wl = W.make(seed=11, seq_lens=[4 * 30 + 2, 70], tokens=[2, 1], n_comp=[30, 17],
                top_k=64, window=16, swa_cap=20, hd=64, n_heads=4)
    idx, n_sel, out = oracle.decode(W.bits(wl.q_idx), wl.w_idx.numpy(), W.bits(wl.k_idx),
                                    W.bits(wl.comp_kv), W.bits(wl.swa_kv), W.bits(wl.q),
                                    wl.tok_seq.numpy(), wl.tok_pos.numpy(), wl.comp_off.numpy(),
                                    wl.swa_first_pos.numpy(), top_k=64, window=16)
    for t in range(wl.num_tokens):
        b = int(wl.tok_seq[t])
        nv = min(int(wl.comp_off[b + 1] - wl.comp_off[b]), int(wl.tok_pos[t]) // 4)
        assert n_sel[t] == nv
        assert list(idx[t, :nv]) == list(range(nv))
        rows = _visible_rows(wl, t, nv)
        q4 = torch.from_numpy(bits_to_f64(W.bits(wl.q)[t]))[None, :, None, :]
        kv = torch.from_numpy(bits_to_f64(rows))[None, None].expand(1, 4, -1, -1)
        ref = torch.nn.functional.scaled_dot_product_attention(q4, kv, kv, scale=wl.scale)
        np.testing.assert_allclose(out[t], ref[0, :, 0].numpy(), rtol=1e-11, atol=1e-12)


def test_decode_causality_perturbation():
    """Changing any block at or after n_vis, or any ring slot outside the
    window, leaves the selection and the output bit-identical."""
    wl = W.make(seed=12, seq_lens=[4 * 40 + 1], tokens=[1], n_comp=[40], comp_capacity=[48],
                top_k=8, window=8, swa_cap=16, hd=32, n_heads=2)
    args = lambda w: (W.bits(w.q_idx), w.w_idx.numpy(), W.bits(w.k_idx), W.bits(w.comp_kv),
                      W.bits(w.swa_kv), W.bits(w.q), w.tok_seq.numpy(), w.tok_pos.numpy(),
                      w.comp_off.numpy(), w.swa_first_pos.numpy())
    idx0, ns0, out0 = oracle.decode(*args(wl), top_k=8, window=8)
    nv = 40
    g = torch.Generator().manual_seed(99)
    wl.k_idx[nv:] = W.bf16_normal(g, 8, wl.ihd) * 50
    wl.comp_kv[nv:] = W.bf16_normal(g, 8, wl.hd) * 50
    p = int(wl.tok_pos[0])
    inside = {x % 16 for x in range(p - 7, p + 1)}
    for slot in range(16):
        if slot not in inside:
            wl.swa_kv[0, slot] = W.bf16_normal(g, wl.hd) * 50
    # grow the packed offsets: the extra rows exist but are not visible at p
    wl.comp_off[1] = 48
    idx1, ns1, out1 = oracle.decode(*args(wl), top_k=8, window=8)
    np.testing.assert_array_equal(idx0, idx1)
    np.testing.assert_array_equal(out0, out1)
    assert (idx0[0, : ns0[0]] < nv).all()


def test_planted_blocks_are_selected():
    wl = W.make(seed=13, seq_lens=[4 * 4096], n_comp=[4096], top_k=128, n_heads=2, hd=32,
                window=4, swa_cap=8)
    W.plant_blocks(wl, 32, 4.0, seed=2)
    sc, nv = oracle.indexer_scores(W.bits(wl.q_idx), wl.w_idx.numpy(), W.bits(wl.k_idx),
                                   [0], wl.tok_pos.numpy(), wl.comp_off.numpy())
    idx, n_sel = oracle.topk(sc[0, : nv[0]], 128)
    assert set(wl.planted.tolist()) <= set(idx[:n_sel].tolist())


# ----------------------------------------------------------------------- HCA

def test_hca_is_dense_attention_over_visible_rows_and_window():
    """HCA (ratio 128): SDPA in float64 over every visible compressed row
    (strictly preceding blocks) followed by the window rows."""
    wl = W.make(seed=14, seq_lens=[128 * 40 + 5, 128 * 3 + 127, 60], tokens=[1, 2, 1],
                n_comp=[40, 4, 0], ratio=128, window=16, swa_cap=24, hd=64, n_heads=4)
    out, kv_len = oracle.hca_decode(W.bits(wl.comp_kv), W.bits(wl.swa_kv), W.bits(wl.q),
                                    wl.tok_seq.numpy(), wl.tok_pos.numpy(), wl.comp_off.numpy(),
                                    wl.swa_first_pos.numpy(), window=16, ratio=128)
    for t in range(wl.num_tokens):
        b = int(wl.tok_seq[t])
        p = int(wl.tok_pos[t])
        nv = min(int(wl.comp_off[b + 1] - wl.comp_off[b]), p // 128)
        rows = _visible_rows(wl, t, nv)
        assert kv_len[t] == len(rows)
        q4 = torch.from_numpy(bits_to_f64(W.bits(wl.q)[t]))[None, :, None, :]
        kv = torch.from_numpy(bits_to_f64(rows))[None, None].expand(1, 4, -1, -1)
        ref = torch.nn.functional.scaled_dot_product_attention(q4, kv, kv, scale=wl.scale)
        np.testing.assert_allclose(out[t], ref[0, :, 0].numpy(), rtol=1e-11, atol=1e-12)
    # token 2 sits at 128*3+127 (p = 511): block 3 holds 384..511 and stays hidden
    assert kv_len[1] == 3 + 16


def test_hca_causality_perturbation():
    wl = W.make(seed=15, seq_lens=[128 * 20 + 3], n_comp=[20], comp_capacity=[30], ratio=128,
                window=8, swa_cap=16, hd=32, n_heads=2)
    args = lambda w: (W.bits(w.comp_kv), W.bits(w.swa_kv), W.bits(w.q), w.tok_seq.numpy(),
                      w.tok_pos.numpy(), w.comp_off.numpy(), w.swa_first_pos.numpy())
    out0, _ = oracle.hca_decode(*args(wl), window=8, ratio=128)
    g = torch.Generator().manual_seed(7)
    wl.comp_kv[20:] = W.bf16_normal(g, 10, wl.hd) * 50
    wl.comp_off[1] = 30
    out1, _ = oracle.hca_decode(*args(wl), window=8, ratio=128)
    np.testing.assert_array_equal(out0, out1)


# --------------------------------------------------------------------- sizes

def test_memory_sizing_matches_pages():
    g = {k: int(v) for k, v in read_golden("memory_sizing.txt")}
    t = W.tiny()
    assert t.k_idx[0].nbytes == g["indexer_key_bytes_per_block"]
    assert t.comp_kv[0].nbytes == g["main_row_bytes_per_block"]
    assert t.swa_kv[0].nbytes == g["swa_ring_bytes_per_layer"]
    n1m = 262144
    assert n1m * W.IHD * 2 == g["indexer_key_bytes_1m"]
    assert n1m * W.HD * 2 == g["main_row_bytes_1m"]


# ---------------------------------------------------------------- FP4 keys
# MXFP4 as the oracle reads it (csa_oracle.h): e2m1 elements, one e8m0 scale
# 2^(E-127) per 32 elements.  The pins below use the format's definition
# (bit fields, the value grid) and properties any correct quantizer has.

def e2m1_from_bits(c: int) -> float:
    """OCP e2m1: sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


E2M1_GRID = np.array([e2m1_from_bits(c) for c in range(8)])


def fp4_fields(rows: np.ndarray):
    """codes [R, 128] (element 2i low nibble of byte i) and scales E [R, 4]."""
    codes = np.empty((rows.shape[0], 128), dtype=np.uint8)
    codes[:, 0::2] = rows[:, :64] & 15
    codes[:, 1::2] = rows[:, :64] >> 4
    return codes, rows[:, 64:68].astype(np.int64)


def test_fp4_e2m1_table():
    for c in range(16):
        assert oracle.e2m1_value(c) == e2m1_from_bits(c), c
    assert list(E2M1_GRID) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_fp4_grid_values_round_trip():
    rng = np.random.default_rng(11)
    R = 64
    vals = np.zeros((R, 128))
    for r in range(R):
        for b in range(4):
            s = int(rng.integers(-6, 6))
            mags = rng.choice(E2M1_GRID, 32) * (2.0 ** s)
            mags[int(rng.integers(0, 32))] = 6.0 * 2.0 ** s     # block amax 6 * 2^s: scale 2^s
            signs = rng.choice([-1.0, 1.0], 32)
            vals[r, b * 32:(b + 1) * 32] = signs * mags
    bits = bf16_bits(vals)
    assert np.array_equal(bits_to_f64(bits), vals)            # grid values are bf16 values
    rows = oracle.fp4_quantize(bits)
    assert rows.shape == (R, 80) and not rows[:, 68:].any()
    # exact round trip (a signed zero comes back as +0: zero magnitude is code 0)
    assert np.array_equal(bits_to_f64(oracle.fp4_dequantize(rows)), vals)
    codes, E = fp4_fields(rows)
    deq = np.array([[e2m1_from_bits(int(c)) for c in row] for row in codes])
    assert np.array_equal(deq * 2.0 ** (np.repeat(E, 32, axis=1) - 127), vals)


def test_fp4_nearest_code_ties_and_saturation():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((200, 128)) * np.exp(rng.uniform(-3, 3, (200, 1)))
    bits = bf16_bits(x)
    xv = bits_to_f64(bits)
    rows = oracle.fp4_quantize(bits)
    codes, E = fp4_fields(rows)
    X = 2.0 ** (np.repeat(E, 32, axis=1) - 127)
    chosen = np.vectorize(e2m1_from_bits)(codes)
    # no e2m1 value (either sign) is nearer to x / X than the chosen one
    cand = np.concatenate([E2M1_GRID, -E2M1_GRID])
    best = np.abs(xv[..., None] / X[..., None] - cand).min(axis=-1)
    assert (np.abs(xv / X - chosen) <= best).all()
    # midpoints of the grid (block scale fixed at 2^0 by an element of 4):
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 7.75]
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0]      # even code, then saturation
    blk = np.zeros(128)
    blk[0] = 4.0
    blk[1:1 + len(mids)] = mids
    blk[32:32 + len(mids)] = -np.array(mids)
    blk[64] = 7.75                                             # amax 7.75: scale still 2^0
    r = oracle.fp4_quantize(bf16_bits(blk[None]))
    c, e = fp4_fields(r)
    assert e[0, 0] == 127 and e[0, 2] == 127
    got = np.vectorize(e2m1_from_bits)(c[0])
    assert list(got[1:1 + len(mids)]) == want
    assert list(got[32:32 + len(mids)]) == [-w if w else 0.0 for w in want]
    assert c[0, 32] == 0 and c[0, 64 + 1] == 0                 # a zero magnitude is code 0


def test_fp4_scale_rule_and_zero_block():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((100, 128)) * np.exp(rng.uniform(-20, 20, (100, 1)))
    x[0, :32] = 0.0
    x[1, 32:64] = -0.0
    bits = bf16_bits(x)
    rows = oracle.fp4_quantize(bits)
    codes, E = fp4_fields(rows)
    amax = np.abs(bits_to_f64(bits)).reshape(100, 4, 32).max(axis=-1)
    X = 2.0 ** (E - 127)
    nz = amax > 0
    ratio = amax[nz] / X[nz]
    assert ((ratio >= 4.0) & (ratio < 8.0)).all()
    assert E[0, 0] == 0 and E[1, 1] == 0
    assert not codes[0, :32].any() and not codes[1, 32:64].any()


def test_fp4_sign_and_power_of_two_covariance():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((50, 128))
    bits = bf16_bits(x)
    r0 = oracle.fp4_quantize(bits)
    c0, e0 = fp4_fields(r0)
    rn = oracle.fp4_quantize(bf16_bits(-bits_to_f64(bits)))
    cn, en = fp4_fields(rn)
    assert np.array_equal(en, e0)
    assert np.array_equal(cn, np.where(c0 & 7, c0 ^ 8, 0))
    r2 = oracle.fp4_quantize(bf16_bits(4.0 * bits_to_f64(bits)))
    c2, e2 = fp4_fields(r2)
    assert np.array_equal(c2, c0) and np.array_equal(e2, e0 + 2)


def test_fp4_error_bound():
    rng = np.random.default_rng(15)
    bits = bf16_bits(rng.standard_normal((100, 128)))
    x = bits_to_f64(bits)
    rows = oracle.fp4_quantize(bits)
    _, E = fp4_fields(rows)
    X = 2.0 ** (np.repeat(E, 32, axis=1) - 127)
    err = np.abs(x - bits_to_f64(oracle.fp4_dequantize(rows)))
    inside = np.abs(x) <= 6.0 * X
    assert (err[inside] <= 1.0 * X[inside]).all()     # half of the widest grid step (4 -> 6)
    assert (err <= 2.0 * X).all()                      # saturation: |x| < 8 X
    assert err.max() > 0


def test_fp4_scores_are_the_indexer_on_dequantized_keys():
    wl = W.tiny(seed=4)
    qb, kb, w = W.bits(wl.q_idx), W.bits(wl.k_idx), wl.w_idx.numpy()
    rows = oracle.fp4_quantize(kb)
    kd = oracle.fp4_dequantize(rows)
    sc, nv = oracle.indexer_scores(qb, w, kd, wl.tok_seq, wl.tok_pos, wl.comp_off)
    q, k = bits_to_f64(qb), bits_to_f64(kd)
    t = 0
    n = int(nv[t])
    ref = (np.maximum(np.einsum("hd,sd->hs", q[t], k[:n]), 0.0) * w[t].astype(np.float64)[:, None]).sum(0)
    np.testing.assert_allclose(sc[t, :n], ref, rtol=1e-12, atol=1e-12)
    # FP4 keys move the scores, but the ranking stays close to the bf16 one
    sb, _ = oracle.indexer_scores(qb, w, kb, wl.tok_seq, wl.tok_pos, wl.comp_off)
    assert np.corrcoef(sc[t, :n], sb[t, :n])[0, 1] > 0.9


def test_fp4_row_size():
    # 64 code bytes + 4 scale bytes + 12 zero bytes per 128-wide key; at 1M
    # context (262,144 blocks) the indexer cache is 20 MiB instead of 64 MiB.
    assert oracle.FP4_ROW == 80
    assert 262144 * oracle.FP4_ROW == 20 * 2 ** 20
