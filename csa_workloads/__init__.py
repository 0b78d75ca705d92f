"""Seeded synthetic inputs for compressed sparse attention (CSA) decode.

This module only draws random tensors and lays them out; it holds none of the
method's arithmetic (no scores, no selection, no attention).  The same
generators feed the CPU oracle (``oracle/``), the CUDA library's tests and
``bench.py``.

Recipe (all draws from a CPU ``torch.Generator`` seeded per workload):
  * bf16 tensors are N(0, 1) draws in fp32 rounded to bf16;
  * indexer head weights w^I are fp32 N(0, 1) / 8;
  * one compressed block per ``ratio`` = 4 tokens; indexer keys are 128 wide
    and shared by the 64 indexer heads; main rows are 512 wide and serve as
    both key and value;
  * the sliding window ring holds position p at slot p mod swa_cap.

The five named workloads follow the pages' 1M-context sizing (64 MB of
indexer keys and 256 MB of compressed rows per CSA layer at 262,144 blocks,
"ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite", PART 2) and the decode
shapes stated alongside them: tiny, 64k (100-step loop), 1m (with 32 planted
blocks), batch32 (ragged 32K..128K contexts) and prefill (4096-token chunk).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

N_IH = 64       # indexer heads
IHD = 128       # indexer head dim (shared key width)
HD = 512        # main head dim (shared key/value row)
WINDOW = 128    # sliding window
RATIO = 4       # tokens per compressed block


@dataclasses.dataclass
class Workload:
    name: str
    # layout
    tok_seq: torch.Tensor        # [T] int32
    tok_pos: torch.Tensor        # [T] int64
    comp_off: torch.Tensor       # [B+1] int64
    swa_first_pos: torch.Tensor  # [B] int64
    swa_cap: int
    # params
    n_ih: int
    ihd: int
    hd: int
    n_heads: int
    top_k: int
    window: int
    ratio: int
    scale: float
    # data (CPU tensors)
    q_idx: torch.Tensor          # [T, n_ih, ihd] bf16
    w_idx: torch.Tensor          # [T, n_ih] fp32
    k_idx: torch.Tensor          # [R, ihd] bf16
    comp_kv: torch.Tensor        # [R, hd] bf16
    swa_kv: torch.Tensor         # [B, swa_cap, hd] bf16
    q: torch.Tensor              # [T, H, hd] bf16
    planted: Optional[torch.Tensor] = None   # [P] int64 planted block indices (seq 0)
    seed: int = 0

    @property
    def num_tokens(self) -> int:
        return int(self.tok_seq.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.comp_off.shape[0] - 1)

    @property
    def total_comp_rows(self) -> int:
        return int(self.comp_off[-1])

    @property
    def max_comp_rows(self) -> int:
        n = self.comp_off[1:] - self.comp_off[:-1]
        return int(n.max()) if n.numel() else 0

    def to(self, device) -> "Workload":
        out = dataclasses.replace(self)
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, torch.Tensor):
                setattr(out, f.name, v.to(device))
        return out


def bf16_normal(gen: torch.Generator, *shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32,
                       device=gen.device).to(torch.bfloat16)


def bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bit patterns (for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def make(name: str = "custom", *, seed: int = 0, seq_lens=None, tokens=None,
         n_comp=None, top_k: int = 64, n_heads: int = 16, n_ih: int = N_IH, ihd: int = IHD,
         hd: int = HD, window: int = WINDOW, ratio: int = RATIO, swa_cap: Optional[int] = None,
         comp_capacity=None, scale: Optional[float] = None, w_scale: float = 1.0 / 8.0,
         device=None) -> Workload:
    """A general seeded workload.

    seq_lens[b]   absolute position of the first query token of sequence b
                  (the context length before it);
    tokens[b]     query tokens of sequence b, at consecutive positions from seq_lens[b];
    n_comp[b]     compressed blocks in the cache (default: every complete block
                  before the last query token, i.e. floor(last_pos / ratio));
    comp_capacity rows reserved per sequence (>= n_comp; extra rows are drawn too).
    device        draw the data tensors there (default: the CPU generator).
    """
    gen = torch.Generator(device=device or "cpu").manual_seed(seed)
    if seq_lens is None:
        seq_lens = [1024]
    B = len(seq_lens)
    if tokens is None:
        tokens = [1] * B
    last_pos = [int(seq_lens[b]) + int(tokens[b]) - 1 for b in range(B)]
    if n_comp is None:
        n_comp = [p // ratio for p in last_pos]
    if comp_capacity is None:
        comp_capacity = list(n_comp)
    if swa_cap is None:
        swa_cap = max(window, window - 1 + max(tokens))
    tok_seq, tok_pos = [], []
    for b in range(B):
        for i in range(tokens[b]):
            tok_seq.append(b)
            tok_pos.append(int(seq_lens[b]) + i)
    T = len(tok_seq)
    rows = [int(c) for c in comp_capacity]
    comp_off = [0]
    for b in range(B):
        comp_off.append(comp_off[-1] + rows[b])
    R = comp_off[-1]
    # The packed offsets describe the *valid* blocks; capacity rows beyond
    # n_comp[b] are laid out only when sequences are packed back to back with
    # no slack, so for B > 1 capacity must equal n_comp.
    if B > 1:
        assert rows == [int(c) for c in n_comp], "packed sequences carry no slack rows"
        off_valid = comp_off
    else:
        off_valid = [0, int(n_comp[0])]
    k_idx = bf16_normal(gen, R, ihd)
    comp_kv = bf16_normal(gen, R, hd)
    swa_kv = bf16_normal(gen, B, swa_cap, hd)
    q_idx = bf16_normal(gen, T, n_ih, ihd)
    w_idx = torch.randn(T, n_ih, generator=gen, dtype=torch.float32, device=gen.device) * w_scale
    q = bf16_normal(gen, T, n_heads, hd)
    # oldest position still resident in each ring: the ring holds the last
    # swa_cap positions up to the last query token of the sequence.
    swa_first = [max(0, last_pos[b] - swa_cap + 1) for b in range(B)]
    return Workload(
        name=name,
        tok_seq=torch.tensor(tok_seq, dtype=torch.int32),
        tok_pos=torch.tensor(tok_pos, dtype=torch.int64),
        comp_off=torch.tensor(off_valid, dtype=torch.int64),
        swa_first_pos=torch.tensor(swa_first, dtype=torch.int64),
        swa_cap=int(swa_cap), n_ih=n_ih, ihd=ihd, hd=hd, n_heads=n_heads, top_k=top_k,
        window=window, ratio=ratio,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(hd)),
        q_idx=q_idx, w_idx=w_idx, k_idx=k_idx, comp_kv=comp_kv, swa_kv=swa_kv, q=q,
        seed=seed)


def plant_blocks(wl: Workload, count: int = 32, factor: float = 4.0, seed: int = 1) -> Workload:
    """Turn `count` seeded blocks of sequence 0 onto the query's positive-weight
    mean direction and scale them by `factor` (in place).

    Direction: mu = normalize(sum_h max(w_h, 0) * q_h) of token 0's indexer
    queries; planted key = factor * |k_s| * mu, rounded to bf16.  The plain
    unweighted mean does not favour the planted blocks because w has random
    signs, so the positive-weight mean is used.
    """
    gen = torch.Generator().manual_seed(seed)
    n0 = int(wl.comp_off[1] - wl.comp_off[0])
    base = int(wl.comp_off[0])
    picks = torch.randperm(n0, generator=gen)[:count].sort().values.to(torch.int64)
    picks = picks.to(wl.k_idx.device)
    qf = wl.q_idx[0].float()                      # [n_ih, ihd]
    wpos = wl.w_idx[0].clamp_min(0.0)             # [n_ih]
    mu = (wpos[:, None] * qf).sum(0)
    mu = mu / mu.norm()
    for s in picks.tolist():
        k = wl.k_idx[base + s].float()
        wl.k_idx[base + s] = (factor * k.norm() * mu).to(torch.bfloat16)
    wl.planted = picks.cpu()
    return wl


# ---- the named workloads -------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    """1 token at position 1024; 256 blocks, all strictly preceding; top_k 64;
    16 main heads; SWA ring of 128."""
    return make("tiny", seed=seed, seq_lens=[1024], tokens=[1], n_comp=[256], top_k=64,
                n_heads=16, swa_cap=128)


def ctx64k(seed: int = 0, steps: int = 100) -> Workload:
    """64K-context single-sequence decode: step i queries position 65536 + i
    with n_comp = 16384 + i // 4 valid blocks; the buffers hold every block the
    loop will reach.  Step 0's state is returned; ``ctx64k_step`` advances it."""
    cap = 16384 + (steps - 1) // 4 + 1
    wl = make("64k", seed=seed, seq_lens=[65536], tokens=[1], n_comp=[16384],
              comp_capacity=[cap], top_k=1024, n_heads=64, swa_cap=128)
    return wl


def ctx64k_step(wl: Workload, i: int, gen: torch.Generator) -> None:
    """Advance the 64K loop to step i (i >= 1) in place: the query moves to
    position 65536 + i, the window ring receives that position's row, and when
    the new position starts a block the block just completed becomes visible
    (its row was drawn with the buffers).  Fresh query activations each step."""
    p = 65536 + i
    wl.tok_pos[0] = p
    wl.comp_off[1] = 16384 + i // 4
    wl.swa_kv[0, p % wl.swa_cap] = bf16_normal(gen, wl.hd)
    wl.swa_first_pos[0] = max(0, p - wl.swa_cap + 1)
    wl.q_idx.copy_(bf16_normal(gen, *wl.q_idx.shape))
    wl.w_idx.copy_(torch.randn(*wl.w_idx.shape, generator=gen) / 8.0)
    wl.q.copy_(bf16_normal(gen, *wl.q.shape))


def ctx1m(seed: int = 0, planted: int = 32, device=None) -> Workload:
    """1M-context single-sequence decode on one CSA layer: 262,144 blocks
    (64 MiB of indexer keys, 256 MiB of rows), top_k 1024, 64 heads, 32
    planted blocks."""
    wl = make("1m", seed=seed, seq_lens=[1 << 20], tokens=[1], n_comp=[262144], top_k=1024,
              n_heads=64, swa_cap=128, device=device)
    if planted:
        plant_blocks(wl, planted, 4.0, seed + 1)
    return wl


def batch32_lens(seed: int = 0, n: int = 32):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(32768, 131072 + 1, (n,), generator=gen).tolist()


def batch32(seed: int = 0, device=None) -> Workload:
    """32 sequences with context lengths uniform in 32K..128K; one query token
    per sequence at position len; n_comp = len // 4, packed with offsets."""
    lens = batch32_lens(seed)
    return make("batch32", seed=seed, seq_lens=lens, tokens=[1] * len(lens),
                n_comp=[l // 4 for l in lens], top_k=1024, n_heads=64, swa_cap=128,
                device=device)


def prefill(seed: int = 0, tokens: int = 4096, device=None) -> Workload:
    """Chunked prefill: `tokens` query tokens at positions 262144 .. of one
    sequence, 66,559 cached blocks (every block any token of the 4096 chunk
    can see), a ring of 8192 window rows covering positions 262017 onwards."""
    last = 262144 + tokens - 1
    return make("prefill", seed=seed, seq_lens=[262144], tokens=[tokens],
                n_comp=[last // 4], top_k=1024, n_heads=64, swa_cap=8192, device=device)


def hca1m(seed: int = 0, device=None) -> Workload:
    """1M-context HCA layer: ratio 128, 8192 compressed rows (8 MiB), dense
    attention over all of them plus the 128-row window, 64 heads."""
    return make("hca1m", seed=seed, seq_lens=[1 << 20], tokens=[1], n_comp=[8192], top_k=1,
                n_heads=64, swa_cap=128, ratio=128, device=device)


NAMED = {"tiny": tiny, "64k": ctx64k, "1m": ctx1m, "batch32": batch32, "prefill": prefill,
         "hca1m": hca1m}
