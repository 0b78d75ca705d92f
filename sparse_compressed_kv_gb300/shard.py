"""Sharded single-sequence decode over G devices (or G shards on one device).

One sequence's compressed blocks are cut into contiguous ranges; shard g
holds blocks [bounds[g], bounds[g+1]) of the indexer keys and of the rows
("ARCHITECTURE & MEMORY AUDIT -- 1M-context viability", PART 2, "Total KV
cache @ 1M context": the KV cache sharded across the GPUs).  A step is
  1. per shard, its best top_k blocks with their scores (csa_shard_candidates);
  2. one all-gather of the candidates, then on every device the global top-k
     (csa_shard_merge), identical to the single-device selection;
  3. per shard, attention over its selected rows, and on the device that
     holds the window ring, over the window rows: unnormalised partials
     (csa_shard_attention, csa_window_attention);
  4. one all-gather of the partials and the log-sum-exp combine
     (csa_shard_combine).
Every computation is a libcsa kernel; this module cuts the ranges, moves the
candidates and partials between devices (torch.distributed all-gathers over
NCCL, or plain stacking when the shards share one device) and orders the
calls.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

from . import csa


def shard_bounds(n_blocks: int, num_shards: int) -> List[int]:
    """Contiguous block ranges of equal size to within one block."""
    if num_shards < 1 or num_shards > csa.MAX_SHARDS:
        raise ValueError(f"1 <= num_shards <= {csa.MAX_SHARDS}")
    return [n_blocks * g // num_shards for g in range(num_shards + 1)]


@dataclass
class Shard:
    """One shard's caches (rows bounds[g] .. bounds[g+1]-1 of the sequence)."""
    lo: int
    hi: int
    k_idx: torch.Tensor      # bf16 [hi - lo, 128]
    comp_kv: torch.Tensor    # bf16 [hi - lo, 512]
    ws: torch.Tensor         # workspace, csa_shard_workspace_size bytes, zeroed once


def make_shard(layout: csa.Layout, prm: csa.csa_params_t, lo: int, hi: int, k_idx: torch.Tensor,
               comp_kv: torch.Tensor) -> Shard:
    """A shard over rows [lo, hi) of the given whole-sequence caches (copied)."""
    dev = k_idx.device
    n = csa.csa_shard_workspace_size(layout, prm, lo, hi)
    return Shard(lo, hi, k_idx[lo:hi].contiguous(), comp_kv[lo:hi].contiguous(),
                 torch.zeros(n, dtype=torch.uint8, device=dev))


def candidates(sh: Shard, layout: csa.Layout, prm: csa.csa_params_t, q_idx, w_idx, status,
               stream=None):
    T, K = int(layout.tok_seq.shape[0]), int(prm.top_k)
    dev = q_idx.device
    score = torch.empty(T, K, dtype=torch.float32, device=dev)
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    n = torch.empty(T, dtype=torch.int32, device=dev)
    csa.csa_shard_candidates(layout, prm, sh.lo, sh.hi, q_idx, w_idx, sh.k_idx, score, idx, n,
                             status, sh.ws, stream=stream)
    return score, idx, n


def merge(bounds: Sequence[int], cand_score, cand_idx, n_cand, status, stream=None):
    """Gathered candidates [G, T, K] -> (idx [T, K], n_sel [T], shard_idx [G, T, K],
    shard_nsel [G, T])."""
    G, T, K = (int(x) for x in cand_idx.shape)
    dev = cand_idx.device
    idx = torch.empty(T, K, dtype=torch.int32, device=dev)
    n_sel = torch.empty(T, dtype=torch.int32, device=dev)
    sidx = torch.empty(G, T, K, dtype=torch.int32, device=dev)
    snsel = torch.empty(G, T, dtype=torch.int32, device=dev)
    csa.csa_shard_merge(bounds, cand_score, cand_idx, n_cand, idx, n_sel, sidx, snsel, status,
                        stream=stream)
    return idx, n_sel, sidx, snsel


def partial(sh: Shard, layout: csa.Layout, prm: csa.csa_params_t, shard_idx, shard_nsel, q,
            status, stream=None):
    T, H = int(layout.tok_seq.shape[0]), int(prm.n_heads)
    o = torch.empty(T, H, int(prm.hd), dtype=torch.float32, device=q.device)
    ml = torch.empty(T, H, 2, dtype=torch.float32, device=q.device)
    csa.csa_shard_attention(layout, prm, sh.lo, sh.hi, shard_idx, shard_nsel, sh.comp_kv, q, o,
                            ml, status, sh.ws, stream=stream)
    return o, ml


def window_partial(layout: csa.Layout, prm: csa.csa_params_t, q, status, ws, stream=None):
    T, H = int(layout.tok_seq.shape[0]), int(prm.n_heads)
    o = torch.empty(T, H, int(prm.hd), dtype=torch.float32, device=q.device)
    ml = torch.empty(T, H, 2, dtype=torch.float32, device=q.device)
    csa.csa_window_attention(layout, prm, q, o, ml, status, ws, stream=stream)
    return o, ml


def combine(part_o, part_ml, status, sinks=None, stream=None):
    """Partials [P, T, H, 512] / [P, T, H, 2] -> out [T, H, 512]."""
    P, T, H, D = (int(x) for x in part_o.shape)
    out = torch.empty(T, H, D, dtype=torch.float32, device=part_o.device)
    csa.csa_shard_combine(part_o, part_ml, out, status, sinks=sinks, stream=stream)
    return out


def all_gather(x: torch.Tensor, group=None) -> torch.Tensor:
    """[world, *x.shape]: every rank's x, in rank order (NCCL on GPUs, gloo on CPU)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x.contiguous(), group=group)
    return torch.stack(parts)


def decode_local(shards: Sequence[Shard], layout: csa.Layout, prm: csa.csa_params_t, q_idx,
                 w_idx, q, status, sinks=None, stream=None):
    """All shards on one device, one after another; the exchanges are stacks.
    Returns (out [T, H, 512], idx [T, K], n_sel [T])."""
    bounds = [shards[0].lo] + [sh.hi for sh in shards]
    cands = [candidates(sh, layout, prm, q_idx, w_idx, status, stream) for sh in shards]
    cs = torch.stack([c[0] for c in cands])
    ci = torch.stack([c[1] for c in cands])
    cn = torch.stack([c[2] for c in cands])
    idx, n_sel, sidx, snsel = merge(bounds, cs, ci, cn, status, stream)
    parts = [partial(sh, layout, prm, sidx[g], snsel[g], q, status, stream)
             for g, sh in enumerate(shards)]
    parts.append(window_partial(layout, prm, q, status, shards[-1].ws, stream))
    po = torch.stack([p[0] for p in parts])
    pm = torch.stack([p[1] for p in parts])
    return combine(po, pm, status, sinks, stream), idx, n_sel


def decode_rank(sh: Shard, bounds: Sequence[int], layout: csa.Layout, prm: csa.csa_params_t,
                q_idx, w_idx, q, status, window_rank: int, sinks=None, group=None,
                stream=None):
    """This rank's part of a step with one shard per rank (torch.distributed
    initialised, rank g holding shard g); the window's partial is computed on
    window_rank (the rank whose layout's ring is current).  Every rank ends
    with the same (out, idx, n_sel)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    cs, ci, cn = candidates(sh, layout, prm, q_idx, w_idx, status, stream)
    gs, gi, gn = all_gather(cs, group), all_gather(ci, group), all_gather(cn, group)
    idx, n_sel, sidx, snsel = merge(bounds, gs, gi, gn, status, stream)
    po, pm = partial(sh, layout, prm, sidx[rank], snsel[rank], q, status, stream)
    if rank == window_rank:
        wo, wm = window_partial(layout, prm, q, status, sh.ws, stream)
    else:
        # no window rows here: a partial that carries nothing (m = -inf, l = 0)
        wo = torch.zeros_like(po)
        wm = torch.zeros_like(pm)
        wm[..., 0] = float("-inf")
    parts_o = torch.cat([all_gather(po, group), all_gather(wo, group)])
    parts_ml = torch.cat([all_gather(pm, group), all_gather(wm, group)])
    return combine(parts_o, parts_ml, status, sinks, stream), idx, n_sel


__all__ = ["Shard", "shard_bounds", "make_shard", "candidates", "merge", "partial",
           "window_partial", "combine", "all_gather", "decode_local", "decode_rank"]
