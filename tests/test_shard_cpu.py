"""The sharded single-sequence step's exchanges on CPU: gloo, world size 2.

Each rank owns half of one sequence's blocks.  It takes its best top_k
blocks (the oracle's scores and top-k on its range), the ranks exchange them
with the library's all-gather, and the best top_k of the gathered candidates
by (score descending, block ascending) must be the whole row's top-k.  Each
rank then forms the oracle partial of its selected rows (rank 1 also the
window's), the partials are exchanged the same way, and their log-sum-exp
merge must equal the oracle's attention over all the rows.  The GPU kernels
of the same steps are covered by tests/test_gpu_shard.py.
"""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import csa_workloads as W
    import oracle
    from sparse_compressed_kv_gb300 import shard
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = W.make("shardcpu", seed=60, seq_lens=[4 * 600], n_comp=[600], top_k=64, n_heads=16)
        K = wl.top_k
        sc, _ = oracle.indexer_scores(W.bits(wl.q_idx), wl.w_idx.numpy(), W.bits(wl.k_idx),
                                      wl.tok_seq.numpy(), wl.tok_pos.numpy(),
                                      wl.comp_off.numpy())
        row = sc[0]                                              # [600] f64
        bounds = shard.shard_bounds(600, world)
        lo, hi = bounds[rank], bounds[rank + 1]
        # this rank's candidates: its range's best K by the oracle's rule
        loc, n_loc = oracle.topk(row[lo:hi].copy(), K)
        cand_idx = np.full(K, -1, np.int64)
        cand_sc = np.full(K, -np.inf)
        cand_idx[:n_loc] = lo + loc[:n_loc]
        cand_sc[:n_loc] = row[lo + loc[:n_loc]]
        g_idx = shard.all_gather(torch.from_numpy(cand_idx)).numpy()      # [world, K]
        g_sc = shard.all_gather(torch.from_numpy(cand_sc)).numpy()
        flat_i, flat_s = g_idx.reshape(-1), g_sc.reshape(-1)
        keep = flat_i >= 0
        order = np.lexsort((flat_i[keep], -flat_s[keep]))          # score desc, index asc
        merged = np.sort(flat_i[keep][order][:K])
        want, n_want = oracle.topk(row.copy(), K)
        ok_sel = n_want == K and np.array_equal(merged, want[:K])

        # partials: this rank's selected rows; the window on rank 1
        kv, kl = oracle.gather(want[None].astype(np.int32), np.array([n_want], np.int32),
                               W.bits(wl.comp_kv), W.bits(wl.swa_kv), wl.tok_seq.numpy(),
                               wl.tok_pos.numpy(), wl.comp_off.numpy(),
                               wl.swa_first_pos.numpy(), top_k=K, window=wl.window,
                               ratio=wl.ratio)
        mine = [j for j in range(n_want) if lo <= want[j] < hi]
        qb = W.bits(wl.q)[0]
        O, m, lv = oracle.attention_partial(qb, kv[0, mine], wl.scale)
        wrows = kv[0, n_want:int(kl[0])] if rank == 1 else kv[0, :0]
        wO, wm, wl_ = oracle.attention_partial(qb, wrows, wl.scale)
        gO = torch.cat([shard.all_gather(torch.from_numpy(O)), shard.all_gather(torch.from_numpy(wO))])
        gm = torch.cat([shard.all_gather(torch.from_numpy(m)), shard.all_gather(torch.from_numpy(wm))])
        gl = torch.cat([shard.all_gather(torch.from_numpy(lv)), shard.all_gather(torch.from_numpy(wl_))])
        out = oracle.combine_partials(gO.numpy(), gm.numpy(), gl.numpy())
        ref = oracle.attention(W.bits(wl.q), kv, kl, wl.scale)[0]
        err = float(np.abs(out - ref).max())
        q.put((rank, bool(ok_sel), err, int(n_loc)))
    finally:
        torch.distributed.destroy_process_group()


def test_sharded_exchange_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ok_sel, err, n_loc in res:
        assert ok_sel, f"rank {rank}: merged selection differs from the whole row's top-k"
        assert err < 1e-12, f"rank {rank}: merged output off by {err}"
        assert n_loc > 0
