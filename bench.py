"""Benchmark: CSA decode tokens/s per layer at 1M context on GB300.

One step = one csa_decode (indexer -> top-k -> sparse shared-KV attention) for
one query token over one CSA layer holding 262,144 compressed blocks (64 MiB
of indexer keys, 256 MiB of 512-wide rows), top_k 1024, a 128-row window and
64 query heads.  Steps rotate over independent layer copies whose caches
total several times the 129 MB L2, so every step streams its keys from HBM.
Steps replay from a CUDA graph holding one step per rotating layer, back to
back as a model captures its layers together (a remainder from single-step
graphs); every step does all of its work.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the
same workload instead (the only other place this file runs the oracle).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import csa_workloads as W  # noqa: E402

METRIC = "CSA decode tokens/s per layer at 1M ctx (batch 1 & 32); % of HBM/tensor roofline"
UNIT = "tokens/s/layer"


# DRAM bytes (read + write) of one launch of the step's dominant kernel (the
# decode indexer with the top-k folded in) on the 1M workload, from the
# committed ncu capture of that step (profiles/), and the SHA-256 prefix of the
# kernel source it was taken on: once the source changes the figure no longer
# describes the kernel, and the roofline reports traffic null.
SELECT_TRAFFIC_BYTES = 67232512 + 129792
SELECT_TRAFFIC_SOURCE = "16e9667bff20d646"


def select_traffic():
    import hashlib
    src = os.path.join(ROOT, "sparse_compressed_kv_gb300", "csrc", "csa_indexer_topk.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return SELECT_TRAFFIC_BYTES if h == SELECT_TRAFFIC_SOURCE else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

class Layer:
    """One CSA layer's cache + one decode token's activations, on the GPU."""

    def __init__(self, wl: W.Workload, device, csa):
        d = wl.to(device)
        self.wl, self.d = wl, d
        self.layout = csa.Layout(d.tok_seq, d.tok_pos, d.comp_off, d.swa_kv, d.swa_first_pos,
                                 max_comp_rows=wl.max_comp_rows,
                                 total_comp_rows=int(wl.k_idx.shape[0]), swa_cap=wl.swa_cap)
        self.prm = csa.params(wl.n_heads, wl.top_k, wl.window, wl.ratio, wl.scale)
        T = wl.num_tokens
        self.out = torch.empty(T, wl.n_heads, wl.hd, dtype=torch.float32, device=device)
        self.idx = torch.empty(T, wl.top_k, dtype=torch.int32, device=device)


def algorithmic_bytes(wl: W.Workload):
    """Bytes the method must move for one step: the visible indexer keys, the
    selected and window rows, the token's activations and its f32 output."""
    keys = rows = scores = 0
    T = wl.num_tokens
    for t in range(T):
        b = int(wl.tok_seq[t])
        n_comp = int(wl.comp_off[b + 1] - wl.comp_off[b])
        p = int(wl.tok_pos[t])
        nv = min(n_comp, p // wl.ratio)
        keys += nv * wl.ihd * 2
        scores += nv * 4
        rows += (min(wl.top_k, nv) + min(wl.window, p + 1)) * wl.hd * 2
    act = T * (wl.n_ih * wl.ihd * 2 + wl.n_ih * 4 + wl.n_heads * wl.hd * 2)
    out = T * wl.n_heads * wl.hd * 4
    # the unfused API's extra traffic: the f32 score row written and read back
    # by the top-k, and the gathered rows written and read back by the attention
    unfused_extra = 2 * scores + 2 * rows
    return {"indexer": keys + T * (wl.n_ih * wl.ihd * 2 + wl.n_ih * 4),
            "step": keys + rows + act + out, "keys": keys, "rows": rows,
            "unfused_extra": unfused_extra}


def make_layers(name: str, n_layers: int, device, csa, seed0: int):
    gen_fn = {"1m": W.ctx1m, "batch32": W.batch32}[name]
    return [Layer(gen_fn(seed=seed0 + i, device=device), device, csa) for i in range(n_layers)]


def launches_in_graph(graph) -> int:
    """Kernel nodes in a captured CUDA graph (through the driver API)."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        h = ctypes.c_void_p(graph.raw_cuda_graph())
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(h, None, ctypes.byref(n)) != 0:
            return -1
        nodes = (ctypes.c_void_p * n.value)()
        cu.cuGraphGetNodes(h, nodes, ctypes.byref(n))
        kinds = ctypes.c_int(0)
        k = 0
        for i in range(n.value):
            cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(kinds))
            k += 1 if kinds.value == 0 else 0    # CU_GRAPH_NODE_TYPE_KERNEL
        return k
    except (OSError, AttributeError):
        return -1


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: every rank's steps must finish inside it."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def capture(fn, stream):
    """Capture fn() into a CUDA graph whose raw handle stays readable (torch
    >= 2.9 keeps it only with keep_graph=True, then instantiates on demand)."""
    try:
        g, kept = torch.cuda.CUDAGraph(keep_graph=True), True
    except TypeError:
        g, kept = torch.cuda.CUDAGraph(), False
    with torch.cuda.graph(g, stream=stream):
        fn()
    if kept:
        g.instantiate()
    return g


def time_graphs(graphs, steps, warmup, stream):
    """Replays go to torch's current stream, so make `stream` current: the
    events then bracket exactly the `steps` replays."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            graphs[(warmup + i) % len(graphs)].replay()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def time_steps(group, singles, steps, warmup, stream, blocks=1):
    """ms per step over `blocks` timed blocks of exactly `steps` steps each:
    replays of `group` (one graph holding one step per rotating layer, back to
    back as a model's layers are captured together), then single-step graphs
    for the remainder.  CUDA events on `stream`, which is made current so
    replays land on it; a barrier (synchronize) on both sides of each block.
    Returns the per-block times (ms per step)."""
    per = len(singles)
    out = []
    with torch.cuda.stream(stream):
        for i in range(max(1, -(-warmup // per))):
            group.replay()
        torch.cuda.synchronize()
        for _ in range(blocks):
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(steps // per):
                group.replay()
            for i in range(steps % per):
                singles[i].replay()
            t1.record(stream)
            torch.cuda.synchronize()
            out.append(t0.elapsed_time(t1) / steps)
    return out


def spread(xs):
    return {"median": round(statistics.median(xs), 5), "min": round(min(xs), 5),
            "max": round(max(xs), 5), "blocks": len(xs)}


def check_status(status, where):
    torch.cuda.synchronize()
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st:#x} in the {where} region")


def e2e_leg(layers, step, stream, steps, warmup, world, passes: int = 8):
    """The step through the public API with host buffers: every step copies
    its activations from pinned host memory, runs csa_decode and copies the
    output back to pinned host memory, all inside the timed region.  As a
    serving loop overlaps them, one CUDA graph holds `passes` rounds of one
    step per rotating layer, with two device sets of each layer's inputs and
    output (alternate rounds): each step's input copy (its three inputs
    packed in one pinned buffer) runs on its own stream as soon as the
    decode two rounds back has read the set, each output copy on
    a third stream right behind its decode, and the decode stream waits once
    per round (for that round's inputs and for the output copies two rounds
    back), so consecutive decodes keep their programmatic launch overlap;
    value = steps / time over whole replays.  `step(L, s, ins, out)` runs one
    decode of layer L on inputs `ins` = (q_idx, w_idx, q) into `out`."""
    nl = len(layers)

    def packed(like, device, pin):
        # the step's three inputs back to back in one byte buffer (offsets
        # 256-byte aligned), so that each step's input copy is one copy;
        # returns the buffer and views of it shaped like `like`
        offs, off = [], 0
        for t in like:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = tuple(buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                      for o, t in zip(offs, like))
        return buf, views

    hpk = []
    for L in layers:
        buf, views = packed((L.d.q_idx, L.d.w_idx, L.d.q), "cpu", True)
        for v, t in zip(views, (L.d.q_idx, L.d.w_idx, L.d.q)):
            v.copy_(t.cpu())
        hpk.append(buf)
    dpk, dins = [], []
    for L in layers:
        sets = [packed((L.d.q_idx, L.d.w_idx, L.d.q), stream.device, False) for _ in range(2)]
        dpk.append([b for b, _ in sets])
        dins.append([v for _, v in sets])
    hout = [torch.empty(layers[0].out.shape, dtype=torch.float32).pin_memory() for _ in layers]
    douts = [[torch.empty_like(L.out) for _ in range(2)] for L in layers]
    s_in = torch.cuda.Stream(device=stream.device)
    s_out = torch.cuda.Stream(device=stream.device)
    n = passes * nl

    def pipeline():
        fork = torch.cuda.Event()
        fork.record(stream)
        s_in.wait_event(fork)
        s_out.wait_event(fork)
        h2d = [torch.cuda.Event() for _ in range(n)]
        dec = [torch.cuda.Event() for _ in range(n)]
        d2h = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            j, r = i % nl, (i // nl) % 2
            with torch.cuda.stream(s_in):
                if i >= 2 * nl:
                    s_in.wait_event(dec[i - 2 * nl])   # the last decode that read this set
                dpk[j][r].copy_(hpk[j], non_blocking=True)
                h2d[i].record(s_in)
        for i in range(n):
            j, r = i % nl, (i // nl) % 2
            if i % nl == 0:
                # once per round: its inputs, and the output copies that read
                # this round's output set two rounds back
                for k in range(i, i + nl):
                    stream.wait_event(h2d[k])
                for k in range(max(0, i - 2 * nl), i - nl):
                    stream.wait_event(d2h[k])
            step(layers[j], stream, dins[j][r], douts[j][r])
            dec[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(dec[i])
                hout[j].copy_(douts[j][r], non_blocking=True)
                d2h[i].record(s_out)
        join_in, join_out = torch.cuda.Event(), torch.cuda.Event()
        join_in.record(s_in)
        join_out.record(s_out)
        stream.wait_event(join_in)
        stream.wait_event(join_out)
    with torch.cuda.stream(stream):
        pipeline()
    torch.cuda.synchronize()
    g = capture(pipeline, stream)
    reps = max(1, (max(3, steps) + n - 1) // n)
    wreps = max(1, (warmup + n - 1) // n)
    with torch.cuda.stream(stream):
        for _ in range(wreps):
            g.replay()
        torch.cuda.synchronize()
        t_start = time.perf_counter()
        for _ in range(reps):
            g.replay()
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t_start) * 1e3 / (reps * n)
    # the copies carried the right data: each layer's last host output equals,
    # bit for bit, what the device-timed steps left in its output
    same = all(torch.equal(hout[j], layers[j].out.cpu()) for j in range(nl))
    h2d_b = hpk[0].numel()   # the three inputs (and any alignment gap between them)
    return {"value": round(world * 1e3 / e2e_ms, 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d_b), "d2h_bytes_per_step": int(hout[0].numel() * 4),
            "ms_per_step": round(e2e_ms, 5), "steps_timed": reps * n,
            "outputs_equal_device_path": bool(same),
            "launch": f"one CUDA graph of {n} steps ({passes} rounds of {nl} layers, two device "
                      "sets of inputs and outputs per layer): each step's inputs in one copy "
                      "(packed q_idx, w_idx, q) on one stream, csa_decode on another (one wait "
                      "per round), each output copy on a third behind its decode"}


def ctx64k_leg(device, csa, stream, status, reps, seed):
    """The 64K workload's 100 consecutive decode steps: step i queries
    position 65536 + i, appends that position's row to the window ring and,
    when a block completes, makes it visible (its key and row are written into
    the caches).  All 100 steps are captured in one graph (the ring is first
    restored to step 0's contents) and replayed; value = steps / time."""
    wl = W.ctx64k(seed=seed)
    gen = torch.Generator().manual_seed(1234)
    steps = 100
    ring0 = wl.swa_kv.clone()
    pos, off, first, rows, qi, wi, qq = [], [], [], [], [], [], []
    for i in range(steps):
        if i:
            W.ctx64k_step(wl, i, gen)
        p = int(wl.tok_pos[0])
        pos.append(wl.tok_pos.clone())
        off.append(wl.comp_off.clone())
        first.append(wl.swa_first_pos.clone())
        rows.append(wl.swa_kv[0, p % wl.swa_cap].clone())
        qi.append(wl.q_idx.clone())
        wi.append(wl.w_idx.clone())
        qq.append(wl.q.clone())
    d = wl.to(device)
    d.swa_kv.copy_(ring0.to(device))
    ring0_d = ring0.to(device)
    pos_d = [x.to(device) for x in pos]
    off_d = [x.to(device) for x in off]
    first_d = [x.to(device) for x in first]
    rows_d = torch.stack(rows).to(device)
    qi_d = [x.to(device) for x in qi]
    wi_d = [x.to(device) for x in wi]
    qq_d = [x.to(device) for x in qq]
    # cache rows written by the steps that complete a block (drawn with the buffers)
    k_src = d.k_idx.clone()
    kv_src = d.comp_kv.clone()
    cap = int(wl.k_idx.shape[0])
    prm = csa.params(wl.n_heads, wl.top_k, wl.window, wl.ratio, wl.scale)
    lays = [csa.Layout(d.tok_seq, pos_d[i], off_d[i], d.swa_kv, first_d[i], max_comp_rows=cap,
                       total_comp_rows=cap, swa_cap=wl.swa_cap) for i in range(steps)]
    ws = csa.workspace(lays[0], prm)
    out = torch.empty(1, wl.n_heads, wl.hd, dtype=torch.float32, device=device)

    def run_all():
        d.swa_kv.copy_(ring0_d)
        for i in range(steps):
            p = int(pos[i][0])
            if i:
                d.swa_kv[0, p % wl.swa_cap].copy_(rows_d[i])
                if int(off[i][1]) > int(off[i - 1][1]):
                    b = int(off[i][1]) - 1
                    d.k_idx[b].copy_(k_src[b])
                    d.comp_kv[b].copy_(kv_src[b])
            csa.csa_decode(lays[i], prm, qi_d[i], wi_d[i], d.k_idx, d.comp_kv, qq_d[i], out,
                           status, ws, stream=stream)

    with torch.cuda.stream(stream):
        run_all()
    check_status(status, "64k")
    g = capture(run_all, stream)
    ms = time_graphs([g], reps, 2, stream)
    check_status(status, "64k")
    return {"workload": "64k: 100 consecutive decode steps at positions 65536..65635, "
                        "16384..16408 visible blocks, top_k 1024, 64 heads; each step appends "
                        "its window row, every 4th a compressed block; one graph of 100 steps",
            "tokens_per_s_per_layer": round(steps * 1e3 / ms, 1),
            "us_per_step": round(ms * 1e3 / steps, 3), "replays": reps,
            "l2": "hot: one layer's 4 MiB of keys and 16 MiB of rows stay in L2 across steps"}


def decode_only_leg(args, device):
    """Eager decode steps of one workload on two rotating layers, one stream,
    events around --steps of them after --warmup: a short, fixed launch
    sequence for profilers (not a bench value)."""
    from sparse_compressed_kv_gb300 import build as cuda_build
    from sparse_compressed_kv_gb300 import csa
    cuda_build.build()
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    name = args.decode_only
    if name == "hca1m":
        wls = [W.hca1m(seed=500 + i, device=device) for i in range(2)]
        runs = []
        for wl in wls:
            d = wl.to(device)
            lay = csa.Layout(d.tok_seq, d.tok_pos, d.comp_off, d.swa_kv, d.swa_first_pos,
                             max_comp_rows=wl.max_comp_rows,
                             total_comp_rows=int(wl.comp_kv.shape[0]), swa_cap=wl.swa_cap)
            prm = csa.params(wl.n_heads, 1, wl.window, wl.ratio, wl.scale)
            runs.append((d, lay, prm, torch.empty(1, wl.n_heads, wl.hd, device=device)))
        ws = csa.hca_workspace(runs[0][1], runs[0][2])

        def step(i):
            d, lay, prm, out = runs[i % 2]
            csa.csa_hca_decode(lay, prm, d.comp_kv, d.q, out, status, ws, stream=stream)
    elif name == "fp4":
        # the 1m workload with its keys quantized to MXFP4 once, before the steps
        layers = make_layers("1m", 2, device, csa, seed0=0)
        ws = csa.workspace(layers[0].layout, layers[0].prm)
        rows = []
        for L in layers:
            r = torch.empty(L.wl.k_idx.shape[0], csa.FP4_ROW, dtype=torch.uint8, device=device)
            csa.csa_fp4_quantize_keys(L.d.k_idx, r, stream=stream)
            rows.append(r)

        def step(i):
            L = layers[i % 2]
            csa.csa_decode_fp4(L.layout, L.prm, L.d.q_idx, L.d.w_idx, rows[i % 2], L.d.comp_kv, L.d.q,
                               L.out, status, ws, idx_out=L.idx, stream=stream)
    else:
        layers = make_layers(name, 2, device, csa, seed0=0 if name == "1m" else 77)
        ws = csa.workspace(layers[0].layout, layers[0].prm)

        def step(i):
            L = layers[i % 2]
            csa.csa_decode(L.layout, L.prm, L.d.q_idx, L.d.w_idx, L.d.k_idx, L.d.comp_kv, L.d.q,
                           L.out, status, ws, idx_out=L.idx, stream=stream)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    check_status(status, name)
    return {"decode_only": name, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step_eager": round(e0.elapsed_time(e1) / args.steps, 5)}


def prefill_leg(args, device, csa, stream, status, rank, tf_peak, peak_kind):
    """The indexer alone on a chunked-prefill workload: `args.prefill_tokens`
    query tokens of one sequence at positions 262144.. share every key tile
    (four tokens per MMA), timed from replays of a one-launch graph."""
    pl = Layer(W.prefill(seed=900 + 1000 * rank, tokens=args.prefill_tokens, device=device),
               device, csa)
    pw = pl.wl
    psc = torch.empty(pw.num_tokens, pw.max_comp_rows, dtype=torch.float32, device=device)

    def pstep():
        csa.csa_indexer_scores(pl.layout, pl.prm, pl.d.q_idx, pl.d.w_idx, pl.d.k_idx, psc,
                               status, stream=stream)
    with torch.cuda.stream(stream):
        pstep()
    torch.cuda.synchronize()
    pgraph = capture(pstep, stream)
    reps = max(3, min(20, args.steps // 10))
    pms = time_graphs([pgraph], reps, 3, stream)
    nvis = [min(int(pw.comp_off[1]), int(pw.tok_pos[t]) // pw.ratio)
            for t in range(pw.num_tokens)]
    flops = 2.0 * pw.n_ih * pw.ihd * float(sum(nvis))
    tflops = flops / (pms * 1e-3) / 1e12
    check_status(status, "prefill")
    return {"workload": f"prefill: indexer alone, {pw.num_tokens} tokens at p = 262144.., "
                        f"65,536..{max(nvis)} visible blocks each, 64 heads x 128",
            "ms_per_launch": round(pms, 4), "tflops": round(tflops, 1),
            "peak_tflops": tf_peak, "peak_kind": peak_kind + " bf16 burst",
            "frac": round(tflops / tf_peak, 4), "launches": reps + 4}


def run_ours(args, rank, world, device):
    from sparse_compressed_kv_gb300 import csa
    from sparse_compressed_kv_gb300 import build as cuda_build
    cuda_build.build()
    csa.load()
    hbm_peak, tf_peak, peak_kind = peaks()
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)

    layers = make_layers("1m", args.layers, device, csa, seed0=1000 * rank)
    wl0 = layers[0].wl
    ab = algorithmic_bytes(wl0)
    ws = csa.workspace(layers[0].layout, layers[0].prm)

    def step(L, s):
        csa.csa_decode(L.layout, L.prm, L.d.q_idx, L.d.w_idx, L.d.k_idx, L.d.comp_kv, L.d.q,
                       L.out, status, ws, idx_out=L.idx, stream=s)

    # eager warm-up outside capture (sets kernel attributes, caches device info)
    with torch.cuda.stream(stream):
        for L in layers:
            step(L, stream)
    torch.cuda.synchronize()
    graphs = [capture(lambda L=L: step(L, stream), stream) for L in layers]
    group = capture(lambda: [step(L, stream) for L in layers], stream)
    per_step_launches = launches_in_graph(graphs[0])

    # ---- timed region: `blocks` blocks of exactly `steps` decode steps
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    blocks = time_steps(group, graphs, args.steps, args.warmup, stream, blocks=args.blocks)
    clk = clocks.stop()
    ms = max_over_ranks(statistics.median(blocks), device)
    check_status(status, "timed")
    assert torch.isfinite(layers[0].out).all()
    # the step's own result for layer 0 (compared with the oracle in cpu_baseline)
    with torch.cuda.stream(stream):
        step(layers[0], stream)
    torch.cuda.synchronize()
    res0 = (layers[0].idx[0].cpu().numpy().copy(), layers[0].out[0].cpu().numpy().copy())

    # ---- the dominant kernel alone (the indexer with the top-k folded in, as
    # the step runs it): one graph holds one launch per rotating layer, so
    # replays carry no host overhead; CUDA events on `stream`
    nsel_buf = torch.empty(wl0.num_tokens, dtype=torch.int32, device=device)

    def select_all():
        for L in layers:
            csa.csa_indexer_topk(L.layout, L.prm, L.d.q_idx, L.d.w_idx, L.d.k_idx, L.idx, nsel_buf,
                                 status, ws, stream=stream)
    with torch.cuda.stream(stream):
        select_all()
    torch.cuda.synchronize()
    sgraph = capture(select_all, stream)
    reps = max(1, args.steps // len(layers))
    sel_blocks = [time_graphs([sgraph], reps, max(1, args.warmup // len(layers)), stream)
                  / len(layers) for _ in range(args.blocks)]
    sel_ms = statistics.median(sel_blocks)

    # ---- the indexer's scores alone (the same kernel without the selection)
    sc_buf = torch.empty(1, wl0.max_comp_rows, dtype=torch.float32, device=device)

    def index_all():
        for L in layers:
            csa.csa_indexer_scores(L.layout, L.prm, L.d.q_idx, L.d.w_idx, L.d.k_idx, sc_buf,
                                   status, stream=stream)
    with torch.cuda.stream(stream):
        index_all()
    torch.cuda.synchronize()
    igraph = capture(index_all, stream)
    idx_blocks = [time_graphs([igraph], reps, max(1, args.warmup // len(layers)), stream)
                  / len(layers) for _ in range(args.blocks)]
    idx_ms = statistics.median(idx_blocks)

    line_extra = {}
    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        def e2e_step(L, s, ins, out):
            csa.csa_decode(L.layout, L.prm, ins[0], ins[1], L.d.k_idx, L.d.comp_kv, ins[2], out,
                           status, ws, idx_out=L.idx, stream=s)
        line_extra["e2e"] = e2e_leg(layers, e2e_step, stream, args.steps, args.warmup, world)
        check_status(status, "e2e")

    # ---- next row: the same 1M step with the indexer keys cached as MXFP4
    # (80 bytes per key instead of 256); the cache is quantized once, untimed
    if not args.no_fp4:
        frows = []
        for L in layers:
            r = torch.empty(L.wl.k_idx.shape[0], csa.FP4_ROW, dtype=torch.uint8, device=device)
            csa.csa_fp4_quantize_keys(L.d.k_idx, r, stream=stream)
            frows.append(r)

        def fstep(i, s):
            L = layers[i]
            csa.csa_decode_fp4(L.layout, L.prm, L.d.q_idx, L.d.w_idx, frows[i], L.d.comp_kv,
                               L.d.q, L.out, status, ws, idx_out=L.idx, stream=s)

        def findex_all():
            for i, L in enumerate(layers):
                csa.csa_indexer_scores_fp4(L.layout, L.prm, L.d.q_idx, L.d.w_idx, frows[i],
                                           sc_buf, status, stream=stream)
        with torch.cuda.stream(stream):
            for i in range(len(layers)):
                fstep(i, stream)
            findex_all()
        torch.cuda.synchronize()
        fsingles = [capture(lambda i=i: fstep(i, stream), stream) for i in range(len(layers))]
        fgroup = capture(lambda: [fstep(i, stream) for i in range(len(layers))], stream)
        fms = statistics.median(time_steps(fgroup, fsingles, args.steps, args.warmup, stream,
                                           blocks=args.blocks))
        figraph = capture(findex_all, stream)
        fims = time_graphs([figraph], max(1, args.steps // len(layers)),
                           max(1, args.warmup // len(layers)), stream) / len(layers)
        # the FP4 selection against the bf16 one on every layer (each exact on
        # its own scores; the bf16 selection is the oracle's, see cpu_baseline)
        rec, planted_kept = [], 0
        for i, L in enumerate(layers):
            ib = torch.empty_like(L.idx)
            csa.csa_decode(L.layout, L.prm, L.d.q_idx, L.d.w_idx, L.d.k_idx, L.d.comp_kv, L.d.q,
                           L.out, status, ws, idx_out=ib, stream=stream)
            fstep(i, stream)
            torch.cuda.synchronize()
            sb = set(ib[0].cpu().tolist()) - {-1}
            sf = set(L.idx[0].cpu().tolist()) - {-1}
            rec.append(len(sb & sf) / max(1, len(sb)))
            if L.wl.planted is not None:
                planted_kept += int(all(int(b) in sf for b in L.wl.planted.tolist()))
        nv = ab["keys"] // (wl0.ihd * 2)
        fidx_bytes = nv * csa.FP4_ROW + (ab["indexer"] - ab["keys"])
        fstep_bytes = ab["step"] - ab["keys"] + nv * csa.FP4_ROW
        line_extra["fp4"] = {
            "workload": "1m with MXFP4 indexer keys (80 B per key: 20 MiB instead of 64 MiB)",
            "tokens_per_s_per_layer": round(world * 1e3 / fms, 1),
            "ms_per_step": round(fms, 5), "indexer_ms": round(fims, 5),
            "indexer_bytes_per_launch": int(fidx_bytes),
            "indexer_hbm_frac": round(fidx_bytes / (fims * 1e-3) / 1e9 / hbm_peak, 4),
            "step_algorithmic_bytes": int(fstep_bytes),
            "step_hbm_frac": round(fstep_bytes / (fms * 1e-3) / 1e9 / hbm_peak, 4),
            "recall_vs_bf16": {"min": round(min(rec), 6), "mean": round(statistics.mean(rec), 6),
                               "layers": len(rec), "planted_all_selected_layers": planted_kept}}
        del fsingles, fgroup, figraph, frows
        check_status(status, "FP4")

    del graphs, group
    # ---- the 64K workload: 100 consecutive decode steps of one layer
    if not args.no_64k:
        torch.cuda.empty_cache()
        line_extra["ctx64k"] = ctx64k_leg(device, csa, stream, status,
                                          reps=max(3, args.steps // 10), seed=7 + 1000 * rank)

    # ---- secondary: batched decode, 32 ragged sequences (32K..128K)
    if not args.no_batch32:
        torch.cuda.empty_cache()
        blayers = make_layers("batch32", 2, device, csa, seed0=77 + 1000 * rank)
        bws = csa.workspace(blayers[0].layout, blayers[0].prm)

        def bstep(L, s):
            csa.csa_decode(L.layout, L.prm, L.d.q_idx, L.d.w_idx, L.d.k_idx, L.d.comp_kv, L.d.q,
                           L.out, status, bws, idx_out=L.idx, stream=s)
        with torch.cuda.stream(stream):
            for L in blayers:
                bstep(L, stream)
        torch.cuda.synchronize()
        bgraphs = [capture(lambda L=L: bstep(L, stream), stream) for L in blayers]
        bgroup = capture(lambda: [bstep(L, stream) for L in blayers], stream)
        bms = statistics.median(time_steps(bgroup, bgraphs, args.steps, args.warmup, stream,
                                           blocks=args.blocks))
        bab = sum(algorithmic_bytes(L.wl)["step"] for L in blayers) / len(blayers)
        line_extra["batch32"] = {
            "workload": "batch32: 32 sequences, contexts U{32K..128K}, one token each",
            "tokens_per_s_per_layer": round(32 * 1e3 / bms, 1), "ms_per_step": round(bms, 5),
            "algorithmic_bytes_per_step": int(bab),
            "hbm_frac": round(bab / (bms * 1e-3) / 1e9 / hbm_peak, 4),
            "launches_per_step": launches_in_graph(bgraphs[0])}
        del bgraphs, bgroup, blayers
        check_status(status, "batch32")

    # ---- next row: HCA decode at 1M context (8192 compressed rows, dense)
    if not args.no_hca:
        torch.cuda.empty_cache()
        hl = [W.hca1m(seed=500 + i + 1000 * rank, device=device) for i in range(32)]
        hd = []
        for wl in hl:
            d = wl.to(device)
            lay = csa.Layout(d.tok_seq, d.tok_pos, d.comp_off, d.swa_kv, d.swa_first_pos,
                             max_comp_rows=wl.max_comp_rows,
                             total_comp_rows=int(wl.comp_kv.shape[0]), swa_cap=wl.swa_cap)
            prm = csa.params(wl.n_heads, 1, wl.window, wl.ratio, wl.scale)
            hd.append((wl, d, lay, prm, torch.empty(1, wl.n_heads, wl.hd, device=device)))
        hws = csa.hca_workspace(hd[0][2], hd[0][3])

        def hstep(x, s):
            wl, d, lay, prm, out = x
            csa.csa_hca_decode(lay, prm, d.comp_kv, d.q, out, status, hws, stream=s)
        with torch.cuda.stream(stream):
            for x in hd:
                hstep(x, stream)
        torch.cuda.synchronize()
        hgraphs = [capture(lambda x=x: hstep(x, stream), stream) for x in hd]
        hgroup = capture(lambda: [hstep(x, stream) for x in hd], stream)
        hms = statistics.median(time_steps(hgroup, hgraphs, args.steps, args.warmup, stream,
                                           blocks=args.blocks))
        hbytes = (8192 + 128) * 1024 + 64 * 1024 + 64 * 2048
        line_extra["hca"] = {
            "workload": "hca1m: HCA decode, 1 token, ratio 128, 8192 compressed rows + 128 "
                        "window rows, 64 heads, dense (32 rotating layers, 270 MB)",
            "tokens_per_s_per_layer": round(world * 1e3 / hms, 1),
            "ms_per_step": round(hms, 5), "algorithmic_bytes_per_step": hbytes,
            "hbm_frac": round(hbytes / (hms * 1e-3) / 1e9 / hbm_peak, 4),
            "launches_per_step": launches_in_graph(hgraphs[0])}
        del hd, hgraphs, hgroup, hl
        check_status(status, "HCA")

    # ---- prefill indexer alone: query tokens of one sequence share every key
    # tile (four tokens per MMA), the tensor-bound case
    if not args.no_prefill:
        torch.cuda.empty_cache()
        line_extra["prefill_indexer"] = prefill_leg(args, device, csa, stream, status, rank,
                                                    tf_peak, peak_kind)

    tok_s = world * 1e3 / ms
    achieved = ab["indexer"] / (sel_ms * 1e-3) / 1e9
    idx_achieved = ab["indexer"] / (idx_ms * 1e-3) / 1e9
    n_vis0 = ab["keys"] // (wl0.ihd * 2)
    line = {
        "metric": METRIC, "value": round(tok_s, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "ms_per_step_blocks": spread(blocks),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "1m: CSA decode, 1 token, 262144 blocks (64 MiB keys, 256 MiB "
                               "rows), top_k 1024, window 128, 64 heads, hd 512, 32 planted",
                   "layers_rotated": args.layers,
                   "l2": f"inputs > L2: {args.layers} independent layer caches "
                         f"({args.layers * 0.34:.1f} GB) rotated, no flush",
                   "parallelism": f"replicas x{world}",
                   "graph": f"one CUDA graph per {len(layers)} steps (one per rotating layer)"},
        "roofline": {"bound": "hbm", "kernel": "indexer + top-k (csa_indexer_topk: tcgen05, TMA)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": select_traffic(),
                     "peak_kind": peak_kind, "kernel_ms": round(sel_ms, 5),
                     "kernel_ms_blocks": spread(sel_blocks),
                     "bytes_per_launch": ab["indexer"]},
        "indexer_scores_alone": {"kernel": "the same indexer without the selection "
                                           "(csa_indexer_scores)",
                                 "achieved": round(idx_achieved, 1), "unit": "GB/s",
                                 "frac": round(idx_achieved / hbm_peak, 4),
                                 "kernel_ms": round(idx_ms, 5),
                                 "kernel_ms_blocks": spread(idx_blocks)},
        "indexer_keys_per_s": round(n_vis0 / (idx_ms * 1e-3), 1),
        "unfused_extra_bytes_per_step": ab["unfused_extra"],
        "step_roofline": {"bound": "hbm", "algorithmic_bytes": ab["step"],
                          "achieved": round(ab["step"] / (ms * 1e-3) / 1e9, 1),
                          "peak": hbm_peak, "unit": "GB/s",
                          "frac": round(ab["step"] / (ms * 1e-3) / 1e9 / hbm_peak, 4)},
        "gpu_launches": per_step_launches * args.steps if per_step_launches > 0 else None,
        "launches_per_step": per_step_launches,
        "clocks": clk,
    }
    line.update(line_extra)
    return line, wl0, res0


# ---------------------------------------------------------------- CPU oracle

def oracle_step(wl):
    import oracle
    return oracle.decode(W.bits(wl.q_idx), wl.w_idx.numpy(), W.bits(wl.k_idx), W.bits(wl.comp_kv),
                         W.bits(wl.swa_kv), W.bits(wl.q), wl.tok_seq.numpy(), wl.tok_pos.numpy(),
                         wl.comp_off.numpy(), wl.swa_first_pos.numpy(), top_k=wl.top_k,
                         window=wl.window, ratio=wl.ratio, scale=wl.scale)


def cpu_baseline(steps: int, wl=None, gpu=None):
    """The oracle as it stands, on full 1M decode steps (one token, one layer
    each), on the GPU leg's first layer when given (else a fresh seeded one).
    With the GPU's result for that layer, also its recall against the
    oracle's selection and the max-abs difference of the outputs."""
    import oracle
    oracle.build()
    wl = W.ctx1m(seed=0) if wl is None else wl.to("cpu")
    idx, n_sel, out = oracle_step(wl)   # warm (page in) and the reference result
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(wl)
    dt = (time.perf_counter() - t0) / steps
    res = {"value": round(1.0 / dt, 4), "unit": UNIT, "cores": oracle.num_threads(),
           "kind": "oracle",
           "sample": f"{steps} full 1m decode steps (262144 blocks, top_k 1024, 64 heads), f64"}
    if gpu is not None:
        gidx, gout = gpu
        k = int(n_sel[0])
        ref = set(idx[0, :k].tolist())
        got = set(int(x) for x in gidx if x >= 0)
        res["vs_gpu"] = {
            "recall": round(len(ref & got) / max(1, len(ref)), 6),
            "max_abs_err": float(np.abs(gout.astype(np.float64) - out[0]).max()),
            "planted_selected": int(len(set(wl.planted.tolist()) & got))
            if wl.planted is not None else None,
            "what": "GPU csa_decode on the timed layer 0 vs the f64 oracle's whole step "
                    "(its own selection)"}
    return res


class OracleSlices:
    """The oracle's decode of one 1m token, cut into `m` steps: steps 0..m-1
    each score a contiguous slice of the blocks (the oracle's indexer on a
    sub-range of the cache); the last one also runs the oracle's top-k, mixed
    gather and attention on the whole score row.  m steps = one token."""

    def __init__(self, wl, m: int):
        import oracle
        self.o = oracle
        self.wl = wl
        self.m = m
        n = int(wl.comp_off[1])
        self.n = n
        self.cuts = [n * i // m for i in range(m + 1)]
        self.scores = np.zeros(n)
        self.qb, self.kb = W.bits(wl.q_idx), W.bits(wl.k_idx)
        self.w = wl.w_idx.numpy()
        self.i = 0

    def step(self):
        o, wl = self.o, self.wl
        j = self.i % self.m
        a, b = self.cuts[j], self.cuts[j + 1]
        if b > a:
            sc, _ = o.indexer_scores(self.qb, self.w, self.kb, [0], [4 * (b - a)], [a, b])
            self.scores[a:b] = sc[0, : b - a]
        if j == self.m - 1:
            idx, ns = o.topk(self.scores, wl.top_k)
            kv, kl = o.gather(idx[None], np.array([ns], np.int32), W.bits(wl.comp_kv),
                              W.bits(wl.swa_kv), wl.tok_seq.numpy(), wl.tok_pos.numpy(),
                              wl.comp_off.numpy(), wl.swa_first_pos.numpy(), top_k=wl.top_k,
                              window=wl.window, ratio=wl.ratio)
            o.attention(W.bits(wl.q), kv, kl, wl.scale)
        self.i += 1


def run_reference(args):
    """--impl reference: the CPU oracle timed on this workload, K steps after W.
    A step is 1/m of one token's decode, m sized so the run takes ~2-3 minutes."""
    import oracle
    oracle.build()
    wl = W.ctx1m(seed=0)
    per_token_s = 2.0                      # ~1.6 s measured on 8 cores; a generous bound
    m = max(1, int(np.ceil((args.steps + args.warmup) * per_token_s / 150.0)))
    sl = OracleSlices(wl, m)
    for _ in range(args.warmup):
        sl.step()
    sl.i = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sl.step()
    dt = time.perf_counter() - t0
    v = round((args.steps / m) / dt, 4)
    sample = (f"each step = 1/{m} of one full 1m decode token (indexer over a contiguous "
              f"1/{m} of the 262144 blocks; every {m}th step also top-k, gather, attention); "
              f"value = (steps/{m}) tokens / time")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "1m: CSA decode, 1 token, 262144 blocks (64 MiB keys, 256 MiB "
                               "rows), top_k 1024, window 128, 64 heads, hd 512, 32 planted",
                   "slices_per_token": m},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--cpu-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-batch32", action="store_true")
    ap.add_argument("--no-hca", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-fp4", action="store_true")
    ap.add_argument("--no-64k", action="store_true")
    ap.add_argument("--blocks", type=int, default=5,
                    help="timed blocks of --steps steps each; the median is reported")
    ap.add_argument("--prefill-tokens", type=int, default=4096)
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill-indexer leg and print its object (for profiling)")
    ap.add_argument("--decode-only", choices=["1m", "batch32", "hca1m", "fp4"], default=None,
                    help="run only eager decode steps of this workload (2 rotating layers) and "
                         "print their mean time (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        # the oracle arm runs on rank 0 only; the other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    if args.decode_only:
        print(json.dumps(decode_only_leg(args, device)), flush=True)
        return
    if args.prefill_only:
        from sparse_compressed_kv_gb300 import build as cuda_build
        from sparse_compressed_kv_gb300 import csa
        cuda_build.build()
        _, tf_peak, peak_kind = peaks()
        torch.cuda.set_device(device)
        stream = torch.cuda.Stream(device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        print(json.dumps(prefill_leg(args, device, csa, stream, status, rank, tf_peak,
                                     peak_kind)), flush=True)
        return
    line, wl0, res0 = run_ours(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_steps, wl0, res0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
