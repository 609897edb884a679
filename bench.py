"""Benchmark of the k8v4 decode hot path on GB300.

Workload (the 238K point of the long-context sweep): one sequence of 237,568
cells, 2 KV heads x 256, 16 query heads (GQA 8), page size 64, shuffled page
table, bf16 K/V/q N(0,1) with 3 outlier channels per head x20.  One step is the
engine's decode step: append the newest token's K/V (quantise + paged write)
and run split-K decode attention over all 237,568 cells (partials + combine with
the inverse Walsh-Hadamard transform), issued as one attn_k8v4_decode_step call.  Two cache replicas alternate between
steps (388 MB > L2), so every step streams its cache from HBM.

Metric: decode-attention GB/s over 816 B/cell (and cells/s); the same line also
reports append cells/s (bulk append of the whole cache, 2,864 B/cell of
algorithmic traffic), the INT8/INT8 (1,056 B/cell) and q4_0 K+V (576 B/cell)
comparison arms, the roofline of the decode call, the end-to-end rate through
the C ABI with host buffers, and the CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl k8v4|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path
has no exchange step); value = cells of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

N_CELLS = 237568
P = 64
H = 2
HQ = 16
CELL_BYTES = 816
CELL_BYTES_INT8 = 1056
CELL_BYTES_Q4 = 576
APPEND_BYTES = 2 * H * 256 * 2 + CELL_BYTES      # bf16 K+V in, 816 B out
METRIC = "k8v4 decode-attn GB/s (% HBM peak) and cells/s @238K ctx; append cells/s"
WORKLOAD = "decode_237568_cells_2kv_16q_gqa8_P64_bf16"
SWEEP = (14848, 118784, 237568, 262144)       # the long-context sweep (page-aligned 15K/119K/238K/262,144)
L2_BYTES = 129 << 20


def config_dict(world: int) -> dict:
    """The workload both arms report (the GPU line and the reference arm)."""
    return {"workload": WORKLOAD, "cells": N_CELLS, "page_size": P, "n_kv_heads": H, "n_q_heads": HQ,
            "step": "append 1 token + split-K decode attention (partials + combine/inverse WHT), one call "
                    "(attn_k8v4_decode_step: the CTA holding the newest cell writes it first)",
            "l2": "inputs larger than L2: two 193.9 MB cache replicas alternate (387.7 MB > 135.5 MB L2)",
            "parallelism": f"replicas x{world}"}


def prefix_workload(big, n_cells: int):
    """The first n_cells of a long-context workload with the page table that
    synth.config3(n_cells) draws (the K/V/q streams are counter-based, so the
    prefix holds config3(n_cells)'s values)."""
    import synth
    n_pages = (n_cells + P - 1) // P
    pt = synth.page_table_shuffled(big.seed, synth.stream_id(synth.T_PT, 0), n_pages, n_pages)
    return synth.Workload(name=f"decode_{n_cells}", seed=big.seed, n_seqs=1, page_size=P, n_kv=H,
                          n_pages=n_pages, max_pages=n_pages, page_table=pt.reshape(1, -1),
                          seq_lens=np.array([n_cells], np.int32), pos=np.array([0], np.int64),
                          k=big.k, v=big.v, q=big.q, dtype=big.dtype)


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_timing(total_ms: float, steps: int, cells_per_rank: int, device=None):
    """Whole-job timing of a replicated step: the slowest rank's wall time over
    `steps` steps sets the step time (an all-reduce MAX when a process group is
    up), and the rate counts the cells of every rank.  Returns (ms per step,
    cells/s of the job, world size)."""
    import torch
    world = 1
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        world = torch.distributed.get_world_size()
        if world > 1:
            t = torch.tensor([total_ms], dtype=torch.float64, device=device)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            total_ms = float(t.item())
    ms_step = total_ms / steps
    return ms_step, world * cells_per_rank / (ms_step / 1e3), world


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when any
    source file the kernel is built from changed since the counters were taken
    (the summary lists the files and the first 16 hex digits of the SHA-256 of
    their concatenation)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_dram.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    h = hashlib.sha256()
    for name in fields.get("source", "").split():
        src = os.path.join(ROOT, "quantized_paged_kv_q8_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    if not fields.get("source") or h.hexdigest()[:16] != fields.get("source_sha256_16"):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_decode_rate(w, n_cells: int, repeats: int, n_threads: int, min_seconds: float = 0.0):
    """Time the CPU oracle's decode attention (16 rows) over the first n_cells of
    the workload, its cache built by its own append (untimed): at least `repeats`
    steps and at least `min_seconds` of them.  Returns GB/s over 816 B/cell,
    seconds per step, steps timed."""
    import oracle
    n_pages = (n_cells + P - 1) // P
    pt = np.arange(n_pages, dtype=np.int32)[None]
    cache = oracle.Cache(n_pages, P, H)
    cache.append(pt, np.array([0]), w.k.f32[None, :n_cells], w.v.f32[None, :n_cells], n_threads=n_threads)
    rs, rh, rv = oracle.decode_rows(1, HQ, [n_cells])
    q = w.q.f32.reshape(-1, 256)
    t0 = time.perf_counter()
    done = 0
    while done < repeats or time.perf_counter() - t0 < min_seconds:
        cache.attention(pt, rs, rh, rv, q, n_threads=n_threads)
        done += 1
    dt = (time.perf_counter() - t0) / done
    return CELL_BYTES * n_cells / dt / 1e9, dt, done


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import synth
    threads = os.cpu_count() or 1
    w = synth.config3(N_CELLS)
    # size each step so that warmup + steps end within about two minutes
    _, t_small, _ = oracle_decode_rate(w, 4096, 1, threads)
    per_cell = t_small / 4096
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_cells = int(min(N_CELLS, max(1024, budget / per_cell)) // P * P)
    import oracle
    n_pages = n_cells // P
    pt = np.arange(n_pages, dtype=np.int32)[None]
    cache = oracle.Cache(n_pages, P, H)
    cache.append(pt, np.array([0]), w.k.f32[None, :n_cells], w.v.f32[None, :n_cells], n_threads=threads)
    rs, rh, rv = oracle.decode_rows(1, HQ, [n_cells])
    q = w.q.f32.reshape(-1, 256)
    for _ in range(args.warmup):
        cache.attention(pt, rs, rh, rv, q, n_threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cache.attention(pt, rs, rh, rv, q, n_threads=threads)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = CELL_BYTES * n_cells / dt / 1e9
    sample = (f"per step: CPU oracle fp64 decode attention, 16 query rows over the first {n_cells} of the "
              f"{N_CELLS}-cell workload (its cache built by its own append, untimed); GB/s over 816 B/cell")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(ws), "sample_cells": n_cells,
            "cells_per_s": n_cells / dt,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_oracle_table(args):
    """The CPU oracle per configuration, on 1 thread and on every host thread
    (the baseline plan's table): decode GB/s over 816 B/cell, verify GB/s over
    the cells read, prefill TFLOP/s over the visible (query, cell) pairs x 16
    heads x 1,024 flop, append cells/s.  Large cases are timed on a stated
    sample and scaled linearly (attention cost is linear in rows)."""
    import oracle
    import synth
    nt = os.cpu_count() or 1

    def timed(fn, min_s=0.5):
        t0 = time.perf_counter()
        n = 0
        while True:
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= min_s:
                return dt / n

    def decode_case(w, n_cells, label):
        n_pages = (n_cells + P - 1) // P
        pt = np.arange(n_pages, dtype=np.int32)[None]
        cache = oracle.Cache(n_pages, P, H)
        cache.append(pt, np.array([0]), w.k.f32[None, :n_cells], w.v.f32[None, :n_cells], n_threads=nt)
        rs, rh, rv = oracle.decode_rows(1, HQ, [n_cells])
        q = w.q.f32.reshape(-1, 256)
        res = {"config": label, "cells": n_cells, "unit": "GB/s"}
        for th in (1, nt):
            dt = timed(lambda: cache.attention(pt, rs, rh, rv, q, n_threads=th))
            res[f"t{th}"] = CELL_BYTES * n_cells / dt / 1e9
        print(json.dumps(res), flush=True)

    # config 1: the tiny fp32 round trip (append + one decode query), cells/s
    w1 = synth.config1()
    for th in (1, nt):
        def rt():
            c = oracle.Cache(w1.n_pages, w1.page_size, w1.n_kv)
            c.append(w1.page_table, w1.pos, w1.k.f32[None], w1.v.f32[None], n_threads=th)
            rs, rh, rv = oracle.decode_rows(1, HQ, w1.seq_lens)
            c.attention(w1.page_table, rs, rh, rv, w1.q.f32.reshape(-1, 256), n_threads=th)
        dt = timed(rt)
        print(json.dumps({"config": "1 tiny round trip", "cells": 1024, "unit": "cells/s", f"t{th}": 1024 / dt}),
              flush=True)
    decode_case(synth.config2(), 32768, "2 decode 32,768")
    big = synth.config3(SWEEP[-1])
    for n in SWEEP:
        decode_case(big, n, f"3 decode {n}")
    # config 4: verify, 8 sequences x 5 queries; 1 thread on sequence 0 (scaled by
    # the cells of all 8), every thread on all 8
    w4 = synth.config4()
    cache4 = oracle.Cache(w4.n_pages, w4.page_size, w4.n_kv)
    for b in range(w4.n_seqs):
        cache4.append(w4.page_table[b:b + 1], np.array([0]), w4.k[b].f32[None], w4.v[b].f32[None], n_threads=nt)
    cells = int(w4.seq_lens.sum())
    res = {"config": "4 verify 8 x 5", "cells": cells, "unit": "GB/s"}
    for th, seqs in ((1, [0]), (nt, list(range(w4.n_seqs)))):
        steps = w4.steps[seqs]
        rs, rh, rv = oracle.multi_query_rows(steps, HQ)
        rs = np.asarray(seqs, np.int32)[rs]
        q = np.concatenate([w4.q[b].f32.reshape(-1, 256) for b in seqs])
        dt = timed(lambda: cache4.attention(w4.page_table, rs, rh, rv, q, n_threads=th))
        done = int(w4.seq_lens[seqs].sum())
        res[f"t{th}"] = CELL_BYTES * cells / (dt * cells / done) / 1e9
    res["sample_t1"] = "sequence 0 only, scaled by cells"
    print(json.dumps(res), flush=True)
    del cache4
    # config 5: prefill of the 8,192-token chunk at 229,376 and its append; a
    # strided query subset, scaled by the visible pairs of the whole chunk
    w5 = synth.config5()
    cache5 = oracle.Cache(w5.n_pages, w5.page_size, w5.n_kv)
    hk, hv = synth.prefill_kv(w5, 0, w5.history)
    cache5.append(w5.page_table, np.array([0]), hk.f32[None], hv.f32[None], n_threads=nt)
    ck, cv = synth.prefill_kv(w5, w5.history, w5.chunk)
    res = {"config": "5 chunk append 8,192", "cells": w5.chunk, "unit": "cells/s"}
    for th in (1, nt):
        dt = timed(lambda: cache5.append(w5.page_table, np.array([w5.history]), ck.f32[None], cv.f32[None],
                                         n_threads=th), min_s=1.0)
        res[f"t{th}"] = w5.chunk / dt
    print(json.dumps(res), flush=True)
    qall = synth.prefill_q(w5).f32.reshape(w5.chunk, HQ, 256)
    pairs = sum(w5.history + t + 1 for t in range(w5.chunk))
    res = {"config": "5 prefill 8,192 @ 229,376", "unit": "TFLOP/s"}
    for th, stride in ((1, 1024), (nt, 64)):
        toks = np.arange(0, w5.chunk, stride)
        rs = np.zeros(len(toks) * HQ, np.int32)
        rh = np.tile(np.arange(HQ, dtype=np.int32), len(toks))
        rv = np.repeat((w5.history + toks + 1).astype(np.int32), HQ)
        q = qall[toks].reshape(-1, 256)
        dt = timed(lambda: cache5.attention(w5.page_table, rs, rh, rv, q, n_threads=th), min_s=0.1)
        sub_pairs = int(np.sum(w5.history + toks + 1))
        res[f"t{th}"] = pairs * HQ * 1024 / (dt * pairs / sub_pairs) / 1e12
        res[f"sample_t{th}"] = f"every {stride}th query token ({len(toks)} tokens x 16 heads), scaled by visible pairs"
    print(json.dumps(res), flush=True)
    print(json.dumps({"host_threads": nt}), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def graph_ms(call, n_calls: int, reps: int) -> float:
    """Per-call device time of `call(i)` for i < n_calls, captured once into a
    CUDA graph and replayed `reps` times between two events (no host launch cost
    inside the timed region)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(min(n_calls, 4)):
            call(i)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for i in range(n_calls):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * n_calls)
    del g
    return ms


def measure_sweep(dev, big, kd_big, vd_big, reps: int = 200):
    """The long-context sweep: decode attention over 14,848, 118,784, 237,568 and
    262,144 cells, the k8v4 format (816 B/cell) beside the INT8/INT8 comparison
    format (1,056 B/cell), each timed over `reps` calls that cycle through enough
    cache replicas to hold four times L2 (every call streams its cache from HBM):
    once as eager calls from Python (host launch cost included) and once as a
    CUDA graph of the same calls replayed (device time of the launches alone)."""
    import math
    import torch
    import quantized_paged_kv_q8_gb300 as k8
    hbm = peaks()[0]
    q = torch.from_numpy(big.q.dev.view(np.int16)).view(torch.bfloat16).reshape(1, HQ, 256).to(dev)
    zero = torch.zeros(1, dtype=torch.int64, device=dev)
    out = torch.empty(1, HQ, 256, dtype=torch.float32, device=dev)
    rows = []
    for n in SWEEP:
        w = prefix_workload(big, n)
        pt = torch.from_numpy(w.page_table).to(dev)
        lens = torch.full((1,), n, dtype=torch.int32, device=dev)
        row = {"cells": n}
        for name, fmt, cb in (("k8v4", k8.FORMAT_K8V4, CELL_BYTES), ("int8", k8.FORMAT_INT8, CELL_BYTES_INT8)):
            n_rep = max(2, math.ceil(4 * L2_BYTES / (n * cb)))
            caches = [k8.PagedCache(w.n_pages, P, H, fmt=fmt, device=dev) for _ in range(n_rep)]
            for c in caches:
                k8.kv_append_k8v4(c, pt, zero, kd_big[:, :n], vd_big[:, :n])
            ws = k8.workspace(caches[0], 1, 1, n, device=dev)
            for i in range(2 * n_rep):
                k8.attn_k8v4_decode(caches[i % n_rep], q, pt, lens, n, out, ws)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(reps):
                k8.attn_k8v4_decode(caches[i % n_rep], q, pt, lens, n, out, ws)
            e1.record()
            torch.cuda.synchronize()
            assert k8.k8v4_last_device_status() == 0
            ms = e0.elapsed_time(e1) / reps
            gbs = cb * n / (ms / 1e3) / 1e9
            gms = graph_ms(lambda i: k8.attn_k8v4_decode(caches[i % n_rep], q, pt, lens, n, out, ws),
                           n_calls=n_rep * max(1, 64 // n_rep), reps=max(2, reps // 64))
            assert k8.k8v4_last_device_status() == 0
            ggbs = cb * n / (gms / 1e3) / 1e9
            row[name] = {"ms_per_step": ms, "gbs": gbs, "frac_hbm": gbs / hbm, "cells_per_s": n / (ms / 1e3),
                         "graph": {"ms_per_step": gms, "gbs": ggbs, "frac_hbm": ggbs / hbm},
                         "replicas": n_rep, "bytes_per_cell": cb}
            del caches, ws
            torch.cuda.empty_cache()
        row["k8v4_speedup"] = row["int8"]["ms_per_step"] / row["k8v4"]["ms_per_step"]
        row["k8v4_speedup_graph"] = row["int8"]["graph"]["ms_per_step"] / row["k8v4"]["graph"]["ms_per_step"]
        rows.append(row)
    return rows


def measure_config2(dev, steps: int = 1000):
    """Config 2: one 32,768-cell sequence (P = 64, shuffled pages, bf16), 1,000
    decode steps (each appends the newest token and decodes, one
    attn_k8v4_decode_step call), cycling through 21 cache replicas (561 MB, four
    times L2).  GB/s over 816 B/cell, as eager calls and as a replayed CUDA graph
    of 1,000 steps."""
    import math
    import torch
    import quantized_paged_kv_q8_gb300 as k8
    import synth
    w = synth.config2()
    n = 32768
    pt = torch.from_numpy(w.page_table).to(dev)
    kd = torch.from_numpy(w.k.dev.view(np.int16)).view(torch.bfloat16).reshape(1, n, H, 256).to(dev)
    vd = torch.from_numpy(w.v.dev.view(np.int16)).view(torch.bfloat16).reshape(1, n, H, 256).to(dev)
    zero = torch.zeros(1, dtype=torch.int64, device=dev)
    n_rep = max(2, math.ceil(4 * L2_BYTES / (n * CELL_BYTES)))
    caches = [k8.PagedCache(w.n_pages, P, H, device=dev) for _ in range(n_rep)]
    for c in caches:
        k8.kv_append_k8v4(c, pt, zero, kd, vd)
    q = torch.from_numpy(w.q.dev.view(np.int16)).view(torch.bfloat16).reshape(1, HQ, 256).to(dev)
    k_new, v_new = kd[0, n - 1:].contiguous(), vd[0, n - 1:].contiguous()
    lens = torch.full((1,), n, dtype=torch.int32, device=dev)
    out = torch.empty(1, HQ, 256, dtype=torch.float32, device=dev)
    ws = k8.workspace(caches[0], 1, 1, n, device=dev)
    for i in range(20):
        k8.attn_k8v4_decode_step(caches[i % n_rep], q, k_new, v_new, pt, lens, n, out, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        k8.attn_k8v4_decode_step(caches[i % n_rep], q, k_new, v_new, pt, lens, n, out, ws)
    e1.record()
    torch.cuda.synchronize()
    assert k8.k8v4_last_device_status() == 0
    ms = e0.elapsed_time(e1) / steps
    gbs = CELL_BYTES * n / (ms / 1e3) / 1e9
    gms = graph_ms(lambda i: k8.attn_k8v4_decode_step(caches[i % n_rep], q, k_new, v_new, pt, lens, n, out, ws),
                   n_calls=steps, reps=3)
    assert k8.k8v4_last_device_status() == 0
    ggbs = CELL_BYTES * n / (gms / 1e3) / 1e9
    return {"workload": "decode_step_32768_cells_x1000", "steps": steps, "replicas": n_rep, "ms_per_step": ms,
            "gbs": gbs, "frac_hbm": gbs / peaks()[0], "cells_per_s": n / (ms / 1e3),
            "graph": {"ms_per_step": gms, "gbs": ggbs, "frac_hbm": ggbs / peaks()[0], "cells_per_s": n / (gms / 1e3)}}


def measure_verify(args, dev, reps: int = 20):
    """Config 4: 8 sequences, lengths U[16,384, 65,536], 5 queries each with steps
    len-4+i, pages interleaved in one pool.  GB/s over 816 B/cell of the cells
    read (each sequence's longest step)."""
    import torch
    import quantized_paged_kv_q8_gb300 as k8
    import synth
    w = synth.config4()
    cache = k8.PagedCache(w.n_pages, w.page_size, w.n_kv, device=dev)
    pt = torch.from_numpy(w.page_table).to(dev)
    for b in range(w.n_seqs):
        n = int(w.seq_lens[b])
        kd = torch.from_numpy(w.k[b].dev.view(np.int16)).view(torch.bfloat16).reshape(1, n, H, 256).to(dev)
        vd = torch.from_numpy(w.v[b].dev.view(np.int16)).view(torch.bfloat16).reshape(1, n, H, 256).to(dev)
        k8.kv_append_k8v4(cache, pt[b:b + 1], torch.zeros(1, dtype=torch.int64, device=dev), kd, vd)
    q = torch.stack([torch.from_numpy(w.q[b].dev.view(np.int16)).view(torch.bfloat16) for b in range(w.n_seqs)]).to(dev)
    steps = torch.from_numpy(w.steps).to(dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    max_len = int(w.seq_lens.max())
    ws = k8.workspace(cache, w.n_seqs, w.n_q, max_len, device=dev)
    for _ in range(3):
        k8.attn_k8v4_verify(cache, q, pt, steps, max_len, out, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        k8.attn_k8v4_verify(cache, q, pt, steps, max_len, out, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    assert k8.k8v4_last_device_status() == 0
    cells = int(w.seq_lens.sum())
    return {"workload": "verify_8seq_x5q_U16K-64K", "cells": cells, "ms_per_call": ms,
            "gbs": CELL_BYTES * cells / (ms / 1e3) / 1e9, "cells_per_s": cells / (ms / 1e3)}


def measure_batched_step(args, dev, n_seqs: int = 32, n_cells: int = 8192, reps: int = 200):
    """The engine's batched decode shape: n_seqs sequences of n_cells cells each,
    pages interleaved in one pool; one attn_k8v4_decode_step call appends every
    sequence's newest token and decodes all of them.  Two cache replicas
    alternate (2 x 214 MB > L2).  GB/s over 816 B/cell of the cells read."""
    import torch
    import quantized_paged_kv_q8_gb300 as k8
    import synth
    seed = synth.config_seed(3) + 1000
    lens = np.full(n_seqs, n_cells, np.int32)
    pt_np, n_pages = synth.interleaved_pool(seed, lens, P)
    pt = torch.from_numpy(pt_np).to(dev)
    caches = [k8.PagedCache(n_pages, P, H, device=dev) for _ in range(2)]
    for b in range(n_seqs):
        k = synth.kv_values(seed, synth.T_K, b, n_cells, H, 3, "bf16")
        v = synth.kv_values(seed, synth.T_V, b, n_cells, H, 3, "bf16")
        kd = torch.from_numpy(k.dev.view(np.int16)).view(torch.bfloat16).reshape(1, n_cells, H, 256).to(dev)
        vd = torch.from_numpy(v.dev.view(np.int16)).view(torch.bfloat16).reshape(1, n_cells, H, 256).to(dev)
        for c in caches:
            k8.kv_append_k8v4(c, pt[b:b + 1], torch.zeros(1, dtype=torch.int64, device=dev), kd, vd)
    qv = synth.q_values(seed, 0, n_seqs, H, "bf16")
    q = torch.from_numpy(qv.dev.view(np.int16)).view(torch.bfloat16).reshape(n_seqs, HQ, 256).to(dev)
    knew = torch.randn(n_seqs, H, 256, generator=torch.Generator().manual_seed(seed & 0xffff)).to(torch.bfloat16).to(dev)
    vnew = torch.randn(n_seqs, H, 256, generator=torch.Generator().manual_seed((seed >> 16) & 0xffff)).to(torch.bfloat16).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    out = torch.empty(n_seqs, HQ, 256, dtype=torch.float32, device=dev)
    ws = k8.workspace(caches[0], n_seqs, 1, n_cells, device=dev)
    for i in range(10):
        k8.attn_k8v4_decode_step(caches[i & 1], q, knew, vnew, pt, lens_d, n_cells, out, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        k8.attn_k8v4_decode_step(caches[i & 1], q, knew, vnew, pt, lens_d, n_cells, out, ws)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    assert k8.k8v4_last_device_status() == 0
    cells = n_seqs * n_cells
    return {"workload": f"decode_step_{n_seqs}seq_x_{n_cells}_cells", "cells": cells, "ms_per_step": ms,
            "gbs": CELL_BYTES * cells / (ms / 1e3) / 1e9, "cells_per_s": cells / (ms / 1e3)}


def measure_stream(args, dev, resident_cells: int = 32768, reps: int = 8):
    """KV streaming at the 238K workload: the page-locked host mirror holds all
    3,712 pages, the device holds a resident window of the newest
    `resident_cells` cells (512 pages, the streaming PR's --kv-resident 32768)
    plus staging slots.  One streamed decode = kv_stream_resolve (the lookups and
    the copy of every non-resident page from the mirror over NVLink-C2C) +
    attn_k8v4_decode over the device table.  Also timed: the mirrored append of
    the whole cache (both copies written), and a plain pinned host -> device
    cudaMemcpyAsync of 256 MiB, the copy rate the page mover is compared with.
    Stream timings are the median of five event-timed batches."""
    import torch
    import quantized_paged_kv_q8_gb300 as k8
    import synth
    w = synth.config3(N_CELLS)
    need = N_CELLS // P
    n_res = resident_cells // P
    host = k8.PagedCache(w.n_pages, P, H, device="pinned")
    devc = k8.PagedCache(n_res + need, P, H, device=dev)
    slot_of_page = np.full(w.n_pages, -1, np.int32)
    slot_of_page[w.page_table[0, need - n_res:need]] = np.arange(n_res, dtype=np.int32)
    sop = torch.from_numpy(slot_of_page).to(dev)
    pt = torch.from_numpy(w.page_table).to(dev)
    kd = torch.from_numpy(w.k.dev.view(np.int16)).view(torch.bfloat16).reshape(1, N_CELLS, H, 256).to(dev)
    vd = torch.from_numpy(w.v.dev.view(np.int16)).view(torch.bfloat16).reshape(1, N_CELLS, H, 256).to(dev)
    zero = torch.zeros(1, dtype=torch.int64, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    k8.kv_append_k8v4_mirrored(host, devc, sop, pt, zero, kd, vd)
    torch.cuda.synchronize()
    ev[0].record()
    for _ in range(3):
        k8.kv_append_k8v4_mirrored(host, devc, sop, pt, zero, kd, vd)
    ev[1].record()
    torch.cuda.synchronize()
    append_ms = ev[0].elapsed_time(ev[1]) / 3
    del kd, vd
    q = torch.from_numpy(w.q.dev.view(np.int16)).view(torch.bfloat16).reshape(1, HQ, 256).to(dev)
    lens = torch.full((1,), N_CELLS, dtype=torch.int32, device=dev)
    dev_pt = torch.empty_like(pt)
    sws = torch.empty(k8.kv_stream_workspace_bytes(1, pt.shape[1]), dtype=torch.uint8, device=dev)
    out = torch.empty(1, HQ, 256, dtype=torch.float32, device=dev)
    wsp = k8.workspace(devc, 1, 1, N_CELLS, device=dev)

    def step():
        k8.kv_stream_resolve(host, devc, sop, n_res, pt, lens, N_CELLS, dev_pt, sws)
        k8.attn_k8v4_decode(devc, q, dev_pt, lens, N_CELLS, out, wsp)

    for _ in range(3):
        step()
    torch.cuda.synchronize()

    def median_ms(fn, batches: int = 5):
        # the host link is shared with other tenants of the machine: time several
        # event-bracketed batches and report the median per-call time
        per = []
        for _ in range(batches):
            ev[2].record()
            for _ in range(reps):
                fn()
            ev[3].record()
            torch.cuda.synchronize()
            per.append(ev[2].elapsed_time(ev[3]) / reps)
        return statistics.median(per)

    step_ms = median_ms(step)
    resolve_ms = median_ms(lambda: k8.kv_stream_resolve(host, devc, sop, n_res, pt, lens, N_CELLS, dev_pt, sws))
    assert k8.k8v4_last_device_status() == 0
    moved = (need - n_res) * devc.page_bytes
    # the plain copy the mover is compared with: 256 MiB pinned -> device
    src = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    copy_ms = median_ms(lambda: dst.copy_(src, non_blocking=True), batches=3)
    h2d_gbs = (256 << 20) / (copy_ms / 1e3) / 1e9
    return {"workload": f"stream_decode_{N_CELLS}_cells_{resident_cells}_resident",
            "resident_pages": n_res, "streamed_pages": need - n_res, "page_bytes": devc.page_bytes,
            "ms_per_step": step_ms, "cells_per_s": N_CELLS / (step_ms / 1e3),
            "resolve_copy_ms": resolve_ms, "copy_gbs": moved / (resolve_ms / 1e3) / 1e9,
            "h2d_memcpy_gbs": h2d_gbs, "copy_frac_of_memcpy": moved / (resolve_ms / 1e3) / 1e9 / h2d_gbs,
            "mirrored_append_ms": append_ms, "mirrored_append_cells_per_s": N_CELLS / (append_ms / 1e3)}


def measure_prefill(args, dev, chunk: int, reps: int = 3):
    """Config 5: 229,376-cell history, then an append of `chunk` tokens at offset
    229,376 (timed: chunk append cells/s) and causal prefill of the chunk (timed:
    TFLOP/s over the visible (query, cell) pairs x 16 heads x 1,024 flop)."""
    import torch
    import quantized_paged_kv_q8_gb300 as k8
    import synth
    w = synth.config5(chunk=chunk)
    cache = k8.PagedCache(w.n_pages, w.page_size, w.n_kv, device=dev)
    pt = torch.from_numpy(w.page_table).to(dev)

    def kv(lo, n):
        k, v = synth.prefill_kv(w, lo, n)
        return (torch.from_numpy(k.dev.view(np.int16)).view(torch.bfloat16).reshape(1, n, H, 256).to(dev),
                torch.from_numpy(v.dev.view(np.int16)).view(torch.bfloat16).reshape(1, n, H, 256).to(dev))
    hk, hv = kv(0, w.history)
    k8.kv_append_k8v4(cache, pt, torch.zeros(1, dtype=torch.int64, device=dev), hk, hv)
    del hk, hv
    ck, cv = kv(w.history, w.chunk)
    off = torch.full((1,), w.history, dtype=torch.int64, device=dev)
    k8.kv_append_k8v4(cache, pt, off, ck, cv)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(10):
        k8.kv_append_k8v4(cache, pt, off, ck, cv)
    a1.record()
    torch.cuda.synchronize()
    app_ms = a0.elapsed_time(a1) / 10
    q = synth.prefill_q(w)
    qd = torch.from_numpy(q.dev.view(np.int16)).view(torch.bfloat16).reshape(w.chunk, HQ, 256).to(dev)
    out = torch.empty(w.chunk, HQ, 256, dtype=torch.float32, device=dev)
    k8.attn_k8v4_prefill(cache, qd, pt[0], w.total, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        k8.attn_k8v4_prefill(cache, qd, pt[0], w.total, out)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    assert k8.k8v4_last_device_status() == 0
    pairs = sum(w.history + t + 1 for t in range(w.chunk))
    flop = pairs * HQ * 1024
    return {"workload": f"prefill_{w.chunk}_tokens_at_{w.history}", "ms_per_call": ms, "tflop": flop / 1e12,
            "tflops": flop / (ms / 1e3) / 1e12,
            "chunk_append": {"cells": w.chunk, "ms": app_ms, "cells_per_s": w.chunk / (app_ms / 1e3),
                             "gbs": APPEND_BYTES * w.chunk / (app_ms / 1e3) / 1e9}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="k8v4", choices=["k8v4", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the CPU oracle per configuration on 1 and all host threads, then exit")
    ap.add_argument("--profile", default=None, choices=["decode", "prefill", "verify", "batched", "stream"],
                    help="lean single-kernel run for ncu (no replicas, INT8 arm, e2e or CPU baseline)")
    ap.add_argument("--chunk", type=int, default=8192, help="prefill chunk length (tokens)")
    ap.add_argument("--format", default="k8v4", choices=["k8v4", "q4", "int8"],
                    help="cache format of the --profile decode run")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.oracle_table:
        run_oracle_table(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import quantized_paged_kv_q8_gb300 as k8
    import synth
    from quantized_paged_kv_q8_gb300 import buildlib
    buildlib.build()
    assert k8.k8v4_device_check() == 0, "libk8v4 needs an sm_103 device"

    if args.profile in ("prefill", "verify", "batched", "stream"):
        res = (measure_prefill(args, dev, args.chunk) if args.profile == "prefill"
               else measure_verify(args, dev) if args.profile == "verify"
               else measure_stream(args, dev) if args.profile == "stream" else measure_batched_step(args, dev))
        if rank == 0:
            print(json.dumps({"profile": args.profile, **res}), flush=True)
        return

    # one long-context workload: its 237,568-cell prefix is the headline, its
    # prefixes the sweep (counter-based streams: the prefix is config3(n))
    big = synth.config3(SWEEP[-1]) if not args.profile else synth.config3(N_CELLS)
    w = prefix_workload(big, N_CELLS)
    n_pages = w.n_pages
    pt = torch.from_numpy(w.page_table).to(dev)
    kd_big = torch.from_numpy(big.k.dev.view(np.int16)).view(torch.bfloat16).reshape(1, -1, H, 256).to(dev)
    vd_big = torch.from_numpy(big.v.dev.view(np.int16)).view(torch.bfloat16).reshape(1, -1, H, 256).to(dev)
    kd, vd = kd_big[:, :N_CELLS], vd_big[:, :N_CELLS]
    zero = torch.zeros(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()

    # ---- bulk append (cache build) timing: append cells/s
    n_rep = 1 if args.profile else 2
    fmt = {"k8v4": k8.FORMAT_K8V4, "q4": k8.FORMAT_Q4, "int8": k8.FORMAT_INT8}[args.format if args.profile else "k8v4"]
    caches = [k8.PagedCache(n_pages, P, H, fmt=fmt, device=dev) for _ in range(n_rep)]
    for c in caches:
        k8.kv_append_k8v4(c, pt, zero, kd, vd)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_app = 5
    a0.record()
    for i in range(n_app):
        k8.kv_append_k8v4(caches[i % n_rep], pt, zero, kd, vd)
    a1.record()
    torch.cuda.synchronize()
    append_s = a0.elapsed_time(a1) / 1e3 / n_app
    assert k8.k8v4_last_device_status() == 0

    # ---- decode step inputs
    q = torch.from_numpy(w.q.dev.view(np.int16)).view(torch.bfloat16).reshape(1, HQ, 256).to(dev)
    k_new = kd[0, N_CELLS - 1:].contiguous()          # [1 sequence][H][256]: the newest token
    v_new = vd[0, N_CELLS - 1:].contiguous()
    lens = torch.full((1,), N_CELLS, dtype=torch.int32, device=dev)
    out = torch.empty(1, HQ, 256, dtype=torch.float32, device=dev)
    wsp = k8.workspace(caches[0], 1, 1, N_CELLS, device=dev)

    if args.profile:
        del kd, vd, kd_big, vd_big
        torch.cuda.empty_cache()

    def step(i):
        # one call: the CTA whose cells hold the newest one appends it, then all attend
        k8.attn_k8v4_decode_step(caches[i % n_rep], q, k_new, v_new, pt, lens, N_CELLS, out, wsp)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        # the timed steps: nothing between the launches, so the decode launch
        # overlaps the tail of the append (programmatic dependent launch)
        t0.record()
        for i in range(K):
            step(i)
        t1.record()
        torch.cuda.synchronize()
        # the roofline's decode-only duration: K decode calls back to back over
        # the alternating replicas (each call streams its cache from HBM),
        # bracketed by two events on the launching stream
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record()
        for i in range(K):
            k8.attn_k8v4_decode(caches[i % n_rep], q, pt, lens, N_CELLS, out, wsp)
        d1.record()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t0.elapsed_time(t1)
    dec_ms = d0.elapsed_time(d1) / K
    assert k8.k8v4_last_device_status() == 0
    ms_step, cells_per_s, _ = job_timing(total_ms, K, N_CELLS, dev)
    value = cells_per_s * CELL_BYTES / 1e9

    if args.profile:
        if rank == 0:
            cb = caches[0].bytes_per_cell
            print(json.dumps({"profile": True, "format": args.format, "ms_per_step": ms_step, "decode_ms": dec_ms,
                              "gbs": cb * N_CELLS / (dec_ms / 1e3) / 1e9, "append_ms": append_s * 1e3,
                              "append_frac": APPEND_BYTES * N_CELLS / append_s / 1e9 / peaks()[0]}), flush=True)
        return

    # ---- comparison formats on the same workload: INT8/INT8 (1,056 B/cell) and
    # q4_0 K+V (576 B/cell), decode calls over two alternating replicas
    def format_arm(fmt, cell_bytes):
        cs = [k8.PagedCache(n_pages, P, H, fmt=fmt, device=dev) for _ in range(2)]
        for c in cs:
            k8.kv_append_k8v4(c, pt, zero, kd, vd)
        wsf = k8.workspace(cs[0], 1, 1, N_CELLS, device=dev)
        for i in range(20):
            k8.attn_k8v4_decode(cs[i & 1], q, pt, lens, N_CELLS, out, wsf)
        Kf = max(20, K // 5)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record()
        for i in range(Kf):
            k8.attn_k8v4_decode(cs[i & 1], q, pt, lens, N_CELLS, out, wsf)
        b1.record()
        torch.cuda.synchronize()
        assert k8.k8v4_last_device_status() == 0
        ms = b0.elapsed_time(b1) / Kf
        del cs, wsf
        torch.cuda.empty_cache()
        return {"gbs": cell_bytes * N_CELLS / (ms / 1e3) / 1e9, "ms_per_step": ms,
                "cells_per_s": N_CELLS / (ms / 1e3), "bytes_per_cell": cell_bytes, "k8v4_speedup": ms / dec_ms}

    int8_arm = format_arm(k8.FORMAT_INT8, CELL_BYTES_INT8)
    q4_arm = format_arm(k8.FORMAT_Q4, CELL_BYTES_Q4)

    # ---- end to end through the C ABI with host buffers: the step's inputs
    # live in one pinned buffer (q | k_new | v_new, bf16; every part starts on a
    # 16-byte boundary) and its output in another.  `e2e`: the call is handed
    # the host buffers and its kernels read the inputs and write the output
    # across the host link (no copy launches); `e2e_copies`: one host -> device
    # copy of the inputs and one device -> host copy of the output per step
    # around the call on device buffers.
    nq, nk = q.numel(), k_new.numel()
    in_h = torch.cat([q.reshape(-1), k_new.reshape(-1), v_new.reshape(-1)]).cpu().pin_memory()
    in_s = torch.empty(in_h.shape, dtype=in_h.dtype, device=dev)
    q_s = in_s[:nq].view(q.shape)
    kn_s = in_s[nq:nq + nk].view(k_new.shape)
    vn_s = in_s[nq + nk:].view(v_new.shape)
    q_h = in_h[:nq].view(q.shape)
    kn_h = in_h[nq:nq + nk].view(k_new.shape)
    vn_h = in_h[nq + nk:].view(v_new.shape)
    out_h = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    Ke = max(20, min(K, 2000))

    def e2e_host_step(i):
        k8.attn_k8v4_decode_step(caches[i % n_rep], q_h, kn_h, vn_h, pt, lens, N_CELLS, out_h, wsp)

    def e2e_copy_step(i):
        in_s.copy_(in_h, non_blocking=True)
        k8.attn_k8v4_decode_step(caches[i % n_rep], q_s, kn_s, vn_s, pt, lens, N_CELLS, out, wsp)
        out_h.copy_(out, non_blocking=True)

    def time_e2e(step):
        for i in range(10):
            step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(Ke):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / Ke

    e2e_ms = time_e2e(e2e_host_step)
    e2e_copies_ms = time_e2e(e2e_copy_step)
    assert k8.k8v4_last_device_status() == 0
    h2d = in_h.numel() * in_h.element_size()
    d2h = out.numel() * 4

    del caches, kd, vd
    torch.cuda.empty_cache()
    sweep = measure_sweep(dev, big, kd_big, vd_big)
    del kd_big, vd_big
    torch.cuda.empty_cache()
    config2 = measure_config2(dev)
    verify = measure_verify(args, dev)
    batched = measure_batched_step(args, dev)
    stream = measure_stream(args, dev)
    prefill = measure_prefill(args, dev, 8192)

    hbm, bf16, bf16_sus, peak_kind = peaks()
    dec_bytes = CELL_BYTES * N_CELLS
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    traffic = traffic_record("decode_kernel_237568")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "storage": "int8 K + q4_0 V, 816 B/cell", "data": "synthetic",
        "config": config_dict(world),
        "cells_per_s": cells_per_s,
        "hbm_frac_of_step": value / hbm,
        "roofline": {"bound": "hbm", "kernel": "attn_k8v4_decode (TMA worker split-K kernel + combine)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "algorithmic_bytes_per_launch": dec_bytes,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)", "ms_per_launch": dec_ms},
        "append": {"cells_per_s": N_CELLS / append_s, "gbs": APPEND_BYTES * N_CELLS / append_s / 1e9,
                   "frac": APPEND_BYTES * N_CELLS / append_s / 1e9 / hbm, "bytes_per_cell": APPEND_BYTES,
                   "ms_per_launch": append_s * 1e3, "cells_per_launch": N_CELLS},
        "int8_arm": {**int8_arm, "frac_hbm": int8_arm["gbs"] / hbm},
        "q4_arm": {**q4_arm, "frac_hbm": q4_arm["gbs"] / hbm},
        "e2e": {"value": dec_bytes / (e2e_ms / 1e3) / 1e9 * world, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "host buffers handed to the call: its kernels read the inputs and write the output "
                       "across the host link"},
        "e2e_copies": {"value": dec_bytes / (e2e_copies_ms / 1e3) / 1e9 * world, "unit": "GB/s",
                       "ms_per_step": e2e_copies_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "how": "one host->device copy of the inputs and one device->host copy of the output "
                              "around the call on device buffers"},
        "sweep": sweep,
        "config2": config2,
        "verify": {**verify, "frac_hbm": verify["gbs"] / hbm},
        "batched_step": {**batched, "frac_hbm": batched["gbs"] / hbm},
        "stream": stream,
        "prefill": {**prefill, "frac_bf16_burst": prefill["tflops"] / bf16,
                    "frac_bf16_sustained": prefill["tflops"] / bf16_sus,
                    "peak_note": "bf16 dense cuBLAS peaks from MEASURED_PEAKS.json (burst and sustained); the "
                                 "kernel's fp16 operands run at the same nominal rate"},
        "gpu_launches": 2 * K,
        "clocks": clk.summary(),
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gbs, dt, reps = oracle_decode_rate(w, N_CELLS, 3, threads, min_seconds=10.0)
        line["cpu_baseline"] = {
            "value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"decode steps (16 query rows each) over the full {N_CELLS}-cell cache, fp64 oracle, "
                      f"{reps} steps in {reps * dt:.1f} s ({dt:.3f} s per step); its cache built by its own "
                      f"append (untimed)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
