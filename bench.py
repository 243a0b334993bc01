#!/usr/bin/env python3
"""Benchmark: one tree-verify MLA attention layer-step on one GB300 (or N replicas).

A step is one full call of the hot path (split-KV attention kernel + LSE combine)
over the 64k verify workload: 1 sequence, 65,536-token prefix, a random 16-node
draft tree, 8 heads, 576-dim bf16 latent rows in a 131,072-slot page_size=1 pool
reached through a random slot permutation. Inputs are seeded and synthetic.

value  = effective KV GB/s = (visible tokens x (1152-B latent row + 4-B slot entry)) / device time
         per step, over all ranks (whole job).
e2e    = the same metric through the public call with host buffers: the step's inputs are
         copied from pinned host memory and the outputs read back inside the timed region.
L2     = each step reads a different one of several distinct pools (together larger than L2).

--impl reference times the float64 CPU oracle on this machine's host cores instead
(the only other program that computes this operation here): each step is one whole
layer-step (all 128 query rows), or a stated row sample scaled to it when K + W whole
steps would run past about two minutes.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/layer-step and effective KV GB/s (% of 8 TB/s HBM) at 64k/185k ctx"
WORKLOAD = ("64k verify: 1 sequence, 65536-token prefix, random 16-node tree, 8 heads, "
            "576-dim bf16 latent rows, 131072-slot pool with a random slot permutation, one layer")
NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_ROTATION = 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value, world):
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, world):
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# the files the tcgen05 attention kernel is built from (with the headers): the ncu traffic
# record below is only used while they are unchanged
TC_SOURCES = ["verify_tc.cu", "common.cuh"]


def traffic_record(fingerprint):
    """dram read+write bytes of the attention kernel from the committed ncu summary, if it is current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("fingerprint") != fingerprint:
        return None
    return d.get("dram_bytes_per_launch")


def cpu_baseline(p, steps, warmup=0, rows_per_step=None):
    """Time the float64 oracle on this machine's host cores. Each step computes ``rows_per_step``
    query rows (all rows of the layer-step by default) over their full visible sets. Returns
    (seconds per full layer-step, OpenMP threads used, rows per step); with a row sample the time
    is scaled to the full layer-step by rows / rows_per_step."""
    import oracle
    from speculative_decode_mla_gb300 import workloads as W
    n = p.rows if rows_per_step is None else min(p.rows, rows_per_step)
    threads = min(oracle.max_threads(), n)
    rng = np.random.default_rng(0)
    times = []
    for it in range(warmup + steps):
        rows = None if n == p.rows else np.sort(rng.choice(p.rows, size=n, replace=False))
        t0 = time.perf_counter()
        oracle.verify_problem(p, W.SOFTMAX_SCALE, rows=rows)
        dt = time.perf_counter() - t0
        if it >= warmup:
            times.append(dt * p.rows / n)
    return float(np.mean(times)), threads, n


def bench_config(world):
    """The workload description both arms print (the same dict for the GPU and the reference arm)."""
    return {"workload": WORKLOAD, "batch": 1, "seq_len": 65536, "tree_nodes": 16, "heads": 8,
            "parallelism": f"replicas x{world}" if world > 1 else "single",
            "l2": f"inputs larger than L2: each step reads the next of {L2_ROTATION} distinct pools"}


def run_reference(args):
    from speculative_decode_mla_gb300 import workloads as W
    rank, world, _ = dist_env()
    if rank != 0:
        return
    p = W.make_problem("64k")
    kv_bytes = W.kv_bytes_per_layer_step(p.seq_lens, p.T)
    # one whole layer-step (all 128 query rows) per step, unless K + W such steps would not end
    # within about two minutes: then a fixed row sample per step, scaled to the layer-step
    t_one, _, _ = cpu_baseline(p, steps=1)
    rows = None
    if t_one * (args.steps + args.warmup) > 120.0:
        rows = max(1, int(p.rows * 120.0 / (t_one * (args.steps + args.warmup))))
    t_step, threads, n = cpu_baseline(p, args.steps, args.warmup, rows_per_step=rows)
    gbs = kv_bytes / t_step / 1e9
    if n == p.rows:
        sample = f"each step is a whole layer-step: all {p.rows} query rows over the 65552-position visible set"
    else:
        sample = (f"{n} of {p.rows} query rows per step over the 65552-position visible set, "
                  f"time scaled x{p.rows / n:.2f} to the layer-step")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "us_per_layer_step": t_step * 1e6, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": bench_config(world),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "host_cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_185k(m, W, dev, steps, warmup, flags=None):
    """The 185k full-depth step: 61 layers, each with its own device-drawn latent pool (about
    13 GB together, far larger than L2) and query, one shared slot table. A step is the 61
    mla_verify_attn calls, replayed from a CUDA graph; returns (s per step, kv bytes per layer, plan)."""
    import torch
    cfg = W.CONFIGS["185k"]
    p0 = W.make_problem(cfg, layer=0, with_kv=False)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    st, sl, tp = t(p0.slot_table), t(p0.seq_lens), t(p0.tree_parent)
    pools = torch.empty((cfg.layers, p0.num_slots, W.D_K), dtype=torch.bfloat16, device=dev)
    qs = torch.empty((cfg.layers, p0.B * p0.T, p0.H, W.D_K), dtype=torch.bfloat16, device=dev)
    for layer in range(cfg.layers):
        m.fill_normal_bf16(pools[layer], W.tensor_seed(cfg.config_id, layer, W.STREAM_KV))
        m.fill_normal_bf16(qs[layer], W.tensor_seed(cfg.config_id, layer, W.STREAM_Q))
    desc = m.make_desc(p0.B, p0.T, p0.H, p0.num_slots, p0.stride, p0.max_seq_len,
                       flags=m.DEFAULT_FLAGS if flags is None else flags)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty((p0.B * p0.T, p0.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p0.B * p0.T, p0.H), dtype=torch.float32, device=dev)
    plan = m.plan(desc, torch.cuda.get_device_properties(dev).multi_processor_count)

    def full_step(sp):
        for layer in range(cfg.layers):
            rc = m.verify_attn_raw(desc, qs[layer].data_ptr(), pools[layer].data_ptr(), st.data_ptr(), sl.data_ptr(),
                                   tp.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp)
            if rc:
                raise m.MLAError(rc, "mla_verify_attn")

    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        full_step(stream.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sp = torch.cuda.current_stream().cuda_stream
        for _ in range(steps):
            full_step(sp)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    step_s = e0.elapsed_time(e1) / 1e3 / steps
    kv = W.kv_bytes_per_layer_step(p0.seq_lens, p0.T)
    del g, pools, qs
    torch.cuda.empty_cache()
    return step_s, kv, plan, cfg.layers


def flush_l2(dev, buf=[]):
    """Write a buffer larger than L2 so the next call starts with cold caches."""
    import torch
    if not buf:
        buf.append(torch.empty(256 << 20, dtype=torch.uint8, device=dev))
    buf[0].fill_(1)


def measure_config(m, W, dev, name, steps, ragged=False):
    """One named workload on a device-drawn pool: graph-replayed µs per call (back to back, same
    pool) and the mean of 5 isolated calls, each after an L2 flush. With ragged=True every sequence
    gets a seeded tree size in 1..T (mla_verify_attn_ragged)."""
    import torch
    p = W.make_problem(name, with_kv=False)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    pool = torch.empty((p.num_slots, W.D_K), dtype=torch.bfloat16, device=dev)
    m.fill_normal_bf16(pool, p.kv_seed)
    q = t(p.q.view(np.int16)).view(torch.bfloat16)
    st, sl, tp = t(p.slot_table), t(p.seq_lens), t(p.tree_parent)
    hint = int((p.seq_lens.astype(np.int64) + p.T).sum())
    desc = m.make_desc(p.B, p.T, p.H, p.num_slots, p.stride, p.max_seq_len, flags=m.DEFAULT_FLAGS,
                       total_tokens_hint=hint if p.B > 1 else 0)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty((p.B * p.T, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B * p.T, p.H), dtype=torch.float32, device=dev)
    plan = m.plan(desc, torch.cuda.get_device_properties(dev).multi_processor_count)

    sizes = t(np.random.default_rng(5).integers(1, p.T + 1, size=p.B).astype(np.int32)) if ragged else None

    def call(sp):
        if ragged:
            rc = m.verify_attn_ragged_raw(desc, q.data_ptr(), pool.data_ptr(), st.data_ptr(), sl.data_ptr(),
                                          sizes.data_ptr(), tp.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                          ws.data_ptr(), ws.numel(), 0, sp)
        else:
            rc = m.verify_attn_raw(desc, q.data_ptr(), pool.data_ptr(), st.data_ptr(), sl.data_ptr(), tp.data_ptr(),
                                   out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp)
        if rc:
            raise m.MLAError(rc, "mla_verify_attn")

    stream = torch.cuda.current_stream()
    for _ in range(3):
        call(stream.cuda_stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sp = torch.cuda.current_stream().cuda_stream
        for _ in range(steps):
            call(sp)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    graph_s = e0.elapsed_time(e1) / 1e3 / steps
    iso = []
    for _ in range(5):
        flush_l2(dev)
        e0.record(stream)
        call(stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        iso.append(e0.elapsed_time(e1) / 1e3)
    kv = W.kv_bytes_per_layer_step(p.seq_lens, p.T)
    if ragged:
        kv = sum(W.kv_bytes_per_layer_step(p.seq_lens[b:b + 1], int(n)) for b, n in enumerate(sizes.cpu().numpy()))
    del g, pool
    torch.cuda.empty_cache()
    return {"us_per_call": graph_s * 1e6, "isolated_us": float(np.mean(iso)) * 1e6,
            "effective_kv_GBs": kv / graph_s / 1e9, "kv_bytes": kv, "splits": plan.num_splits,
            "row_tiles": plan.row_tiles, "graph_steps": steps}


def measure_kv_ops(m, W, dev, p, pools, tables, steps):
    """The KV-pool steps around verification on the 64k workload: Tier-0 compaction of the sequence's
    65552 rows (read + write bytes, against the copy peak), tree-KV append and accept-commit (T = 16)."""
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    N = int(p.seq_lens[0]) + p.T
    sl = t(p.seq_lens)
    dst = torch.empty((N, W.D_K), dtype=torch.bfloat16, device=dev)
    base = t(np.zeros(1, dtype=np.int64))
    new_t = torch.empty_like(tables[0])
    stream = torch.cuda.current_stream()

    def timed(fn):
        for i in range(3):
            fn(i)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                fn(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / steps

    def compact(i):
        r = i % len(pools)
        m.kv_compact(pools[r], dst, tables[r], sl, base, num_nodes=p.T, max_seq_len=p.max_seq_len, new_slot_table=new_t)

    s_compact = timed(compact)
    moved = 2 * N * W.D_K * 2
    tree_kv = torch.zeros((p.T, W.D_K), dtype=torch.bfloat16, device=dev)
    pool_w = pools[0].clone()
    s_append = timed(lambda i: m.tree_kv_append(pool_w, tree_kv, tables[0], sl, max_seq_len=p.max_seq_len))
    st_w, sl_w, tp = tables[0].clone(), sl.clone(), t(p.tree_parent)
    acc = t(np.full((1, p.T), -1, dtype=np.int32))
    zero = t(np.zeros(1, dtype=np.int32))  # an empty accepted path: the call's cost without changing state
    s_commit = timed(lambda i: m.tree_accept_commit(st_w, sl_w, tp, acc, zero, max_seq_len=p.max_seq_len))
    peak = float(peaks()[0]["hbm_gbs"])
    del pool_w, dst

    # Hybrid addressing on compacted pools: each rotated pool compacted to one contiguous prefix at
    # slot 0 (tree after it), then the same verify through the slot table and through
    # mla_verify_attn_hybrid (2-D TMA tiles for the prefix). 4 pools x 76 MB defeat L2.
    L = int(p.seq_lens[0])
    q = t(p.q.view(np.int16)).view(torch.bfloat16)
    tp = t(p.tree_parent)
    cpools, ctables = [], []
    for r in range(len(pools)):
        cp_ = torch.empty((N, W.D_K), dtype=torch.bfloat16, device=dev)
        ct = torch.empty_like(tables[r])
        m.kv_compact(pools[r], cp_, tables[r], sl, base, num_nodes=p.T, max_seq_len=p.max_seq_len, new_slot_table=ct)
        cpools.append(cp_)
        ctables.append(ct)
    tree = ctables[0][:, L:L + p.T].contiguous()
    zero64 = t(np.zeros(1, dtype=np.int64))
    desc = m.make_desc(p.B, p.T, p.H, N, p.stride, p.max_seq_len, flags=m.DEFAULT_FLAGS)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty((p.T, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.T, p.H), dtype=torch.float32, device=dev)
    tp_ = t(p.tree_parent)

    def via_table(i):
        r = i % len(cpools)
        rc = m.verify_attn_raw(desc, q.data_ptr(), cpools[r].data_ptr(), ctables[r].data_ptr(), sl.data_ptr(),
                               tp_.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0,
                               torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc

    def via_hybrid(i):
        r = i % len(cpools)
        rc = m.verify_attn_hybrid_raw(desc, q.data_ptr(), cpools[r].data_ptr(), zero64.data_ptr(), tree.data_ptr(),
                                      sl.data_ptr(), tp_.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                                      ws.numel(), 0, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, rc

    s_table = timed(via_table)
    s_hybrid = timed(via_hybrid)
    del cpools, ctables
    return {"kv_compact": {"us": s_compact * 1e6, "rows": N, "read_plus_write_GBs": moved / s_compact / 1e9,
                           "frac_of_measured_copy": moved / s_compact / 1e9 / peak},
            "tree_kv_append_us": s_append * 1e6, "tree_accept_commit_us": s_commit * 1e6,
            "tree_nodes": p.T,
            "hybrid_addressing_64k": {"workload": "64k verify on compacted pools (contiguous prefix, tree after it)",
                                      "slot_table_us_per_layer_step": s_table * 1e6,
                                      "hybrid_us_per_layer_step": s_hybrid * 1e6,
                                      "hybrid_effective_kv_GBs": W.kv_bytes_per_layer_step(p.seq_lens, p.T) / s_hybrid / 1e9}}


def run_gpu(args):
    import torch
    import speculative_decode_mla_gb300 as m
    from speculative_decode_mla_gb300 import _build
    from speculative_decode_mla_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    _build.build()
    m.load_library()
    stream = torch.cuda.current_stream()

    p = W.make_problem("64k")
    kv_bytes = W.kv_bytes_per_layer_step(p.seq_lens, p.T)
    alg_bytes = W.algorithmic_bytes(p.seq_lens, p.T, p.H)
    flops = W.algorithmic_flops(p.seq_lens, p.T, p.H)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q = t(p.q.view(np.int16)).view(torch.bfloat16)
    st, sl, tp = t(p.slot_table), t(p.seq_lens), t(p.tree_parent)
    pools = [t(p.kv.view(np.int16)).view(torch.bfloat16)]
    for r in range(1, L2_ROTATION):  # distinct pools with the same logical content (slots permuted)
        perm = np.random.default_rng(r).permutation(p.num_slots)
        pools.append(pools[0][torch.from_numpy(perm).to(dev)].contiguous())
    tables = [st] + [None] * (L2_ROTATION - 1)
    for r in range(1, L2_ROTATION):
        perm = np.random.default_rng(r).permutation(p.num_slots)
        tables[r] = t(np.argsort(perm)[p.slot_table].astype(np.int32))
    flags = m.DEFAULT_FLAGS
    desc = m.make_desc(p.B, p.T, p.H, p.num_slots, p.stride, p.max_seq_len, flags=flags)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty((p.B * p.T, p.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((p.B * p.T, p.H), dtype=torch.float32, device=dev)
    props = torch.cuda.get_device_properties(dev)
    plan = m.plan(desc, props.multi_processor_count)

    def step(i, sptr):
        r = i % L2_ROTATION
        rc = m.verify_attn_raw(desc, q.data_ptr(), pools[r].data_ptr(), tables[r].data_ptr(), sl.data_ptr(),
                               tp.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0, sptr)
        if rc:
            raise m.MLAError(rc, "mla_verify_attn")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def capture(fn, n):
        """A CUDA graph of n calls of fn(i, stream): replays the real calls without host launch overhead."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sp = torch.cuda.current_stream().cuda_stream
            for i in range(n):
                fn(i, sp)
        return g

    for i in range(args.warmup):
        step(i, stream.cuda_stream)
    barrier()
    graph = capture(step, args.steps)
    graph.replay()  # untimed: uploads the graph
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        # untimed replays while the sampler starts, so the timed replay begins at load clocks
        t_end = time.time() + 0.3
        while time.time() < t_end:
            graph.replay()
            torch.cuda.synchronize()
        barrier()
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        barrier()
        # keep the GPU busy long enough for a few clock samples when the steps are short
        t_end = time.time() + 0.6
        while time.time() < t_end:
            graph.replay()
            torch.cuda.synchronize()
    step_s = ev0.elapsed_time(ev1) / 1e3 / args.steps
    step_s_max = max_over_ranks(step_s, world)

    # the same step graph with MLA_FLAG_PREFIX_STABLE (consecutive calls never write the pools,
    # slot tables or lengths, so the promise holds): the next call's first prefix tiles are
    # gathered while the previous call's combine is still running
    desc_ps = m.make_desc(p.B, p.T, p.H, p.num_slots, p.stride, p.max_seq_len, flags=flags | m.MLA_FLAG_PREFIX_STABLE)

    def step_ps(i, sptr):
        r = i % L2_ROTATION
        rc = m.verify_attn_raw(desc_ps, q.data_ptr(), pools[r].data_ptr(), tables[r].data_ptr(), sl.data_ptr(),
                               tp.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0, sptr)
        if rc:
            raise m.MLAError(rc, "mla_verify_attn")

    for i in range(3):
        step_ps(i, stream.cuda_stream)
    graph_ps = capture(step_ps, args.steps)
    graph_ps.replay()
    barrier()
    p0_, p1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0_.record(stream)
    graph_ps.replay()
    p1_.record(stream)
    barrier()
    step_ps_s = max_over_ranks(p0_.elapsed_time(p1_) / 1e3 / args.steps, world)
    del graph_ps

    # combine kernel alone on this step's own partials (to isolate the attention kernel's time)
    part_o = ws[: plan.num_splits * p.rows * 512 * 2].view(torch.float16).view(plan.num_splits, p.rows, 512)
    lse_off = ((plan.num_splits * p.rows * 512 * 2 + 255) // 256) * 256
    part_l = ws[lse_off: lse_off + plan.num_splits * p.rows * 4].view(torch.float32).view(plan.num_splits, p.rows)
    o2, l2 = out.view(p.rows, 512).clone(), lse.view(-1).clone()

    def comb(i, sp):
        rc = m.load_library().mla_verify_combine(plan.num_splits, p.rows, 512, part_o.data_ptr(), m.MLA_DTYPE_F16,
                                                 part_l.data_ptr(), o2.data_ptr(), l2.data_ptr(), m.MLA_DTYPE_BF16, sp)
        if rc:
            raise m.MLAError(rc, "mla_verify_combine")

    for i in range(3):
        comb(i, stream.cuda_stream)
    cgraph = capture(comb, args.steps)
    cgraph.replay()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    cgraph.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    combine_s = c0.elapsed_time(c1) / 1e3 / args.steps

    # the attention (split) kernel alone, through mla_verify_attn_partials, on the same rotated pools
    def split_only(i, sptr):
        r = i % L2_ROTATION
        rc = m.verify_attn_partials_raw(desc, q.data_ptr(), pools[r].data_ptr(), tables[r].data_ptr(), sl.data_ptr(),
                                        tp.data_ptr(), ws.data_ptr(), ws.numel(), 0, sptr)
        if rc:
            raise m.MLAError(rc, "mla_verify_attn_partials")

    for i in range(3):
        split_only(i, stream.cuda_stream)
    agraph = capture(split_only, args.steps)
    agraph.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    agraph.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    attn_s = a0.elapsed_time(a1) / 1e3 / args.steps
    del agraph, cgraph

    # end to end through the public call with host buffers
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_q, h_kv = pin(p.q.view(np.int16)), pin(p.kv.view(np.int16))
    h_st, h_sl, h_tp = pin(p.slot_table), pin(p.seq_lens), pin(p.tree_parent)
    h_out = torch.empty((p.B * p.T, p.H, 512), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty((p.B * p.T, p.H), dtype=torch.float32).pin_memory()
    d_q = torch.empty_like(h_q, device=dev)
    d_kv, d_st = torch.empty_like(h_kv, device=dev), torch.empty_like(h_st, device=dev)
    d_sl, d_tp = torch.empty_like(h_sl, device=dev), torch.empty_like(h_tp, device=dev)
    h2d = sum(x.numel() * x.element_size() for x in (h_q, h_kv, h_st, h_sl, h_tp))
    d2h = h_out.numel() * 2 + h_lse.numel() * 4

    def e2e_step():
        for d_, h_ in ((d_q, h_q), (d_kv, h_kv), (d_st, h_st), (d_sl, h_sl), (d_tp, h_tp)):
            d_.copy_(h_, non_blocking=True)
        rc = m.verify_attn_raw(desc, d_q.data_ptr(), d_kv.data_ptr(), d_st.data_ptr(), d_sl.data_ptr(),
                               d_tp.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0,
                               stream.cuda_stream)
        if rc:
            raise m.MLAError(rc, "mla_verify_attn")
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / e2e_steps, world)

    total_kv = sum_over_ranks(kv_bytes, world)
    value = total_kv / step_s_max / 1e9
    pk, pk_kind = peaks()
    peak_hbm = float(pk["hbm_gbs"])
    achieved = alg_bytes / attn_s / 1e9
    traffic = traffic_record(_build.source_fingerprint(TC_SOURCES)) if plan.kernel == 0 else None
    launches = 2 * args.steps  # attention kernel + combine kernel per step

    base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_cpu, cores, _ = cpu_baseline(p, steps=2)
        base = {"value": kv_bytes / t_cpu / 1e9, "unit": "GB/s", "cores": cores, "host_cores": os.cpu_count(),
                "kind": "oracle",
                "sample": f"2 whole layer-steps: all {p.rows} query rows over the 65552-position visible set",
                "us_per_layer_step": t_cpu * 1e6}
    clocks = clk.summary()
    # the metric's own config also as a single isolated call (L2 flushed before it)
    iso = []
    for _ in range(5):
        flush_l2(dev)
        e0.record(stream)
        step(0, stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        iso.append(e0.elapsed_time(e1) / 1e3)
    isolated_s = float(np.mean(iso))
    others = None
    if not args.no_extra:
        others = {name: measure_config(m, W, dev, name, steps=st_)
                  for name, st_ in (("tiny", 50), ("batched", 20), ("wide", 5), ("wide_identity", 5))}
        others["batched_ragged_trees"] = measure_config(m, W, dev, "batched", steps=20, ragged=True)
    kv_ops = None if args.no_extra else measure_kv_ops(m, W, dev, p, pools, tables, steps=20)
    at_185k = None
    if not args.no_185k:
        s185, kv185, plan185, layers = measure_185k(m, W, dev, steps=max(3, min(args.steps, 10)), warmup=args.warmup)
        s185ps, _, _, _ = measure_185k(m, W, dev, steps=max(3, min(args.steps, 10)), warmup=args.warmup,
                                       flags=m.DEFAULT_FLAGS | m.MLA_FLAG_PREFIX_STABLE)
        s185ps = max_over_ranks(s185ps, world)
        s185 = max_over_ranks(s185, world)
        gbs185 = sum_over_ranks(kv185, world) * layers / s185 / 1e9
        at_185k = {"workload": ("185k full-depth step: 1 sequence, 184320-token prefix, random 32-node tree, "
                                "8 heads, 61 layers each with its own 184352-slot pool (12.95 GB), shared slot table"),
                   "us_per_layer_step": s185 / layers * 1e6, "ms_per_step": s185 * 1e3, "value": gbs185,
                   "unit": "GB/s", "hbm_frac_of_8tbs": gbs185 / world / NOMINAL_HBM_GBS,
                   "hbm_frac_of_measured": gbs185 / world / float(peaks()[0]["hbm_gbs"]),
                   "splits": plan185.num_splits, "row_tiles": plan185.row_tiles,
                   "with_prefix_stable_flag": {"us_per_layer_step": s185ps / layers * 1e6,
                                               "value": sum_over_ranks(kv185, world) * layers / s185ps / 1e9},
                   "steps": max(3, min(args.steps, 10)), "gpu_launches": 2 * layers * max(3, min(args.steps, 10))}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s_max * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": bench_config(world),
            "plan": {"kernel": "simt" if plan.kernel == 1 else "tcgen05", "splits": plan.num_splits,
                     "chunk_tokens": plan.chunk_tokens},
            "us_per_layer_step": step_s_max * 1e6,
            "hbm_frac_of_8tbs": value / world / NOMINAL_HBM_GBS,
            "hbm_frac_of_measured": value / world / peak_hbm,
            "tensor_frac_of_measured": flops / step_s_max / 1e12 / float(pk["bf16_tflops"]),
            "attn_kernel_us": attn_s * 1e6, "combine_kernel_us": combine_s * 1e6,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_hbm, "unit": "GB/s",
                         "frac": achieved / peak_hbm, "traffic": traffic,
                         "peak_kind": f"{pk_kind} copy bandwidth (burst)",
                         "algorithmic_bytes_per_launch": alg_bytes},
            "e2e": {"value": total_kv / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "us_per_step": e2e_s * 1e6},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        if base is not None:
            line["cpu_baseline"] = base
        if at_185k is not None:
            line["at_185k"] = at_185k
        line["isolated_us_per_layer_step"] = isolated_s * 1e6
        line["with_prefix_stable_flag"] = {
            "us_per_layer_step": step_ps_s * 1e6, "value": total_kv / step_ps_s / 1e9, "unit": "GB/s",
            "note": "MLA_FLAG_PREFIX_STABLE: the caller promises the preceding kernel writes no prefix input; "
                    "results are bit-identical (tests/test_gpu_prefix_stable.py)"}
        if others is not None:
            line["other_configs"] = others
        if kv_ops is not None:
            line["kv_pool_steps"] = kv_ops
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_only(args):
    """One named workload: 3 eager calls, then ``--steps`` calls replayed from a graph and 5 isolated
    calls (see measure_config); prints one JSON line of its figures."""
    import torch
    import speculative_decode_mla_gb300 as m
    from speculative_decode_mla_gb300 import _build
    from speculative_decode_mla_gb300 import workloads as W
    if args.only not in W.CONFIGS:
        raise SystemExit(f"--only: unknown workload {args.only!r} (one of {', '.join(W.CONFIGS)})")
    _build.build()
    m.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    r = measure_config(m, W, dev, args.only, steps=args.steps)
    print(json.dumps({"workload": args.only, **r}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-185k", action="store_true", help="skip the 185k full-depth step measurement")
    ap.add_argument("--no-extra", action="store_true", help="skip the tiny/batched/wide timings")
    ap.add_argument("--only", default=None,
                    help="time one named workload alone (tiny, 64k, 185k = one of its layers, batched, wide, "
                         "wide_identity) and print its figures; a small, self-contained case for profilers")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = dist_env()[1]
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} needs {args.gpus} processes, one per GPU (torchrun --nproc-per-node "
                 f"{args.gpus}); this run has WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
