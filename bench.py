"""Benchmark of the paged-KV attention hot path on one GB300 (or N replicas).

A step is one decode step of one attention layer on the largest single-GPU
decode workload, the Qwen3-8B attention shape: batch 256, 32 q / 8 kv heads,
head_dim 128, block_size 256, context_lens lognormal (median 1024, capped
8192), sequences 0..127 sharing their first 4 physical blocks (prefix cache,
ref_count 128), pool = 1.2x the blocks needed, random block permutation, bf16
N(0,1).  The step is one call of pa_decode_shared_prefix with the new token's
store fused: a prefix kernel attends the 128 sharing sequences' query heads to
their 4 shared blocks once per kv head, then the split-KV GQA decode kernel
stores each sequence's new K/V row to its slot, reads every other context row
through the block tables and merges the prefix partials.  All inputs are
resident in HBM before the timed region; L2 is flushed before every timed
step (a 256 MiB write, then a 256 MiB read of another buffer, so that the
step starts with no line of its inputs and no dirty line in L2).  `value` is decode tokens/s (one layer) over all
ranks; `e2e` is the same metric through the public API with the step's
inputs copied from pinned host memory and the output copied back inside the
timed region.  The roofline counts the bytes the step must move with every
physical K/V row once (the 4 shared blocks once, not once per sequence);
the logical figure (shared rows counted per sequence) is reported beside it.

Sub-records, each with its own roofline: the other decode workloads (tiny,
Qwen3-0.6B, 32k long context), the varlen prefill with prefix cache, and
the Gumbel-max sampler.  `cpu_baseline` is the oracle timed on the host's
cores (single-threaded and on all cores) on the same workload.

`--impl reference` runs the CPU oracle (the only reference this path has) on
the same workload and prints its own line.

Multi-GPU (torchrun): every rank serves its own batch with its own pool
(replicas, weak scaling); no collective is on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn tokens/s and HBM GB/s vs GB300 peak; prefill TFLOP/s"
HEADLINE_CONFIG = 3
WORKLOAD = ("qwen3-8b decode step, 1 layer: batch 256, 32 q / 8 kv heads, head_dim 128, block_size 256, "
            "context_lens lognormal (median 1024, sigma 1, capped 8192), sequences 0..127 share their first 4 "
            "physical blocks (prefix cache), pool = 1.2x blocks needed, random block permutation; "
            "pa_decode_shared_prefix with the new token's store fused (shared prefix attended once per kv head, "
            "split-KV decode over each sequence's own blocks)")
SUB_DECODE_CONFIGS = (1, 2, 4)
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, 1900.0, "fallback"


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


DECODE_SOURCES = ["paged_kv_cache_store_gb300/csrc/pa_decode.cu", "paged_kv_cache_store_gb300/csrc/pa_tcgen05.cuh",
                  "paged_kv_cache_store_gb300/csrc/pa_internal.cuh"]
PREFILL_SOURCES = ["paged_kv_cache_store_gb300/csrc/pa_prefill.cu", "paged_kv_cache_store_gb300/csrc/pa_tcgen05.cuh",
                   "paged_kv_cache_store_gb300/csrc/pa_internal.cuh"]


def recorded_traffic(kernel: str, workload_key: str, sources=DECODE_SOURCES):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel, {}).get(workload_key)
    if not rec or rec.get("source_digest") != source_digest(sources):
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks, throttle reasons and utilisation
    during the timed region (into a temporary CSV, or `path`)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index: int, path: str | None = None):
        import tempfile
        self.proc = None
        self.gpu = gpu_index
        self.keep = path is not None
        if path is None:
            fd, path = tempfile.mkstemp(prefix="pa_clocks_", suffix=".csv")
            os.close(fd)
        self.path = path

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, busy_sm, reasons, n_busy = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                c = [x.strip() for x in ln.split(",")]
                if len(c) < 10:
                    continue
                try:
                    clk, cmax, util = float(c[1]), float(c[2]), float(c[9])
                except ValueError:
                    continue
                sm.append(clk)
                mx.append(cmax)
                if util >= 50.0:  # a sample taken while kernels were running
                    n_busy += 1
                    busy_sm.append(clk)
                    for n, v in zip(names, c[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(busy_sm or sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": n_busy}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dev, ws: int) -> float:
    """The largest of every rank's x (all ranks get it); x itself when alone.
    The job's time is its slowest rank's."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws: int, units_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job units/s: every rank processed units_per_rank per step (weak
    scaling), and the job took the slowest rank's total_ms."""
    return ws * units_per_rank * steps / (total_ms / 1000.0)


def decode_bytes(inp):
    """Algorithmic bytes of one fused store + decode launch.

    Every context row of every (sequence, kv head) is read once, q is read
    and out written, and each sequence's new K/V row is read and written to
    its slot.  `unique` counts each physical pool row once (rows of blocks
    that several sequences share are read from HBM once; their re-reads come
    from L2); `logical` counts them once per sequence that reads them."""
    row = inp.num_kv_heads * inp.head_dim * 2 * 2            # K and V of one token, all kv heads
    ctx = inp.context_lens.astype(np.int64)
    logical_rows = int(ctx.sum())
    rows_in_block = {}
    for b in range(inp.batch):
        n = int(ctx[b])
        for j in range((n + inp.block_size - 1) // inp.block_size):
            blk = int(inp.block_tables[b, j])
            used = min(inp.block_size, n - j * inp.block_size)
            rows_in_block[blk] = max(rows_in_block.get(blk, 0), used)
    unique_rows = sum(rows_in_block.values())
    qo = 2 * inp.batch * inp.num_q_heads * inp.head_dim * 2
    new_rows = 2 * inp.batch * row                           # read from new_k/new_v, written to the slot
    return {"logical": logical_rows * row + qo + new_rows, "unique": unique_rows * row + qo + new_rows,
            "logical_rows": logical_rows, "unique_rows": unique_rows}


def oracle_decode_step(inp, O, threads: int):
    """One step of the oracle on a decode workload: slot mapping, store of the
    new rows into copies of the caches, decode attention (on `threads` host
    threads; 1 = the oracle as it stands)."""
    from oracle import parallel as OP
    kc, vc = inp.k_cache.copy(), inp.v_cache.copy()
    slots = np.array([O.decode_slot(inp.block_tables[b], inp.block_size, int(inp.context_lens[b]))
                      for b in range(inp.batch)], np.int32)
    O.store_kvcache(inp.new_k, inp.new_v, kc, vc, slots)
    if threads == 1:
        return O.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale)
    return OP.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale, threads=threads)


def time_oracle(inp, O, threads: int, budget_s: float):
    """Oracle decode steps on the workload for about budget_s seconds (at
    least one); returns (tokens/s, steps, seconds)."""
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle_decode_step(inp, O, threads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return steps * inp.batch / el, steps, el


def cpu_baseline(inp, budget_s: float):
    """The oracle as it stands (float64 C, scalar loops) on the host cores:
    on all cores (rows split between threads) for about budget_s, and one
    single-threaded step."""
    import oracle as O
    from oracle import parallel as OP
    O.lib()
    n = OP.host_threads()
    tps, steps, el = time_oracle(inp, O, n, budget_s)
    tps1, steps1, el1 = time_oracle(inp, O, 1, 0.0)
    return {"value": tps, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{steps} full steps of the same workload in {el:.1f} s on {n} threads "
                      f"(rows split between threads, each row by the unchanged float64 oracle)",
            "single_thread": {"value": tps1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{steps1} full step(s) in {el1:.1f} s"}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as O
    from oracle import parallel as OP
    from paged_kv_cache_store_gb300.workloads import decode_config
    inp = decode_config(HEADLINE_CONFIG)
    O.lib()
    n = OP.host_threads()
    for _ in range(args.warmup):
        oracle_decode_step(inp, O, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_decode_step(inp, O, n)
    el = time.perf_counter() - t0
    value = args.steps * inp.batch / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": WORKLOAD, "global_batch": inp.batch, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle",
                             "sample": f"full workload, {args.steps} steps, rows split over {n} threads"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def prefill_pairs(p):
    """Unmasked (query, key) pairs of the causal prefill: query i of a sequence
    with c cached tokens sees c + i + 1 keys."""
    tot = 0
    for s in range(p.num_seqs):
        c, lq = int(p.seqlens_k[s] - p.seqlens_q[s]), int(p.seqlens_q[s])
        tot += lq * c + lq * (lq + 1) // 2
    return tot


def _to_dev(a, dev, bf=False):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf else np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if bf else t).to(dev)


class L2Flush:
    """Leaves L2 cold and clean before a timed call: a 256 MiB write evicts
    every line the call could reuse, then a 256 MiB read of a second buffer
    writes the first buffer's dirty lines back to HBM before the timed region
    starts.  After the write alone, L2 (129 MB) is full of dirty lines and
    the timed call would pay for writing them back as its first reads
    allocate lines (3-7 us on the decode workloads)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
        self.s = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.s)


def _event_times(fn, steps, stream, flush):
    """Per-call CUDA-event times (ms) of `steps` calls of fn, L2 flushed before each."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a_, b_ in ev:
        flush()
        a_.record(stream)
        fn()
        b_.record(stream)
    torch.cuda.synchronize()
    return [a_.elapsed_time(b_) for a_, b_ in ev]


def _check_device(pa):
    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")


def measure_decode_config(cfg, args, dev, stream, flush, hbm_peak):
    """A decode workload's fused store + decode step (one launch), L2 flushed
    before each call: time, tokens/s and its own roofline."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import decode_config
    inp = decode_config(cfg)
    kc, vc, q = _to_dev(inp.k_cache, dev, True), _to_dev(inp.v_cache, dev, True), _to_dev(inp.q, dev, True)
    nk, nv = _to_dev(inp.new_k, dev, True), _to_dev(inp.new_v, dev, True)
    bt, ctx = _to_dev(inp.block_tables, dev), _to_dev(inp.context_lens, dev)
    out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
    wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev)

    def step():
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv)

    for _ in range(max(3, args.warmup)):
        step()
    ms = _event_times(step, args.steps, stream, flush)
    _check_device(pa)
    ms_avg = sum(ms) / len(ms)
    by = decode_bytes(inp)
    gbs = by["unique"] / (ms_avg / 1000.0) / 1e9
    del kc, vc
    torch.cuda.empty_cache()
    return {"workload": inp.name, "batch": inp.batch, "ms": ms_avg, "ms_median": float(np.median(ms)),
            "tokens_per_s": inp.batch / (ms_avg / 1000.0),
            "roofline": {"bound": "hbm", "kernel": f"decode_kernel<{inp.num_q_heads // inp.num_kv_heads}, store>",
                         "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "frac_of_nominal_8TBps": gbs / 8000.0, "algorithmic_bytes_per_launch": by["unique"],
                         "traffic": None},
            "note": "launch-latency bound (about 1 MB moved)" if cfg == 1 else None}


def measure_prefill(args, dev, stream, flush, bf16_peak):
    """The varlen prefill workload: slot mapping + store of the uncached suffix,
    then causal prefill over the paged pool; and the same step as one fused
    launch.  Returns a JSON-able dict."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import prefill_config

    p = prefill_config(5)
    kc, vc = _to_dev(p.k_cache, dev, True), _to_dev(p.v_cache, dev, True)
    q, nk, nv = _to_dev(p.q, dev, True), _to_dev(p.new_k, dev, True), _to_dev(p.new_v, dev, True)
    bt, cq, ck = _to_dev(p.block_tables, dev), _to_dev(p.cu_seqlens_q, dev), _to_dev(p.cu_seqlens_k, dev)
    slots = torch.empty(p.total_q, dtype=torch.int32, device=dev)
    out = torch.empty(p.total_q, p.num_q_heads, p.head_dim, dtype=torch.bfloat16, device=dev)
    mq, mk = int(p.seqlens_q.max()), int(p.seqlens_k.max())

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q, out=slots)
        if ev:
            ev[3].record(stream)
        pa.store_kvcache(nk, nv, kc, vc, slots)
        if ev:
            ev[1].record(stream)
        pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out)
        if ev:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for e in evs:
        flush()
        step(e)
    torch.cuda.synchronize()
    _check_device(pa)
    pre_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)
    step3_ms = sum(e[0].elapsed_time(e[2]) for e in evs) / len(evs)
    # The same step as one launch: the fused store + prefill (cooperative).
    wsf = pa.prefill_store_workspace(dev)

    def fused():
        pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out, new_k=nk, new_v=nv,
                          workspace=wsf)

    for _ in range(3):
        fused()
    fused_ms = sum(_event_times(fused, args.steps, stream, flush)) / args.steps
    _check_device(pa)
    slotmap_store_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    store_ms = sum(e[3].elapsed_time(e[1]) for e in evs) / len(evs)
    flops = 4 * p.head_dim * p.num_q_heads * prefill_pairs(p)
    tflops = flops / (pre_ms / 1000.0) / 1e12
    store_bytes = p.total_q * p.num_kv_heads * p.head_dim * 2 * 4
    del kc, vc
    torch.cuda.empty_cache()
    return {"workload": "varlen causal prefill, 16 seqs, 32 q / 8 kv heads, Lk ~ U[128,2048], 0..3 cached "
                        "blocks per seq, block_size 256 (suffix stored via slot_mapping first)",
            "total_q": p.total_q, "ms_prefill": pre_ms, "ms_slotmap_store": slotmap_store_ms, "ms_store": store_ms,
            "ms_step_3_launches": step3_ms, "ms_step_fused": fused_ms,
            "algorithmic_flops": flops,
            "roofline": {"bound": "tensor", "kernel": "prefill_pair_kernel<0>", "achieved": tflops, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": tflops / bf16_peak, "peak_kind": "burst (timed alone)",
                         "traffic": recorded_traffic("prefill_pair_kernel<0>", "prefill", PREFILL_SOURCES)},
            "store_gbs": store_bytes / (store_ms / 1000.0) / 1e9}


def measure_sampler(args, dev, stream, flush, hbm_peak):
    """The Gumbel-max sampler after the decode step: 64 rows over the Qwen3
    vocabulary (bf16 logits, fp32 Exp(1) draws).  HBM-bound: every logit and
    draw is read once."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import sampler_config

    sp = sampler_config(64)
    lg = _to_dev(sp.logits, dev, True)
    temps = torch.from_numpy(sp.temperatures).to(dev)
    noise = torch.from_numpy(sp.exp_noise).to(dev)
    out = torch.empty(sp.batch, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        pa.sample_gumbel(lg, temps, noise, out=out)
    ms = sum(_event_times(lambda: pa.sample_gumbel(lg, temps, noise, out=out), args.steps, stream, flush))
    ms /= args.steps
    _check_device(pa)
    alg = sp.batch * sp.vocab * (2 + 4) + sp.batch * (4 + 4)
    gbs = alg / (ms / 1000.0) / 1e9
    return {"workload": sp.name + ", fp32 Exp(1) draws", "ms": ms, "algorithmic_bytes": alg,
            "roofline": {"bound": "hbm", "kernel": "sample_gumbel_kernel", "achieved": gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs / hbm_peak, "traffic": None},
            "l2": "flushed (256 MiB write + 256 MiB read) before every timed call; inputs 58 MB"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import decode_config

    dev = torch.device("cuda", local)
    hbm, bf16_peak, peak_kind = peaks()
    inp = decode_config(HEADLINE_CONFIG)
    kc, vc = _to_dev(inp.k_cache, dev, True), _to_dev(inp.v_cache, dev, True)
    q = _to_dev(inp.q, dev, True)
    nk, nv = _to_dev(inp.new_k, dev, True), _to_dev(inp.new_v, dev, True)
    bt, ctx = _to_dev(inp.block_tables, dev), _to_dev(inp.context_lens, dev)
    slots = torch.empty(inp.batch, dtype=torch.int32, device=dev)
    out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
    wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev)
    wsx = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev, shared_prefix=True)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    by = decode_bytes(inp)
    L2 = (f"flushed (256 MiB write + 256 MiB read) before every timed step; K/V pool {kc.numel() * 4 / 2**30:.2f} GiB > L2")

    def step():  # prefix kernel + decode kernel (which stores the new K/V rows, then attends)
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsx, out=out, new_k=nk, new_v=nv, shared_prefix=True)

    def step_plain():  # one kernel, no grouping: every sequence streams its whole context
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv)

    def step_unfused():  # the same work as three launches
        pa.slot_mapping_decode(bt, ctx, inp.block_size, out=slots)
        pa.store_kvcache(nk, nv, kc, vc, slots)
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out)

    for _ in range(max(3, args.warmup)):
        step()
        step_plain()
        step_unfused()
    torch.cuda.synchronize()
    _check_device(pa)

    def flushed_steps(n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a_, b_ in ev:
            flush()
            a_.record(stream)
            step()
            b_.record(stream)
        return ev

    # Clocks: sampled while the same flushed steps run back to back for at
    # least `sustain_s` (so the sampler sees the GPU under this load), then
    # through the timed region itself.
    probe = flushed_steps(8)
    torch.cuda.synchronize()
    est = (float(np.median([a.elapsed_time(b) for a, b in probe])) + 0.05) / 1000.0
    n_sustain = int(math.ceil(args.sustain_s / est))
    with ClockSampler(local, args.clock_log) as clk:
        sus = flushed_steps(n_sustain)
        torch.cuda.synchronize()
        # Headline: exactly `steps` whole steps, L2 flushed before each,
        # bracketed by a barrier and a synchronize on both sides.
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ev = flushed_steps(args.steps)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
    _check_device(pa)
    sus_ms = [a.elapsed_time(b) for a, b in sus]
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dev, ws)
    ms_per_step = total_ms / args.steps
    value = job_throughput(ws, inp.batch, args.steps, total_ms)

    # The same step without grouping (one launch of the fused kernel), and as
    # three launches (slot mapping, store, decode), for comparison.
    plain_ms = sum(_event_times(step_plain, args.steps, stream, flush)) / args.steps
    unfused_ms = sum(_event_times(step_unfused, args.steps, stream, flush)) / args.steps
    # The plain decode launch alone (store done before it).
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        pa.slot_mapping_decode(bt, ctx, inp.block_size, out=slots)
        kev[i][0].record(stream)
        pa.store_kvcache(nk, nv, kc, vc, slots)
        kev[i][1].record(stream)
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out)
        kev[i][2].record(stream)
    torch.cuda.synchronize()
    store_ms = [e[0].elapsed_time(e[1]) for e in kev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in kev]

    # End to end through the public API: host inputs -> device, step, output -> host.
    # The step's inputs (q, new K/V rows, block tables, context lengths) sit in
    # one pinned host buffer and go over in one copy; the kernel reads device
    # views of the copy.
    host_parts = [np.ascontiguousarray(x).view(np.uint8).reshape(-1)
                  for x in (inp.q, inp.new_k, inp.new_v, inp.block_tables, inp.context_lens)]
    offs, tot = [], 0
    for x in host_parts:
        offs.append(tot)
        tot += (x.size + 255) // 256 * 256
    h_pack = torch.zeros(tot, dtype=torch.uint8).pin_memory()
    hp = h_pack.numpy()
    for o, x in zip(offs, host_parts):
        hp[o:o + x.size] = x
    d_pack = torch.empty(tot, dtype=torch.uint8, device=dev)

    def dview(i, dtype, shape):
        n = host_parts[i].size
        return d_pack[offs[i]:offs[i] + n].view(dtype).view(shape)

    e_q = dview(0, torch.bfloat16, q.shape)
    e_nk, e_nv = dview(1, torch.bfloat16, nk.shape), dview(2, torch.bfloat16, nv.shape)
    e_bt, e_ctx = dview(3, torch.int32, bt.shape), dview(4, torch.int32, ctx.shape)
    h_out = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(x.size for x in host_parts)
    d2h = h_out.numel() * h_out.element_size()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps + 2):
        if i >= 2:
            flush()
            e2e_ev[i - 2][0].record(stream)
        d_pack.copy_(h_pack, non_blocking=True)
        pa.decode(e_q, kc, vc, e_bt, e_ctx, inp.scale, workspace=wsx, out=out, new_k=e_nk, new_v=e_nv,
                  shared_prefix=True)
        h_out.copy_(out, non_blocking=True)
        if i >= 2:
            e2e_ev[i - 2][1].record(stream)
    torch.cuda.synchronize()
    if not np.array_equal(h_out.view(torch.int16).numpy(), out.cpu().view(torch.int16).numpy()):
        raise RuntimeError("end-to-end output differs from the device output")
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), dev, ws)
    e2e_value = job_throughput(ws, inp.batch, args.steps, e2e_ms)
    _check_device(pa)
    del kc, vc, flush
    torch.cuda.empty_cache()

    flush = L2Flush(dev)
    sub = {}
    for cfg in SUB_DECODE_CONFIGS:
        sub[f"decode_config{cfg}"] = measure_decode_config(cfg, args, dev, stream, flush, hbm)
    prefill = None if args.no_prefill else measure_prefill(args, dev, stream, flush, bf16_peak)
    sampler = measure_sampler(args, dev, stream, flush, hbm)

    if rank == 0:
        achieved = by["unique"] / (ms_per_step / 1000.0) / 1e9
        achieved_logical = by["logical"] / (ms_per_step / 1000.0) / 1e9
        traffic = recorded_traffic("decode_prefix_tc_kernel<4> + decode_kernel<4, store>", "qwen3-8b")
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic (seeded N(0,1) bf16, random block tables)",
            "config": {"workload": WORKLOAD, "global_batch": inp.batch * ws, "seq_len": "lognormal(1024), cap 8192",
                       "parallelism": f"replicas x{ws}", "l2": L2},
            "roofline": {"bound": "hbm",
                         "kernel": "decode_prefix_tc_kernel<4> + decode_kernel<4, store> (one pa_decode_shared_prefix call)",
                         "achieved": achieved,
                         "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "peak_kind": peak_kind,
                         "frac_of_nominal_8TBps": achieved / 8000.0, "traffic": traffic,
                         "algorithmic_bytes_per_launch": by["unique"],
                         "bytes_basis": "unique: every physical K/V row once (the 4 shared blocks once)",
                         "logical": {"algorithmic_bytes_per_launch": by["logical"], "achieved": achieved_logical,
                                     "frac": achieved_logical / hbm,
                                     "basis": "shared prefix rows counted once per sequence that reads them"},
                         "launch_ms": ms_per_step, "duration_basis": "the whole call (both kernels), CUDA events",
                         "plain_decode_ms": sum(dec_ms) / len(dec_ms), "store_ms": sum(store_ms) / len(store_ms)},
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * args.steps,
            "sustained": {"steps": n_sustain, "seconds": sum(sus_ms) / 1000.0,
                          "ms_median": float(np.median(sus_ms)),
                          "note": "the same flushed step back to back before the timed region, for the clock record"},
            "plain_fused_step": {"ms_per_step": plain_ms, "kernels": "decode_kernel<4, store> (pa_decode_store, no grouping)",
                                 "tokens_per_s": ws * inp.batch / (plain_ms / 1000.0),
                                 "frac_unique_bytes": by["unique"] / (plain_ms / 1000.0) / 1e9 / hbm},
            "unfused_step": {"ms_per_step": unfused_ms, "kernels": "slot_mapping_decode + store_kvcache + decode",
                             "tokens_per_s": ws * inp.batch / (unfused_ms / 1000.0)},
            "clocks": clk.summary(),
            "decode_configs": sub,
            "prefill": prefill,
            "sampler": sampler,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_report(args):
    """The per-configuration results table (markdown on stdout): decode
    configurations 1-4 run the fused store + decode step, configuration 5 the
    varlen prefill (and its fused store + prefill step).  Device time: median
    of `steps` calls, CUDA events, L2 flushed before each.  Parity: against
    the oracle on the same inputs, every output row.  Oracle time: one step
    of the oracle on all host cores (rows split between threads) and, for
    decode, one single-threaded step."""
    import torch
    import oracle as O
    from oracle import parallel as OP
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import decode_config, prefill_config, bf16_bits_to_f32
    O.lib()
    nthr = OP.host_threads()
    dev = torch.device("cuda", 0)
    hbm, bf16_peak, kind = peaks()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        ms = _event_times(fn, args.steps, stream, flush)
        _check_device(pa)
        return float(np.median(ms))

    def host(t):
        return bf16_bits_to_f32(t.cpu().view(torch.int16).numpy().view(np.uint16)).astype(np.float64)

    lines = ["| Config | GPU time | tokens/s (decode, 1 layer) | GB/s (algorithmic, unique rows) | TFLOP/s "
             "| % roofline | Oracle (all cores / 1 thread) | Parity, all rows (max / mean abs) |", "|" + "---|" * 8]
    for cfg in (1, 2, 3, 4):
        inp = decode_config(cfg)
        kc, vc, q = _to_dev(inp.k_cache, dev, True), _to_dev(inp.v_cache, dev, True), _to_dev(inp.q, dev, True)
        nk, nv = _to_dev(inp.new_k, dev, True), _to_dev(inp.new_v, dev, True)
        bt, ctx = _to_dev(inp.block_tables, dev), _to_dev(inp.context_lens, dev)
        out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
        wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev)
        ms = timed(lambda: pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv))
        ms_plain = None
        if cfg == 3:  # the shared-prefix call is the one that counts; the plain fused step beside it
            ms_plain = ms
            wsx = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev, shared_prefix=True)
            ms = timed(lambda: pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsx, out=out, new_k=nk, new_v=nv,
                                         shared_prefix=True))
        t0 = time.perf_counter()
        want = oracle_decode_step(inp, O, nthr)
        oracle_s = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle_decode_step(inp, O, 1)
        oracle_1 = time.perf_counter() - t0
        err = np.abs(host(out) - want)
        by = decode_bytes(inp)
        gbs = by["unique"] / (ms / 1000.0) / 1e9
        note = f" ({by['logical'] / (ms / 1000.0) / 1e9:,.0f} logical)" if by["logical"] != by["unique"] else ""
        if ms_plain is not None:
            note += f"; without grouping {ms_plain * 1000:.1f} us, {by['unique'] / (ms_plain / 1000.0) / 1e9:,.0f}"
        lines.append(f"| {cfg} {inp.name} | {ms * 1000:.1f} us | {inp.batch / (ms / 1000.0):,.0f} | "
                     f"{gbs:,.0f}{note} | — | {100 * gbs / hbm:.1f} % of {hbm:.0f} ({kind}) | "
                     f"{oracle_s:.2f} s on {nthr} / {oracle_1:.2f} s | {err.max():.2e} / {err.mean():.2e} |")
        del kc, vc
        torch.cuda.empty_cache()
    p = prefill_config(5)
    kc, vc, q = _to_dev(p.k_cache, dev, True), _to_dev(p.v_cache, dev, True), _to_dev(p.q, dev, True)
    nk, nv = _to_dev(p.new_k, dev, True), _to_dev(p.new_v, dev, True)
    bt, cq, ck = _to_dev(p.block_tables, dev), _to_dev(p.cu_seqlens_q, dev), _to_dev(p.cu_seqlens_k, dev)
    out = torch.empty(p.total_q, p.num_q_heads, p.head_dim, dtype=torch.bfloat16, device=dev)
    mq, mk = int(p.seqlens_q.max()), int(p.seqlens_k.max())
    slots = pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q)
    pa.store_kvcache(nk, nv, kc, vc, slots)
    ms = timed(lambda: pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out))
    wsf = pa.prefill_store_workspace(dev)
    ms_fused = timed(lambda: pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out,
                                               new_k=nk, new_v=nv, workspace=wsf))
    flops = 4 * p.head_dim * p.num_q_heads * prefill_pairs(p)
    okc, ovc = p.k_cache.copy(), p.v_cache.copy()
    oslots = np.concatenate([O.slot_mapping(p.block_tables[s], p.block_size, int(p.seqlens_k[s] - p.seqlens_q[s]),
                                            int(p.seqlens_k[s])) for s in range(p.num_seqs)])
    O.store_kvcache(p.new_k, p.new_v, okc, ovc, oslots)
    t0 = time.perf_counter()
    want = OP.prefill(p.q, okc, ovc, p.cu_seqlens_q, p.cu_seqlens_k, p.scale, block_tables=p.block_tables)
    oracle_s = time.perf_counter() - t0
    err = np.abs(host(out) - want)
    tf = flops / (ms / 1000.0) / 1e12
    lines.append(f"| 5 {p.name} | {ms * 1000:.1f} us (fused store + prefill: {ms_fused * 1000:.1f} us) | — | — | "
                 f"{tf:.0f} | {100 * tf / bf16_peak:.1f} % of {bf16_peak:.0f} ({kind}) | "
                 f"{oracle_s:.1f} s on {nthr} | {err.max():.2e} / {err.mean():.2e} |")
    print("\n".join(lines))
    return 0


def run_profile_case(args):
    """Small launch sequences for ncu captures (no JSON line).

    decode-small: the Qwen3-0.6B shape (batch 64, 16 q / 8 kv heads, fused
    store) with context lengths ~ U[1, 1536], about 190 MB of K/V (more than
    the 129 MB L2, a fraction of the full case), for multi-pass captures.
    decode-qwen3-8b: the headline workload itself (about 2.4 GB on the
    device; pa_decode_shared_prefix: a prefix kernel and a decode kernel
    per call), for single-pass captures (DRAM bytes and duration).
    decode-shared-small: the same shape at batch 64 (32/8 heads, lognormal
    contexts, sequences 0..31 share their first 4 blocks; about 0.4 GB of
    K/V), pa_decode_shared_prefix, for multi-pass captures of both kernels.
    prefill: the prefill workload (plain prefill launches after one store).
    Each runs `warmup` then `steps` launches with an L2 flush before each."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import make_decode, decode_config, prefill_config
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    if args.profile_case == "prefill":
        p = prefill_config(5)
        kc, vc, q = _to_dev(p.k_cache, dev, True), _to_dev(p.v_cache, dev, True), _to_dev(p.q, dev, True)
        bt, cq, ck = _to_dev(p.block_tables, dev), _to_dev(p.cu_seqlens_q, dev), _to_dev(p.cu_seqlens_k, dev)
        slots = pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q)
        pa.store_kvcache(_to_dev(p.new_k, dev, True), _to_dev(p.new_v, dev, True), kc, vc, slots)
        out = torch.empty(p.total_q, p.num_q_heads, p.head_dim, dtype=torch.bfloat16, device=dev)
        mq, mk = int(p.seqlens_q.max()), int(p.seqlens_k.max())
        for _ in range(args.warmup + args.steps):
            flush()
            pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out)
        torch.cuda.synchronize()
        _check_device(pa)
        print(f"profile case: prefill, {p.total_q} query tokens, {args.warmup + args.steps} launches")
        return 0
    if args.profile_case == "decode-small":
        rng = np.random.default_rng(1002)
        inp = make_decode("qwen3-0.6b decode b64 h16/8 ctx~U[1,1536]", 2, 64, 16, 8, rng.integers(1, 1537, size=64))
    elif args.profile_case == "decode-shared-small":
        rng = np.random.default_rng(1003)
        ctx = np.clip(np.round(1024.0 * np.exp(rng.standard_normal(64))), 1, 8192).astype(np.int64)
        ctx[:32] = np.maximum(ctx[:32], 4 * 256 + 1)
        inp = make_decode("qwen3-8b shape b64 h32/8 ctx~lognormal(1024) 32 seqs share 4 blocks", 3, 64, 32, 8, ctx,
                          shared_prefix_seqs=32, shared_prefix_blocks=4)
    else:
        inp = decode_config(HEADLINE_CONFIG)
    kc, vc, q = _to_dev(inp.k_cache, dev, True), _to_dev(inp.v_cache, dev, True), _to_dev(inp.q, dev, True)
    nk, nv = _to_dev(inp.new_k, dev, True), _to_dev(inp.new_v, dev, True)
    bt, ctx = _to_dev(inp.block_tables, dev), _to_dev(inp.context_lens, dev)
    out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
    shared = args.profile_case in ("decode-qwen3-8b", "decode-shared-small")  # shared prefix grouped
    wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev, shared_prefix=shared)
    for _ in range(args.warmup + args.steps):
        flush()
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv, shared_prefix=shared)
    torch.cuda.synchronize()
    _check_device(pa)
    print(f"profile case: {inp.name}: {inp.batch} seqs, {int(inp.context_lens.sum())} context tokens, "
          f"{args.warmup + args.steps} fused decode launches")
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sustain-s", type=float, default=1.5,
                    help="seconds of back-to-back flushed steps run under the clock sampler before the timed steps")
    ap.add_argument("--clock-log", default=None, help="keep the nvidia-smi clock samples in this CSV file")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--report", action="store_true",
                    help="print the per-configuration results table (markdown) instead of the JSON line")
    ap.add_argument("--profile-case", choices=["decode-small", "decode-qwen3-8b", "decode-shared-small", "prefill"],
                    default=None,
                    help="run only a small launch sequence for an ncu capture (no JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_case:
        return run_profile_case(args)
    if args.report:
        return run_report(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
