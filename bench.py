"""Benchmark of the paged-KV attention hot path on one GB300 (or N replicas).

A step is one decode step of one attention layer on the Qwen3-0.6B-shaped
workload (batch 64, 16 q / 8 kv heads, head_dim 128, block_size 256,
context_lens ~ U{1..4096}, pool sized for all sequences + 20 %, random block
permutation, bf16 N(0,1)):
  1. slot mapping of each sequence's newest token (address translation),
  2. store_kvcache of the 64 new K/V rows,
  3. split-KV GQA decode attention over all context tokens.
All inputs are resident in HBM before the timed region; L2 is flushed (a
256 MiB write) before every timed step.  The printed `value` is decode
tokens/s (one layer) over all ranks; `e2e` is the same metric through the
public API with the step's inputs copied from pinned host memory and the
output copied back inside the timed region.  The decode kernel's own CUDA-
event time gives the HBM roofline fraction.  The CPU oracle, timed on the
host cores on a bounded sample, is reported as `cpu_baseline`.

`--impl reference` runs the CPU oracle (the only reference this path has) on
the same workload and prints its own line.

Multi-GPU (torchrun): every rank serves its own batch of 64 sequences with
its own pool (replicas, weak scaling); no collective is on the data path.
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
WORKLOAD = ("qwen3-0.6b decode step, 1 layer: batch 64, 16 q / 8 kv heads, head_dim 128, block_size 256, "
            "context_lens ~ U[1,4096], pool = 1.2x blocks needed, random block permutation, "
            "store of the new token fused into the split-KV decode kernel (pa_decode_store)")
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


DECODE_SOURCES = ["paged_kv_cache_store_gb300/csrc/pa_decode.cu", "paged_kv_cache_store_gb300/csrc/pa_internal.cuh"]


def recorded_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel, {}).get(workload_key)
    if not rec or rec.get("source_digest") != source_digest(DECODE_SOURCES):
        return None
    return float(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{gpu_index}.csv") \
            if os.path.isdir(os.path.join(ROOT, "gpurun_out")) else f"/tmp/pa_clocks_{os.getpid()}.csv"

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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                c = [x.strip() for x in ln.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    mx.append(float(c[2]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


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


def time_oracle_step(inp, O, budget_s: float):
    """Runs the oracle's step (slot mapping, store, decode) on the workload for
    about budget_s seconds; returns (tokens/s, steps)."""
    steps, t0 = 0, time.perf_counter()
    while True:
        kc, vc = inp.k_cache.copy(), inp.v_cache.copy()
        slots = np.array([O.decode_slot(inp.block_tables[b], inp.block_size, int(inp.context_lens[b]))
                          for b in range(inp.batch)], np.int32)
        O.store_kvcache(inp.new_k, inp.new_v, kc, vc, slots)
        O.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return steps * inp.batch / el, steps, el


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as O
    from paged_kv_cache_store_gb300.workloads import decode_config
    inp = decode_config(2)
    O.lib()
    for _ in range(args.warmup):
        time_oracle_step(inp, O, 0.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle_step(inp, O, 0.0)
    el = time.perf_counter() - t0
    value = args.steps * inp.batch / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": WORKLOAD, "global_batch": inp.batch, "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"full workload, {args.steps} steps"},
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


def measure_prefill(args, dev, stream, flush, bf16_peak):
    """The varlen prefill workload: slot mapping + store of the uncached suffix,
    then causal prefill over the paged pool.  Returns a JSON-able dict."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import prefill_config

    p = prefill_config(5)

    def to_dev(a, bf=False):
        if bf:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    kc, vc = to_dev(p.k_cache, True), to_dev(p.v_cache, True)
    q, nk, nv = to_dev(p.q, True), to_dev(p.new_k, True), to_dev(p.new_v, True)
    bt, cq, ck = to_dev(p.block_tables), to_dev(p.cu_seqlens_q), to_dev(p.cu_seqlens_k)
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
        flush.zero_()
        step(e)
    torch.cuda.synchronize()
    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")
    pre_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)
    step3_ms = sum(e[0].elapsed_time(e[2]) for e in evs) / len(evs)
    # The same step as one launch: the fused store + prefill (cooperative).
    wsf = pa.prefill_store_workspace(dev)

    def fused():
        pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out, new_k=nk, new_v=nv,
                          workspace=wsf)

    for _ in range(3):
        fused()
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a_, b_ in fev:
        flush.zero_()
        a_.record(stream)
        fused()
        b_.record(stream)
    torch.cuda.synchronize()
    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")
    fused_ms = sum(a_.elapsed_time(b_) for a_, b_ in fev) / len(fev)
    slotmap_store_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    store_ms = sum(e[3].elapsed_time(e[1]) for e in evs) / len(evs)
    flops = 4 * p.head_dim * p.num_q_heads * prefill_pairs(p)
    tflops = flops / (pre_ms / 1000.0) / 1e12
    store_bytes = p.total_q * p.num_kv_heads * p.head_dim * 2 * 4
    del kc, vc
    return {"workload": "varlen causal prefill, 16 seqs, 32 q / 8 kv heads, Lk ~ U[128,2048], 0..3 cached "
                        "blocks per seq, block_size 256 (suffix stored via slot_mapping first)",
            "total_q": p.total_q, "ms_prefill": pre_ms, "ms_slotmap_store": slotmap_store_ms, "ms_store": store_ms,
            "ms_step_3_launches": step3_ms, "ms_step_fused": fused_ms,
            "algorithmic_flops": flops,
            "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": tflops, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": tflops / bf16_peak, "traffic": None},
            "store_gbs": store_bytes / (store_ms / 1000.0) / 1e9}


def measure_sampler(args, dev, stream, flush, hbm_peak):
    """The Gumbel-max sampler after the decode step: 64 rows over the Qwen3
    vocabulary (bf16 logits, fp32 Exp(1) draws).  HBM-bound: every logit and
    draw is read once."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import sampler_config

    sp = sampler_config(64)
    lg = torch.from_numpy(np.ascontiguousarray(sp.logits).view(np.int16)).view(torch.bfloat16).to(dev)
    temps = torch.from_numpy(sp.temperatures).to(dev)
    noise = torch.from_numpy(sp.exp_noise).to(dev)
    out = torch.empty(sp.batch, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        pa.sample_gumbel(lg, temps, noise, out=out)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        pa.sample_gumbel(lg, temps, noise, out=out)
        b.record(stream)
    torch.cuda.synchronize()
    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    alg = sp.batch * sp.vocab * (2 + 4) + sp.batch * (4 + 4)
    gbs = alg / (ms / 1000.0) / 1e9
    return {"workload": sp.name + ", fp32 Exp(1) draws", "ms": ms, "algorithmic_bytes": alg,
            "roofline": {"bound": "hbm", "kernel": "sample_gumbel_kernel", "achieved": gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": gbs / hbm_peak, "traffic": None},
            "l2": "flushed (256 MiB write) before every timed call; inputs 58 MB"}


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
    inp = decode_config(2)

    def to_dev(a, dt):
        if dt == torch.bfloat16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    kc, vc = to_dev(inp.k_cache, torch.bfloat16), to_dev(inp.v_cache, torch.bfloat16)
    q = to_dev(inp.q, torch.bfloat16)
    nk, nv = to_dev(inp.new_k, torch.bfloat16), to_dev(inp.new_v, torch.bfloat16)
    bt, ctx = to_dev(inp.block_tables, torch.int32), to_dev(inp.context_lens, torch.int32)
    slots = torch.empty(inp.batch, dtype=torch.int32, device=dev)
    out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
    wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    L2 = "flushed (256 MiB write) before every timed step; KV pool 621 MiB > L2"

    def step():  # one kernel: the decode kernel stores the new K/V rows, then attends
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv)

    def step_unfused():  # the same work as three launches
        pa.slot_mapping_decode(bt, ctx, inp.block_size, out=slots)
        pa.store_kvcache(nk, nv, kc, vc, slots)
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out)

    for _ in range(max(3, args.warmup)):
        step()
        step_unfused()
    torch.cuda.synchronize()
    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")

    # Headline: whole steps, L2 flushed before each.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dev, ws)
    ms_per_step = total_ms / args.steps
    value = job_throughput(ws, inp.batch, args.steps, total_ms)

    # The same step as three launches (slot mapping, store, decode: programmatic
    # dependent launches back to back), for comparison.
    uev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in uev:
        flush.zero_()
        a.record(stream)
        step_unfused()
        b.record(stream)
    torch.cuda.synchronize()
    unfused_ms = sum(a.elapsed_time(b) for a, b in uev) / args.steps

    # Per-kernel durations for the roofline: events around the store and the
    # decode launch of the unfused step (same inputs, L2 flushed before each).
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
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
            flush.zero_()
            e2e_ev[i - 2][0].record(stream)
        d_pack.copy_(h_pack, non_blocking=True)
        pa.decode(e_q, kc, vc, e_bt, e_ctx, inp.scale, workspace=wsp, out=out, new_k=e_nk, new_v=e_nv)
        h_out.copy_(out, non_blocking=True)
        if i >= 2:
            e2e_ev[i - 2][1].record(stream)
    torch.cuda.synchronize()
    if not np.array_equal(h_out.view(torch.int16).numpy(), out.cpu().view(torch.int16).numpy()):
        raise RuntimeError("end-to-end output differs from the device output")
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), dev, ws)
    e2e_value = job_throughput(ws, inp.batch, args.steps, e2e_ms)

    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")
    prefill = None
    if not args.no_prefill:
        del kc, vc
        torch.cuda.empty_cache()
        prefill = measure_prefill(args, dev, stream, flush, peaks()[1])
    sampler = measure_sampler(args, dev, stream, flush, peaks()[0])

    if rank == 0:
        hbm, _, peak_kind = peaks()
        kv_bytes = int(inp.context_lens.astype(np.int64).sum()) * inp.num_kv_heads * inp.head_dim * 2 * 2
        qo_bytes = 2 * inp.batch * inp.num_q_heads * inp.head_dim * 2
        # The headline step is one launch of the fused kernel: it reads every
        # context token's K/V row once, q, and the new rows, and writes out and
        # the new rows' slots.
        new_row_bytes = inp.batch * inp.num_kv_heads * inp.head_dim * 2 * 2
        alg_bytes = kv_bytes + qo_bytes + 2 * new_row_bytes
        dec_avg = sum(dec_ms) / len(dec_ms)
        achieved = alg_bytes / (ms_per_step / 1000.0) / 1e9
        traffic = recorded_traffic("decode_kernel<2, store>", "qwen3-0.6b")
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic (seeded N(0,1) bf16, random block tables)",
            "config": {"workload": WORKLOAD, "global_batch": inp.batch * ws, "seq_len": "U[1,4096]",
                       "parallelism": f"replicas x{ws}", "l2": L2},
            "roofline": {"bound": "hbm", "kernel": "decode_kernel<2, store> (pa_decode_store)", "achieved": achieved,
                         "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "peak_kind": peak_kind,
                         "frac_of_nominal_8TBps": achieved / 8000.0, "traffic": traffic,
                         "algorithmic_bytes_per_launch": alg_bytes, "launch_ms": ms_per_step,
                         "plain_decode_ms": dec_avg, "store_ms": sum(store_ms) / len(store_ms)},
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "unfused_step": {"ms_per_step": unfused_ms, "kernels": "slot_mapping_decode + store_kvcache + decode",
                             "tokens_per_s": ws * inp.batch / (unfused_ms / 1000.0)},
            "clocks": clk.summary(),
            "prefill": prefill,
            "sampler": sampler,
        }
        if not args.no_cpu_baseline:
            import oracle as O
            O.lib()
            tps, steps, el = time_oracle_step(inp, O, args.cpu_seconds)
            line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                    "sample": f"{steps} full steps of the same workload ({el:.1f} s, 1 thread)"}
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
    the oracle on the same inputs (all outputs for decode; 2048 sampled
    (token, head) rows for prefill).  Oracle time: one single-threaded oracle
    step (for prefill, the sampled rows, extrapolated by their share of the
    visible (query, key) pairs)."""
    import torch
    import oracle as O
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import decode_config, prefill_config, bf16_bits_to_f32
    O.lib()
    dev = torch.device("cuda", 0)
    hbm, bf16_peak, kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def to(a, bf=False):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf else np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if bf else t).to(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a_, b_ in ev:
            flush.zero_()
            a_.record()
            fn()
            b_.record()
        torch.cuda.synchronize()
        code, where = pa.get_device_error()
        if code:
            raise RuntimeError(f"device error {code} at {where}")
        return float(np.median([a_.elapsed_time(b_) for a_, b_ in ev]))

    def host(t):
        return bf16_bits_to_f32(t.cpu().view(torch.int16).numpy().view(np.uint16)).astype(np.float64)

    traffic = recorded_traffic("decode_kernel<2, store>", "qwen3-0.6b")
    lines = ["| Config | GPU time | tokens/s (decode, 1 layer) | GB/s (algorithmic) | TFLOP/s | % roofline "
             "| ncu DRAM GB/s | Oracle 1-thread | Parity (max / mean abs) |", "|" + "---|" * 9]
    for cfg in (1, 2, 3, 4):
        inp = decode_config(cfg)
        kc, vc, q = to(inp.k_cache, True), to(inp.v_cache, True), to(inp.q, True)
        nk, nv = to(inp.new_k, True), to(inp.new_v, True)
        bt, ctx = to(inp.block_tables), to(inp.context_lens)
        out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
        wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev)
        ms = timed(lambda: pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv))
        t0 = time.perf_counter()
        okc, ovc = inp.k_cache.copy(), inp.v_cache.copy()
        slots = np.array([O.decode_slot(inp.block_tables[b], inp.block_size, int(inp.context_lens[b]))
                          for b in range(inp.batch)], np.int32)
        O.store_kvcache(inp.new_k, inp.new_v, okc, ovc, slots)
        want = O.decode(inp.q, okc, ovc, inp.block_tables, inp.context_lens, inp.scale)
        oracle_s = time.perf_counter() - t0
        err = np.abs(host(out) - want)
        row = inp.num_kv_heads * inp.head_dim * 2
        alg = int(inp.context_lens.astype(np.int64).sum()) * row * 2 + 2 * inp.batch * inp.num_q_heads * \
            inp.head_dim * 2 + 2 * inp.batch * row * 2
        gbs = alg / (ms / 1000.0) / 1e9
        note = " (logical; shared blocks counted per sequence)" if cfg == 3 else ""
        ncu = f"{traffic / (ms / 1000.0) / 1e9:.0f} ({traffic / 1e6:.1f} MB)" if cfg == 2 and traffic else "—"
        lines.append(f"| {cfg} {inp.name} | {ms * 1000:.1f} us | {inp.batch / (ms / 1000.0):,.0f} | "
                     f"{gbs:,.0f}{note} | — | {100 * gbs / hbm:.1f} % of {hbm:.0f} ({kind}) | {ncu} | "
                     f"{oracle_s:.2f} s ({inp.batch / oracle_s:,.0f} tokens/s) | {err.max():.2e} / {err.mean():.2e} |")
        del kc, vc
        torch.cuda.empty_cache()
    p = prefill_config(5)
    kc, vc, q = to(p.k_cache, True), to(p.v_cache, True), to(p.q, True)
    nk, nv = to(p.new_k, True), to(p.new_v, True)
    bt, cq, ck = to(p.block_tables), to(p.cu_seqlens_q), to(p.cu_seqlens_k)
    out = torch.empty(p.total_q, p.num_q_heads, p.head_dim, dtype=torch.bfloat16, device=dev)
    mq, mk = int(p.seqlens_q.max()), int(p.seqlens_k.max())
    slots = pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q)
    pa.store_kvcache(nk, nv, kc, vc, slots)
    ms = timed(lambda: pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out))
    wsf = pa.prefill_store_workspace(dev)
    ms_fused = timed(lambda: pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt, out=out,
                                               new_k=nk, new_v=nv, workspace=wsf))
    pairs = prefill_pairs(p)
    flops = 4 * p.head_dim * p.num_q_heads * pairs
    okc, ovc = p.k_cache.copy(), p.v_cache.copy()
    oslots = np.concatenate([O.slot_mapping(p.block_tables[s], p.block_size, int(p.seqlens_k[s] - p.seqlens_q[s]),
                                            int(p.seqlens_k[s])) for s in range(p.num_seqs)])
    O.store_kvcache(p.new_k, p.new_v, okc, ovc, oslots)
    rows = np.sort(np.random.default_rng(5).choice(p.total_q * p.num_q_heads, 2048, replace=False))
    t0 = time.perf_counter()
    want = O.prefill(p.q, okc, ovc, p.cu_seqlens_q, p.cu_seqlens_k, p.scale, block_tables=p.block_tables,
                     rows=rows)
    oracle_s = time.perf_counter() - t0
    seq_of = np.searchsorted(p.cu_seqlens_q, rows // p.num_q_heads, side="right") - 1
    keys = (p.seqlens_k - p.seqlens_q)[seq_of] + (rows // p.num_q_heads - p.cu_seqlens_q[seq_of]) + 1
    oracle_full = oracle_s * (pairs * p.num_q_heads) / float(keys.sum())
    err = np.abs(host(out).reshape(-1, p.head_dim)[rows] - want)
    tf = flops / (ms / 1000.0) / 1e12
    lines.append(f"| 5 {p.name} | {ms * 1000:.1f} us (fused store + prefill: {ms_fused * 1000:.1f} us) | — | — | "
                 f"{tf:.0f} | {100 * tf / bf16_peak:.1f} % of {bf16_peak:.0f} ({kind}) | — | "
                 f"~{oracle_full:.0f} s (2048 rows in {oracle_s:.1f} s) | {err.max():.2e} / {err.mean():.2e} |")
    print("\n".join(lines))
    return 0


def run_profile_case(args):
    """A reduced decode workload for captures that replay each launch many
    times (ncu --set full): the Qwen3-0.6B shape (batch 64, 16 q / 8 kv
    heads, fused store) with context lengths ~ U[1, 1536], about 190 MB of
    K/V (more than the 129 MB L2, a fraction of the full case).  Runs
    `warmup` then `steps` fused decode steps with an L2 flush before each."""
    import torch
    import paged_kv_cache_store_gb300 as pa
    from paged_kv_cache_store_gb300.workloads import make_decode
    rng = np.random.default_rng(1002)
    inp = make_decode("qwen3-0.6b decode b64 h16/8 ctx~U[1,1536]", 2, 64, 16, 8, rng.integers(1, 1537, size=64))
    dev = torch.device("cuda", 0)

    def to_dev(a, bf=False):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf else np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if bf else t).to(dev)

    kc, vc, q = to_dev(inp.k_cache, True), to_dev(inp.v_cache, True), to_dev(inp.q, True)
    nk, nv = to_dev(inp.new_k, True), to_dev(inp.new_v, True)
    bt, ctx = to_dev(inp.block_tables), to_dev(inp.context_lens)
    out = torch.empty(inp.batch, inp.num_q_heads, inp.head_dim, dtype=torch.bfloat16, device=dev)
    wsp = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup + args.steps):
        flush.zero_()
        pa.decode(q, kc, vc, bt, ctx, inp.scale, workspace=wsp, out=out, new_k=nk, new_v=nv)
    torch.cuda.synchronize()
    code, where = pa.get_device_error()
    if code:
        raise RuntimeError(f"device error {code} at {where}")
    print(f"profile case: {inp.batch} seqs, {int(inp.context_lens.sum())} context tokens, "
          f"{args.warmup + args.steps} fused decode launches")
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--report", action="store_true",
                    help="print the per-configuration results table (markdown) instead of the JSON line")
    ap.add_argument("--profile-case", choices=["decode-small"], default=None,
                    help="run only a reduced case for a multi-pass ncu capture (no JSON line)")
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
