#!/usr/bin/env python3
"""Benchmark of the sparse MLA forward on GB300 (one JSON line on rank 0).

Default workload: prefill at the 16k footprint -- T=1024 query tokens, H=64,
context 16384 (256 pages of 64 rows, 656-byte FP8 rows), topk 512 then 1024
unique indices per query row, per-head sinks, bf16 q.  One step runs the
whole hot path over that batch at both widths (two prefill launches).
``--workload`` selects the other workloads (few-head, decode, large) for
profiling; their numbers go to the same JSON format.

value: query tokens processed per second (each width counts its 1024 tokens),
device-timed with CUDA events around the launches, inputs resident in HBM,
L2 flushed (256 MiB write) between steps.  e2e: the same through the public
API from pinned host buffers with the H2D copy of q/indices and the D2H copy
of out/lse inside the timed region.  cpu_baseline / --impl reference: the
CPU oracle on a bounded sample of tokens on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA query-tokens/s at 1 GB300; % of roofline (tensor-core or HBM)"
UNIT = "query-tokens/s"
ROW = 656


def workloads(tokens=None):
    """The benchmark workloads.  ``tokens`` shrinks the query-token count of a
    prefill workload (for a small profiling case of the same kernel)."""
    from sparse_mla_attention_03_gb300 import inputs
    T16 = tokens or 1024
    TF = tokens or 8192
    TL = tokens or 4096
    return {
        "prefill16k": dict(name=f"prefill_T{T16}_H64_ctx16384_k512+k1024", kind="prefill", bound="tensor",
                           parts=[("k512", lambda s: inputs.prefill_16k(512, seed=s, T=T16)),
                                  ("k1024", lambda s: inputs.prefill_16k(1024, seed=s, T=T16))]),
        "fewhead": dict(name=f"fewhead_prefill_T{TF}_H8_ctx32768_k640_ld1024_ragged", kind="prefill",
                        bound="hbm", parts=[("all", lambda s: inputs.fewhead_prefill(seed=s, T=TF))]),
        "decode": dict(name="decode_64req_x2_H64_ctx32768_k2048_paged", kind="decode", bound="hbm",
                       parts=[("all", lambda s: inputs.batched_decode(seed=s))]),
        "large": dict(name=f"large_prefill_T{TL}_H128_ctx131072_k2048_neg0.1", kind="prefill", bound="tensor",
                      parts=[("all", lambda s: inputs.large_prefill(seed=s, T=TL))]),
        "tiny": dict(name="tiny_prefill_T4_H8_ctx256_k64", kind="prefill", bound="hbm",
                     parts=[("all", lambda s: inputs.tiny_prefill(seed=s))]),
        "dual_decode": dict(name="dual_decode_64req_x2_H64_ctx32768_k1024+ctx8192_k2176_paged", kind="dual_decode",
                            bound="hbm", parts=[("all", lambda s: inputs.dual_decode(seed=s))]),
        "prefill16k_int8": dict(name=f"prefill_T{T16}_H64_ctx16384_k1024_int8", kind="prefill", bound="tensor",
                                parts=[("k1024", lambda s: inputs.prefill_16k_int8(1024, seed=s, T=T16))]),
    }


def _valid_in_list(indices, topk, topk_length, num_pages, block_table):
    import numpy as np
    idx = indices.numpy()[:, :topk].astype(np.int64)
    T = idx.shape[0]
    lens = np.full(T, topk) if topk_length is None else np.clip(topk_length.numpy(), 0, topk)
    inlen = np.arange(topk)[None, :] < lens[:, None]
    if block_table is None:
        ok = inlen & (idx >= 0) & (idx < num_pages * 64)
    else:
        ok = inlen & (idx >= 0) & (idx // 64 < block_table.shape[1])
    return int(ok.sum())


def valid_slots(wl):
    """Number of valid (token, slot) pairs: the units the algorithmic work counts
    (both lists of the dual-cache form)."""
    v = _valid_in_list(wl.indices, wl.topk, wl.topk_length, wl.num_pages, wl.block_table)
    if wl.dual:
        v += _valid_in_list(wl.extra_indices, wl.extra_topk, wl.extra_topk_length, wl.extra_kv.shape[0],
                            wl.extra_block_table)
    return v


def work_of(wl):
    v = valid_slots(wl)
    T, H = wl.T, wl.H
    flops = 2.0 * H * (576 + 512) * v
    gather = v * ROW
    io = T * H * (576 * 2 + 512 * 2 + 4) + T * (wl.topk + wl.extra_topk) * 4
    return dict(valid=v, flops=flops, bytes=gather + io, gather_bytes=gather)


def dram_traffic(workload):
    """DRAM bytes per launch of the attention kernel from a committed ncu capture
    (profiles/dram_traffic.json), or None when there is none for this workload or
    the kernel sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        rec = json.load(f).get(workload)
    if not rec:
        return None, None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src)) as f:
            h.update(_code_only(f.read()).encode())
    if h.hexdigest() != rec["sources_sha256"]:
        return None, "kernel changed since the capture"
    return rec["dram_bytes_per_launch"], rec["capture"]


def _code_only(src):
    """C++ source without comments, trailing blanks and empty lines: the text
    the kernel's code depends on (comment edits keep a capture valid)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.split("\n") if line.strip())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], tflops=d["bf16_tflops"], tflops_sus=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, tflops=1900.0, tflops_sus=1700.0, src="fallback")


# ------------------------------------------------------------------------------------------ oracle
def _oracle_chunk(args):
    import numpy as np
    import oracle.sparse_mla_oracle as O
    (q, kv, idx, topk, sm, tl, sink, bt, tpr, toks, extra, fmt, layout) = args
    if extra is None:
        O.sparse_mla_forward(q, kv, idx, topk, sm, topk_length=tl, attn_sink=sink, block_table=bt,
                             tokens_per_req=tpr, tokens=toks, q_selected=True, kv_format=fmt, layout=layout)
    else:
        kv2, idx2, topk2, tl2, bt2 = extra
        O.sparse_mla_forward_dual(q, kv, idx, topk, kv2, idx2, topk2, sm, topk_length=tl, extra_topk_length=tl2,
                                  attn_sink=sink, block_table=bt, extra_block_table=bt2, tokens_per_req=tpr,
                                  tokens=toks, q_selected=True, kv_format=fmt, layout=layout)
    return len(toks)


def oracle_time(wl, n_tokens, cores, pool=None):
    """Oracle wall time on n_tokens tokens spread over `cores` spawn processes
    (a pool of them is made here unless one is passed in)."""
    import numpy as np
    import torch
    toks = np.arange(min(n_tokens, wl.T))
    chunks = [c for c in np.array_split(toks, cores) if len(c)]
    kv = wl.kv.numpy()
    idx = wl.indices.numpy()
    tl = None if wl.topk_length is None else wl.topk_length.numpy()
    sink = None if wl.attn_sink is None else wl.attn_sink.numpy().astype(np.float64)
    bt = None if wl.block_table is None else wl.block_table.numpy()
    np_ = lambda x: None if x is None else x.numpy()
    extra = (wl.extra_kv.numpy(), wl.extra_indices.numpy(), wl.extra_topk, np_(wl.extra_topk_length),
             np_(wl.extra_block_table)) if wl.dual else None
    jobs = [(wl.q[torch.as_tensor(c)].to(torch.float64).numpy(), kv, idx, wl.topk, wl.sm_scale, tl, sink, bt,
             wl.tokens_per_req, c, extra, wl.kv_format, wl.layout) for c in chunks]
    own = pool is None
    if own:
        pool = mp.get_context("spawn").Pool(cores, initializer=_pin_threads)
    try:
        pool.map(_oracle_chunk, jobs[:1])  # warm the workers' imports
        t0 = time.perf_counter()
        n = sum(pool.map(_oracle_chunk, jobs))
        dt = time.perf_counter() - t0
    finally:
        if own:
            pool.close()
            pool.join()
    return n, dt


def _pin_threads():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        self.path = os.path.join(tempfile.gettempdir(), f"smla_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------------------------------------------ ranks
def rank_seed(seed, rank):
    """Each rank draws its own batch of the workload (weak scaling: no shared data, no collective)."""
    return seed + 1000003 * rank


def global_elapsed_ms(local_ms, world, device=None):
    """The job's time is the slowest rank's: max over ranks (a timing-only all-reduce)."""
    if world <= 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step, steps, world, elapsed_ms):
    """Whole-job query tokens per second: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / (elapsed_ms / 1e3)


# ------------------------------------------------------------------------------------------ runs
def make_call(kind, binding, d, wl, out, lse, ws, num_splits):
    if kind == "prefill":
        def call(stream=None):
            binding.sparse_mla_prefill(d["q"], d["kv"], d["indices"], wl.sm_scale, topk=wl.topk,
                                       topk_length=d["topk_length"], attn_sink=d["attn_sink"],
                                       block_table=d["block_table"], tokens_per_req=wl.tokens_per_req,
                                       out=out, lse=lse, stream=stream, kv_format=wl.kv_format, layout=wl.layout)
    elif kind == "decode":
        def call(stream=None):
            binding.sparse_mla_decode(d["q"], d["kv"], d["indices"], wl.sm_scale, topk=wl.topk,
                                      topk_length=d["topk_length"], attn_sink=d["attn_sink"],
                                      block_table=d["block_table"], tokens_per_req=wl.tokens_per_req,
                                      num_splits=num_splits, workspace=ws, out=out, lse=lse, stream=stream,
                                      kv_format=wl.kv_format, layout=wl.layout)
    else:
        def call(stream=None):
            binding.sparse_mla_decode_dual(d["q"], d["kv"], d["indices"], d["extra_kv"], d["extra_indices"],
                                           wl.sm_scale, topk=wl.topk, topk_length=d["topk_length"],
                                           extra_topk=wl.extra_topk, extra_topk_length=d["extra_topk_length"],
                                           attn_sink=d["attn_sink"], block_table=d["block_table"],
                                           extra_block_table=d["extra_block_table"],
                                           tokens_per_req=wl.tokens_per_req, num_splits=num_splits, workspace=ws,
                                           out=out, lse=lse, stream=stream, kv_format=wl.kv_format, layout=wl.layout)
    return call


def run_ours(args, rank, world, local_rank):
    import torch
    from sparse_mla_attention_03_gb300 import binding

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    binding.load()
    spec = workloads(args.tokens)[args.workload]
    peaks = load_peaks()
    parts = []
    for tag, mk in spec["parts"]:
        wl = mk(rank_seed(args.seed, rank))
        d = {k: (None if getattr(wl, k) is None else getattr(wl, k).to(dev))
             for k in ("q", "kv", "indices", "topk_length", "attn_sink", "block_table", "extra_kv",
                       "extra_indices", "extra_topk_length", "extra_block_table")}
        out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device=dev)
        ws = None
        if spec["kind"] != "prefill":
            width = binding.dual_width(wl.topk, wl.extra_topk) if wl.dual else wl.topk
            ws = torch.empty(max(256, binding.decode_workspace_size(wl.T, wl.H, width, args.num_splits)),
                             dtype=torch.uint8, device=dev)
        call = make_call(spec["kind"], binding, d, wl, out, lse, ws, args.num_splits)
        # kernels per call: the attention kernel, plus the combine when decode splits
        launches = 1
        if spec["kind"] != "prefill":
            launches = 1 if binding.decode_num_splits(wl.T, wl.H, width, args.num_splits) == 1 else 2
        parts.append(dict(tag=tag, wl=wl, d=d, out=out, lse=lse, ws=ws, call=call, work=work_of(wl),
                          launches=launches))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        for p in parts:
            p["call"]()
    barrier()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
          for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        barrier()
        t0 = time.perf_counter()
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            for j, p in enumerate(parts):
                ev[s][j][0].record(stream)
                p["call"]()
                ev[s][j][1].record(stream)
        barrier()
        wall = time.perf_counter() - t0
    per_part_ms = [[ev[s][j][0].elapsed_time(ev[s][j][1]) for s in range(args.steps)] for j in range(len(parts))]
    step_ms = [sum(per_part_ms[j][s] for j in range(len(parts))) for s in range(args.steps)]
    total_ms = global_elapsed_ms(sum(step_ms), world, dev)
    tokens_per_step = sum(p["wl"].T for p in parts)
    value = job_throughput(tokens_per_step, args.steps, world, total_ms)

    # roofline of the dominant kernel (the attention kernel; for decode the split kernel dominates)
    flops = sum(p["work"]["flops"] for p in parts)
    nbytes = sum(p["work"]["bytes"] for p in parts)
    avg_step_s = total_ms / args.steps / 1e3
    if spec["bound"] == "tensor":
        achieved = flops / avg_step_s / 1e12
        roof = dict(bound="tensor", achieved=round(achieved, 2), peak=peaks["tflops"], unit="TFLOP/s",
                    frac=round(achieved / peaks["tflops"], 4), traffic=None,
                    peak_source=f"{peaks['src']} bf16 dense burst (fp16 operands run at the same rate)")
    else:
        achieved = nbytes / avg_step_s / 1e9
        roof = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm"], unit="GB/s",
                    frac=round(achieved / peaks["hbm"], 4), traffic=None,
                    peak_source=f"{peaks['src']} HBM copy bandwidth")
    traffic, src = dram_traffic(args.workload)
    if traffic is not None:
        roof["traffic"] = traffic
        roof["traffic_unit"] = "bytes per launch (mean), ncu dram__bytes_read.sum + dram__bytes_write.sum"
    if src is not None:
        roof["traffic_source"] = src
    roof["per_launch"] = {p["tag"]: dict(ms=round(statistics.mean(per_part_ms[j]), 4),
                                         tflops=round(p["work"]["flops"] / (statistics.mean(per_part_ms[j]) / 1e3) / 1e12, 2),
                                         gbs=round(p["work"]["bytes"] / (statistics.mean(per_part_ms[j]) / 1e3) / 1e9, 1))
                          for j, p in enumerate(parts)}

    e2e = run_e2e(args, parts, dev, stream, world)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f16",
        "precision": "fp8 e4m3 cache and bf16 q in; f16 MMA operands with fp32 accumulation; bf16 out, fp32 lse",
        "data": "synthetic (seeded numpy PCG64; no dataset or weights involved)",
        "config": {"workload": spec["name"], "global_batch_tokens": tokens_per_step * world,
                   "parallelism": f"dp{world} (independent token shards, no collective)",
                   "l2": "flushed between steps (256 MiB write)", "seed": args.seed,
                   "num_splits": args.num_splits if spec["kind"] != "prefill" else None},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(p["launches"] for p in parts),
        "clocks": clk.summary(),
        "wall_s": round(wall, 3),
    }
    return line, parts


def run_e2e(args, parts, dev, stream, world):
    """The metric through the public API from pinned host buffers: every step
    copies that step's inputs (q and every index input) host -> device, runs
    the call and copies out and lse device -> host, all inside the timed
    region.  As a caller would, it pipelines the steps over three streams with
    double-buffered device inputs and outputs: the copy-in of step s+1 and the
    copy-out of step s-1 overlap the kernels of step s (events order each
    buffer's reuse)."""
    import torch
    from sparse_mla_attention_03_gb300 import binding
    keys = ("q", "indices", "topk_length", "extra_indices", "extra_topk_length")
    for p in parts:
        wl = p["wl"]
        p["h_in"] = {k: getattr(wl, k).pin_memory() for k in keys if getattr(wl, k) is not None}
        p["h_out"] = (torch.empty(p["out"].shape, dtype=p["out"].dtype).pin_memory(),
                      torch.empty(p["lse"].shape, dtype=p["lse"].dtype).pin_memory())
        p["bufs"] = []
        for _ in range(2):
            d = dict(p["d"])
            for k in p["h_in"]:
                d[k] = torch.empty_like(p["d"][k])
            out, lse = torch.empty_like(p["out"]), torch.empty_like(p["lse"])
            kind = "prefill" if p["ws"] is None else ("dual_decode" if wl.dual else "decode")
            p["bufs"].append((d, out, lse, make_call(kind, binding, d, wl, out, lse, p["ws"], args.num_splits)))
    steps = max(2, min(args.steps, 20))
    h2d = sum(sum(t.numel() * t.element_size() for t in p["h_in"].values()) for p in parts)
    d2h = sum(p["h_out"][0].numel() * 2 + p["h_out"][1].numel() * 4 for p in parts)
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "cmp", "out")}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record(s_in)
    for s in range(steps):
        b = s % 2
        if s >= 2:
            s_in.wait_event(ev["cmp"][b])  # step s-2 no longer reads input buffer b
        with torch.cuda.stream(s_in):
            for p in parts:
                for k, t in p["h_in"].items():
                    p["bufs"][b][0][k].copy_(t, non_blocking=True)
        ev["in"][b].record(s_in)
        s_cmp.wait_event(ev["in"][b])
        if s >= 2:
            s_cmp.wait_event(ev["out"][b])  # step s-2's outputs in buffer b are copied out
        for p in parts:
            p["bufs"][b][3](stream=s_cmp)
        ev["cmp"][b].record(s_cmp)
        s_out.wait_event(ev["cmp"][b])
        with torch.cuda.stream(s_out):
            for p in parts:
                p["h_out"][0].copy_(p["bufs"][b][1], non_blocking=True)
                p["h_out"][1].copy_(p["bufs"][b][2], non_blocking=True)
        ev["out"][b].record(s_out)
    end.record(s_out)
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end)
    tokens = sum(p["wl"].T for p in parts) * steps * world
    return {"value": round(tokens / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelined": "H2D of step s+1 and D2H of step s-1 overlap the kernels of step s (3 streams)"}


def cpu_baseline(parts_or_wls, budget_tokens, min_seconds=10.0, max_passes=12):
    """The oracle timed on the first budget_tokens tokens of each part, repeated
    until about min_seconds of CPU work have been measured (bounded passes)."""
    cores = min(host_cores(), 32)
    n_tot, t_tot, passes = 0, 0.0, 0
    descs = []
    with mp.get_context("spawn").Pool(cores, initializer=_pin_threads) as pool:
        while passes < max_passes and (passes == 0 or t_tot < min_seconds):
            for wl in parts_or_wls:
                n, dt = oracle_time(wl, budget_tokens, cores, pool)
                n_tot += n
                t_tot += dt
                if passes == 0:
                    descs.append(f"{wl.name}: first {n} tokens")
            passes += 1
    return {"value": round(n_tot / t_tot, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "; ".join(descs) + f", {passes} passes (fp64 numpy oracle, {cores} spawn processes, "
                      f"{t_tot:.1f} s)"}


def run_reference(args, seconds=120.0):
    """The CPU oracle as the reference arm.  Each step is a bounded token sample
    of each part: its size is set from a calibration pass so that the timed
    steps take about `seconds` in all, whatever --steps is (one process pool
    serves every step)."""
    spec = workloads(args.tokens)[args.workload]
    wls = [mk(args.seed) for _, mk in spec["parts"]]
    cores = min(host_cores(), 32)
    times, toks = [], 0
    with mp.get_context("spawn").Pool(cores, initializer=_pin_threads) as pool:
        # calibration (also the warm-up): one token per process on each part
        n_cal, t_cal = 0, 0.0
        for wl in wls:
            n, dt = oracle_time(wl, cores, cores, pool)
            n_cal += n
            t_cal += dt
        rate = n_cal / max(t_cal, 1e-9)  # tokens/s over the parts, all processes busy
        per_part = int(rate * seconds / max(1, args.steps) / len(wls))
        per_part = max(1, min(args.ref_tokens, per_part))
        for _ in range(args.steps):
            t = 0.0
            for wl in wls:
                n, dt = oracle_time(wl, per_part, cores, pool)
                t += dt
                toks += n
            times.append(t)
    total = sum(times)
    value = toks / total
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": spec["name"], "sample_tokens_per_part": per_part},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"first {per_part} tokens of each part per step, {args.steps} steps "
                                       f"({total:.1f} s of oracle time)"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["prefill16k", "fewhead", "decode", "large", "tiny", "dual_decode",
                                           "prefill16k_int8"],
                    default="prefill16k")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-tokens", type=int, default=512, help="oracle sample per part for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=128, help="oracle sample per part per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=None,
                    help="query tokens of a prefill workload (smaller profiling case; default: the full workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line, parts = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if args.no_cpu_baseline:
            line["cpu_baseline"] = None
        else:
            line["cpu_baseline"] = cpu_baseline([p["wl"] for p in parts], args.cpu_tokens)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
