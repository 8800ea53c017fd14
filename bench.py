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
# The oracle runs in spawn processes that map each workload's arrays from
# files written once (np.memmap, shared page cache): a timed call sends only
# token numbers, so the measured rate is the oracle's, not the cost of
# shipping a cache to every process.
_WORKER = {}


def _worker_init(spec):
    import numpy as np
    for key, fields in spec.items():
        d = {}
        for k, v in fields.items():
            if isinstance(v, tuple) and len(v) == 4 and v[0] == "mmap":
                d[k] = np.memmap(v[1], dtype=v[2], mode="r", shape=v[3])
            else:
                d[k] = v
        _WORKER[key] = d


def _oracle_job(args):
    import numpy as np
    import oracle.sparse_mla_oracle as O
    key, toks = args
    w = _WORKER[key]
    q = np.asarray(w["q"][toks], dtype=np.float64)
    kw = dict(topk_length=w["topk_length"], attn_sink=w["attn_sink"], block_table=w["block_table"],
              tokens_per_req=w["tokens_per_req"], tokens=toks, q_selected=True, kv_format=w["kv_format"],
              layout=w["layout"])
    if w["extra_kv"] is None:
        O.sparse_mla_forward(q, w["kv"], w["indices"], w["topk"], w["sm_scale"], **kw)
    else:
        O.sparse_mla_forward_dual(q, w["kv"], w["indices"], w["topk"], w["extra_kv"], w["extra_indices"],
                                  w["extra_topk"], w["sm_scale"], extra_topk_length=w["extra_topk_length"],
                                  extra_block_table=w["extra_block_table"], **kw)
    return len(toks)


class OraclePool:
    """A pool of `cores` spawn processes holding the given workloads (by name)."""

    def __init__(self, wls, cores):
        import shutil  # noqa: F401  (cleanup in close)
        import numpy as np
        import torch
        self.cores = cores
        self.dir = tempfile.mkdtemp(prefix="smla_oracle_")
        spec = {}
        for wl in wls:
            fields = {}
            for k in ("q", "kv", "indices", "topk_length", "attn_sink", "block_table", "extra_kv", "extra_indices",
                      "extra_topk_length", "extra_block_table"):
                t = getattr(wl, k)
                if t is None:
                    fields[k] = None
                    continue
                a = t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()
                if k == "attn_sink":
                    fields[k] = a.astype(np.float64)
                    continue
                path = os.path.join(self.dir, f"{len(spec)}_{k}.bin")
                a = np.ascontiguousarray(a)
                a.tofile(path)
                fields[k] = ("mmap", path, a.dtype.str, a.shape)
            fields.update(topk=wl.topk, extra_topk=wl.extra_topk, sm_scale=wl.sm_scale,
                          tokens_per_req=wl.tokens_per_req, kv_format=wl.kv_format, layout=wl.layout)
            spec[wl.name] = fields
        self.T = {wl.name: wl.T for wl in wls}
        # one BLAS thread per process: the children read these at start-up,
        # before anything (the unpickled arguments included) loads numpy
        keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        os.environ.update({k: "1" for k in keys})
        try:
            self.pool = mp.get_context("spawn").Pool(cores, initializer=_worker_init, initargs=(spec,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for wl in wls:  # warm the workers' imports and mappings (untimed)
            self.pool.map(_oracle_job, [(wl.name, np.arange(1))] * cores)

    def time(self, name, n_tokens):
        """Oracle wall time on the first n_tokens tokens of workload `name`."""
        import numpy as np
        toks = np.arange(min(n_tokens, self.T[name]))
        jobs = [(name, c) for c in np.array_split(toks, self.cores) if len(c)]
        t0 = time.perf_counter()
        n = sum(self.pool.map(_oracle_job, jobs))
        return n, time.perf_counter() - t0

    def close(self):
        import shutil
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


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


def prepare_parts(spec, seed, dev, num_splits):
    """Device copies, outputs and the call of every part of a workload."""
    import torch
    from sparse_mla_attention_03_gb300 import binding
    parts = []
    for tag, mk in spec["parts"]:
        wl = mk(seed)
        d = {k: (None if getattr(wl, k) is None else getattr(wl, k).to(dev))
             for k in ("q", "kv", "indices", "topk_length", "attn_sink", "block_table", "extra_kv",
                       "extra_indices", "extra_topk_length", "extra_block_table")}
        out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device=dev)
        ws = None
        launches = 1  # kernels per call: the attention kernel, plus the combine when decode splits
        splits = None
        if spec["kind"] != "prefill":
            width = binding.dual_width(wl.topk, wl.extra_topk) if wl.dual else wl.topk
            ws = torch.empty(max(256, binding.decode_workspace_size(wl.T, wl.H, width, num_splits)),
                             dtype=torch.uint8, device=dev)
            splits = binding.decode_num_splits(wl.T, wl.H, width, num_splits)
            launches = 1 if splits == 1 else 2
        call = make_call(spec["kind"], binding, d, wl, out, lse, ws, num_splits)
        parts.append(dict(tag=tag, wl=wl, d=d, out=out, lse=lse, ws=ws, call=call, work=work_of(wl),
                          launches=launches, splits=splits))
    return parts


def time_parts(parts, steps, warmup, flush, stream, barrier):
    """Per-part CUDA-event times (ms) of `steps` timed steps after `warmup`
    untimed ones; the L2 is flushed (a write larger than L2) before each step."""
    import torch
    for _ in range(warmup):
        for p in parts:
            p["call"]()
    barrier()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
          for _ in range(steps)]
    barrier()
    for s in range(steps):
        flush.fill_(s & 0xFF)
        for j, p in enumerate(parts):
            ev[s][j][0].record(stream)
            p["call"]()
            ev[s][j][1].record(stream)
    barrier()
    return [[ev[s][j][0].elapsed_time(ev[s][j][1]) for s in range(steps)] for j in range(len(parts))]


def roofline_of(bound, work, ms, peaks, workload, launches=1):
    """Roofline entry of the attention launches of one step (`launches` of
    them in `ms`): algorithmic flops (tensor-bound paths) or bytes
    (gather/HBM-bound paths) over the measured time, against the measured
    peak; `traffic` is the ncu DRAM bytes per launch when a capture of the
    current kernel sources exists, and `dram_gbs` the DRAM rate it gives."""
    sec = ms / 1e3
    if bound == "tensor":
        achieved = work["flops"] / sec / 1e12
        r = dict(bound="tensor", achieved=round(achieved, 2), peak=peaks["tflops"], unit="TFLOP/s",
                 frac=round(achieved / peaks["tflops"], 4), traffic=None,
                 peak_source=f"{peaks['src']} bf16 dense burst (fp16 operands run at the same rate)")
    else:
        achieved = work["bytes"] / sec / 1e9
        r = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm"], unit="GB/s",
                 frac=round(achieved / peaks["hbm"], 4), traffic=None,
                 peak_source=f"{peaks['src']} HBM copy bandwidth",
                 achieved_kind="algorithmic bytes (gather + q/out/lse/indices) per launch / time")
    traffic, src = dram_traffic(workload)
    if traffic is not None:
        r["traffic"] = traffic
        r["traffic_unit"] = "bytes per launch (mean), ncu dram__bytes_read.sum + dram__bytes_write.sum"
        r["dram_gbs"] = round(traffic * launches / sec / 1e9, 1)
        r["dram_frac"] = round(traffic * launches / sec / 1e9 / peaks["hbm"], 4)
    if src is not None:
        r["traffic_source"] = src
    return r


# The other workloads, timed in the same run and with the same protocol as
# the headline one (rank 0's numbers).
PER_CONFIG = ("fewhead", "decode", "large", "dual_decode", "prefill16k_int8")


def run_per_config(args, dev, stream, barrier, flush, peaks, l2_bytes):
    import torch
    res = {}
    for key in PER_CONFIG:
        if key == args.workload:
            continue
        spec = workloads(None)[key]
        parts = prepare_parts(spec, args.seed, dev, args.num_splits)
        ms_lists = time_parts(parts, max(3, min(args.steps, 50)), args.warmup, flush, stream, barrier)
        ms = sum(statistics.median(m) for m in ms_lists)
        work = {k: sum(p["work"][k] for p in parts) for k in ("flops", "bytes", "valid")}
        tokens = sum(p["wl"].T for p in parts)
        cache = sum(p["wl"].kv.numel() + (p["wl"].extra_kv.numel() if p["wl"].dual else 0) for p in parts)
        e = dict(workload=spec["name"], ms=round(ms, 4), query_tokens_per_s=round(tokens / (ms / 1e3), 1),
                 roofline=roofline_of(spec["bound"], work, ms, peaks, key, launches=len(parts)), cache_bytes=cache,
                 cache_in_l2=bool(cache <= l2_bytes), gpu_launches_per_step=sum(p["launches"] for p in parts))
        if parts[0]["splits"] is not None:
            e["num_splits"] = parts[0]["splits"]
        res[key] = e
        del parts
        torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    from sparse_mla_attention_03_gb300 import binding

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    binding.load()
    spec = workloads(args.tokens)[args.workload]
    peaks = load_peaks()
    parts = prepare_parts(spec, rank_seed(args.seed, rank), dev, args.num_splits)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        per_part_ms = time_parts(parts, args.steps, args.warmup, flush, stream, barrier)
        wall = time.perf_counter() - t0
    step_ms = [sum(per_part_ms[j][s] for j in range(len(parts))) for s in range(args.steps)]
    total_ms = global_elapsed_ms(sum(step_ms), world, dev)
    tokens_per_step = sum(p["wl"].T for p in parts)
    value = job_throughput(tokens_per_step, args.steps, world, total_ms)

    # roofline of the dominant kernel (the attention kernel; for decode the split kernel dominates)
    work = {k: sum(p["work"][k] for p in parts) for k in ("flops", "bytes", "valid")}
    roof = roofline_of(spec["bound"], work, total_ms / args.steps, peaks, args.workload, launches=len(parts))
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
    if not args.no_per_config and rank == 0:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        # rank 0 alone: a local barrier (no collective the other ranks would miss)
        line["per_config"] = run_per_config(args, dev, stream, lambda: torch.cuda.synchronize(dev), flush, peaks,
                                            l2)
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


# One sampling protocol for both CPU numbers (cpu_baseline and the reference
# arm): the oracle on the first ORACLE_SAMPLE tokens of each part per pass,
# spread over the host's cores, passes repeated to a time budget.
ORACLE_SAMPLE = 256


def oracle_rate(wls, seconds, max_passes=50, min_passes=1, pool=None):
    """Tokens/s of the oracle over `wls`, timed pass by pass (one pass = the
    first ORACLE_SAMPLE tokens of every part) until `seconds` of oracle time."""
    cores = min(host_cores(), 32)
    own = pool is None
    if own:
        pool = OraclePool(wls, cores)
    try:
        n_tot, t_tot, passes, per_pass = 0, 0.0, 0, []
        while passes < max_passes and (passes < min_passes or t_tot < seconds):
            t_pass = 0.0
            for wl in wls:
                n, dt = pool.time(wl.name, ORACLE_SAMPLE)
                n_tot += n
                t_pass += dt
            per_pass.append(t_pass)
            t_tot += t_pass
            passes += 1
    finally:
        if own:
            pool.close()
    return dict(value=n_tot / t_tot, cores=cores, passes=passes, seconds=t_tot, per_pass=per_pass,
                tokens_per_pass=sum(min(ORACLE_SAMPLE, wl.T) for wl in wls))


def cpu_baseline(wls, seconds=10.0):
    r = oracle_rate(wls, seconds)
    return {"value": round(r["value"], 2), "unit": UNIT, "cores": r["cores"], "kind": "oracle",
            "sample": f"first {ORACLE_SAMPLE} tokens of each of {', '.join(wl.name for wl in wls)} per pass, "
                      f"{r['passes']} passes (fp64 numpy oracle, {r['cores']} spawn processes, "
                      f"{r['seconds']:.1f} s)"}


def run_reference(args, seconds=60.0):
    """The CPU oracle as the reference arm: each step is one pass of the same
    sample as cpu_baseline (the first ORACLE_SAMPLE tokens of each part),
    after --warmup untimed passes; --steps is capped so that the run stays
    within a few minutes (the line says how many steps ran)."""
    spec = workloads(args.tokens)[args.workload]
    wls = [mk(args.seed) for _, mk in spec["parts"]]
    cores = min(host_cores(), 32)
    with OraclePool(wls, cores) as pool:
        for _ in range(min(args.warmup, 3)):
            for wl in wls:
                pool.time(wl.name, ORACLE_SAMPLE)
        first = oracle_rate(wls, 0.0, max_passes=1, pool=pool)
        steps = max(1, min(args.steps, int(seconds / max(first["seconds"], 1e-6))))
        r = oracle_rate(wls, float("inf"), max_passes=steps - 1, min_passes=steps - 1, pool=pool) \
            if steps > 1 else None
    per_pass = first["per_pass"] + (r["per_pass"] if r else [])
    total = sum(per_pass)
    toks = first["tokens_per_pass"] * len(per_pass)
    value = toks / total
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": args.gpus,
            "steps": len(per_pass), "warmup": args.warmup, "ms_per_step": round(total / len(per_pass) * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64)",
            "config": {"workload": spec["name"], "sample_tokens_per_part": ORACLE_SAMPLE,
                       "steps_requested": args.steps},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"first {ORACLE_SAMPLE} tokens of each part per step, {len(per_pass)} steps "
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
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the selected workload (skip the other workloads' entries)")
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
            line["cpu_baseline"] = cpu_baseline([p["wl"] for p in parts])
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
