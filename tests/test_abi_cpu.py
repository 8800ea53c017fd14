"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
the header declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from sparse_mla_attention_03_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from sparse_mla_attention_03_gb300 import build
        build.build()
    return binding.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "sparse_mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sparse_mla_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert len(names) >= 8, names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.SYMBOLS), (set(names) ^ set(binding.SYMBOLS))


def _c_layout(struct, fields):
    """sizeof and offsetof of a header struct, from a C program built with gcc."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    body = "".join(f'  printf("%zu\\n", offsetof({struct}, {f}));\n' for f in fields)
    src = (f"#include <stddef.h>\n#include <stdio.h>\n#include \"sparse_mla.h\"\n"
           f"int main(void) {{\n  printf(\"%zu\\n\", sizeof({struct}));\n{body}  return 0;\n}}\n")
    with tempfile.TemporaryDirectory() as d:
        c, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(c, "w") as f:
            f.write(src)
        subprocess.run([cc, "-I", inc, c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()]
    return vals[0], dict(zip(fields, vals[1:]))


@pytest.mark.parametrize("ctype,struct", [(binding.SmlaArgs, "smla_args"), (binding.SmlaExtraArgs, "smla_extra_args")])
def test_struct_layout_matches_header(ctype, struct):
    fields = [f for f, _ in ctype._fields_]
    size, offs = _c_layout(struct, fields)
    assert ctypes.sizeof(ctype) == size
    for f in fields:
        assert getattr(ctype, f).offset == offs[f], f


def _args(**kw):
    a = binding.SmlaArgs()
    a.q, a.q_stride_t = 0x1000, 8 * 576
    a.kv, a.num_pages = 0x2000, 4
    a.topk, a.indices, a.idx_stride_t = 64, 0x3000, 64
    a.sm_scale, a.T, a.H = 0.04, 4, 8
    a.out, a.out_stride_t = 0x4000, 8 * 512
    a.lse, a.lse_stride_t = 0x5000, 8
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("bad", [
    dict(H=0), dict(H=129), dict(topk=0), dict(T=-1), dict(q_stride_t=100), dict(out_stride_t=8 * 512 + 2),
    dict(lse_stride_t=4), dict(idx_stride_t=10), dict(q=0), dict(kv=0x2001), dict(out=0x4002),
    dict(kv_format=2), dict(layout=2), dict(reserved1=1), dict(sm_scale=float("nan")), dict(num_pages=-1),
    dict(block_table=0x6000, bt_rows=1, bt_cols=8, bt_stride=8, tokens_per_req=2),  # 2 tokens/row x 1 row < 4
    dict(block_table=0x6000, bt_rows=4, bt_cols=8, bt_stride=4, tokens_per_req=1),  # stride < cols
])
def test_invalid_arguments_rejected_without_cuda(lib, bad):
    a = _args(**bad)
    rc = lib.sparse_mla_prefill(ctypes.byref(a), None)
    assert rc == binding.SMLA_ERR_INVALID
    assert lib.sparse_mla_last_error().decode()
    rc = lib.sparse_mla_decode(ctypes.byref(a), 0, None, 0, None)
    assert rc == binding.SMLA_ERR_INVALID


def test_zero_tokens_is_a_no_op(lib):
    a = _args(T=0, q=0, out=0, lse=0, indices=0)
    assert lib.sparse_mla_prefill(ctypes.byref(a), None) == binding.SMLA_OK
    assert lib.sparse_mla_decode(ctypes.byref(a), 0, None, 0, None) == binding.SMLA_OK
    assert lib.sparse_mla_decode_workspace_size(0, 8, 64, 0) == 0


def test_null_args_and_bad_splits(lib):
    assert lib.sparse_mla_prefill(None, None) == binding.SMLA_ERR_INVALID
    a = _args()
    assert lib.sparse_mla_decode(ctypes.byref(a), 65, None, 0, None) == binding.SMLA_ERR_INVALID
    assert lib.sparse_mla_decode(ctypes.byref(a), -1, None, 0, None) == binding.SMLA_ERR_INVALID


def test_explicit_split_arithmetic(lib):
    # explicit splits need no device: effective count never exceeds the 64-slot chunks
    assert lib.sparse_mla_decode_num_splits(128, 64, 2048, 8) == 8
    assert lib.sparse_mla_decode_num_splits(128, 64, 2048, 64) == 32
    assert lib.sparse_mla_decode_num_splits(4, 8, 100, 3) == 2
    assert lib.sparse_mla_decode_num_splits(4, 8, 640, 3) == 3
    ws = lib.sparse_mla_decode_workspace_size(128, 64, 2048, 8)
    assert ws == 128 * 64 * 8 * 512 * 4 + 128 * 64 * 8 * 4
    assert lib.sparse_mla_abi_version() == 5


# Split choice for a described device (host only).  The wave model alone picks
# these counts at 152 SMs (they match measured split sweeps on GB300); the
# L2-footprint guard only acts when a token's rows are gathered by more than
# one CTA (H=128 on the tcgen05 kernel, H=24 on the 8-head warp-MMA kernel).
L2_GB300 = 126_500_000


@pytest.mark.parametrize("T,H,topk,want", [
    (8, 64, 2048, 16), (32, 64, 2048, 4), (64, 64, 2048, 2), (128, 64, 2048, 1), (256, 64, 2048, 1),
    (32, 128, 2048, 2), (16, 64, 8192, 8), (64, 64, 512, 2), (8, 8, 4096, 32), (32, 8, 2048, 16),
    (128, 8, 2048, 4), (512, 8, 1024, 1), (64, 16, 2048, 4), (16, 24, 2048, 8), (256, 8, 640, 2),
])
def test_wave_model_picks(lib, T, H, topk, want):
    assert lib.sparse_mla_plan_num_splits(T, H, topk, 0, 152, L2_GB300) == want
    assert lib.sparse_mla_plan_num_splits(T, H, topk, 0, 152, 0) == want  # no L2 figure: guard off


def test_l2_footprint_guard():
    lib = binding.load()
    plan = lambda T, H, topk, l2: lib.sparse_mla_plan_num_splits(T, H, topk, 0, 152, l2)
    chunk = 64 * 656
    # one CTA per token (H=64): no row is read twice, the guard never acts
    assert plan(128, 64, 3200, L2_GB300) == plan(128, 64, 3200, 10 ** 15) == 1
    assert plan(128, 64, 3200, 1) == 1
    # H=128, T=64, topk 2048: the two head-group CTAs of a token read its rows
    # side by side (span 2 at one split): 2 x 32 chunks of rows, far inside
    # GB300's L2, so the wave model's pick (one split) stands
    assert plan(64, 128, 2048, L2_GB300) == plan(64, 128, 2048, 10 ** 15) == 1
    # with an L2 smaller than that footprint the guard moves to the cheapest
    # count that fits: S=2 streams 3 CTAs x 16 chunks between the reads
    assert 2 * 32 * chunk > 3 * 16 * chunk
    assert plan(64, 128, 2048, 3 * 16 * chunk) == 2
    assert plan(64, 128, 2048, 5 * 8 * chunk) == 4
    # and falls back to the unconstrained pick when nothing fits
    assert plan(64, 128, 2048, 1) == 1
    # an explicit count is never changed by the guard
    assert lib.sparse_mla_plan_num_splits(64, 128, 2048, 1, 152, 1) == 1
    # invalid descriptions
    assert lib.sparse_mla_plan_num_splits(64, 128, 2048, 0, 0, L2_GB300) == 0
    assert lib.sparse_mla_plan_num_splits(64, 128, 2048, 0, 152, -1) == 0


def test_noalloc_scratch_size_matches_header(lib):
    src = open(os.path.join(ROOT, "include", "sparse_mla.h")).read()
    m = re.search(r"#define SMLA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    assert m
    assert binding.noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_wait_limit_setter_round_trips(lib):
    prev = binding.set_wait_limit_ns(12345)
    try:
        assert prev == 1_000_000_000
        assert binding.set_wait_limit_ns(0) == 12345
    finally:
        binding.set_wait_limit_ns(prev)
    assert binding.set_wait_limit_ns(prev) == prev


def test_test_stall_setter_round_trips(lib):
    assert binding.set_test_stall(True) is False
    try:
        assert binding.set_test_stall(True) is True
    finally:
        binding.set_test_stall(False)
    assert binding.set_test_stall(False) is False


# ----------------------------------------------------------------------------- bench helpers (host logic)
def test_bench_traffic_record_tracks_kernel_sources(tmp_path, monkeypatch):
    import json
    import bench
    src = tmp_path / "k.cu"
    src.write_text("// a comment\n__global__ void k() { int x = 1; }  // trailing\n")
    rec = {"w": {"dram_bytes_per_launch": 123, "sources": [str(src)], "capture": "c.md"}}
    import hashlib
    h = hashlib.sha256(bench._code_only(src.read_text()).encode()).hexdigest()
    rec["w"]["sources_sha256"] = h
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.dram_traffic("w") == (123, "c.md")
    assert bench.dram_traffic("other") == (None, None)
    # a comment edit keeps the record, a code edit drops it
    src.write_text("// another comment\n__global__ void k() { int x = 1; }\n")
    assert bench.dram_traffic("w") == (123, "c.md")
    src.write_text("__global__ void k() { int x = 2; }\n")
    assert bench.dram_traffic("w")[0] is None


def test_bench_counts_valid_slots_of_both_lists():
    import bench
    from sparse_mla_attention_03_gb300 import inputs
    wl = inputs.make_dual_prefill("vs", T=3, H=8, ctx=256, topk=70, extra_ctx=128, extra_topk=40, seed=5,
                                  ragged=True)
    want = int(wl.topk_length.clamp(0, 70).sum()) + int(wl.extra_topk_length.clamp(0, 40).sum())
    assert bench.valid_slots(wl) == want
    w = bench.work_of(wl)
    assert w["flops"] == 2.0 * 8 * (576 + 512) * want and w["gather_bytes"] == want * 656


def test_bench_roofline_entries():
    import bench
    peaks = dict(hbm=6000.0, tflops=2000.0, tflops_sus=1800.0, src="measured")
    work = dict(flops=2.0e12, bytes=3.0e9, valid=1)
    # tensor-bound: algorithmic flops over the time, against the bf16 peak
    r = bench.roofline_of("tensor", work, 2.0, peaks, "no-such-workload")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == 1000.0 and r["frac"] == 0.5 and r["traffic"] is None
    # HBM-bound: algorithmic bytes over the time, labelled as such
    r = bench.roofline_of("hbm", work, 1.0, peaks, "no-such-workload")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] == 3000.0 and r["frac"] == 0.5
    assert "algorithmic" in r["achieved_kind"]
    # the DRAM rate counts every launch of the step
    import json
    rec_dir = os.path.join(str(bench.ROOT), "profiles")
    traffic, _ = bench.dram_traffic("prefill16k")
    if traffic is not None:
        r2 = bench.roofline_of("tensor", work, 1.0, peaks, "prefill16k", launches=2)
        assert r2["dram_gbs"] == round(traffic * 2 / 1e-3 / 1e9, 1)
    # every workload timed beside the headline is a bench workload
    assert set(bench.PER_CONFIG) <= set(bench.workloads())
