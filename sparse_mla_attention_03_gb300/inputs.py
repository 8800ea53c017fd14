"""Seeded synthetic inputs for sparse MLA attention (prefill and decode).

The only module that both the CUDA path's tests/benchmark and the CPU oracle
consume.  It draws random numbers and packs them into the cache row format; it
holds none of the attention arithmetic (no dequantisation, no softmax).

Row format written here (FlashInfer PR #4802 "Refactor Sparse MLA SM120",
review note on the DSv3.2 per-token KV layout): bytes ``[0:512)`` e4m3 codes,
``[512:528)`` four little-endian fp32 scales (one per 128 codes, powers of
two), ``[528:656)`` 64 bf16 rope values.

Recipe: nope values ``x ~ N(0,1)``; per 128-block ``scale =
2^ceil(log2(amax/448))``; stored code = e4m3(x / scale) rounded to nearest
even (torch's float8_e4m3fn cast) -- or, for the int8 cache format, ``scale =
amax/127`` and code = rint(x / scale) as a signed byte; rope ``~ N(0,1)`` rounded to bf16; q ``~
N(0,1)`` rounded to bf16; sinks ``N(0,1)`` (or zeros); unique random indices
per query row.  numpy PCG64, seed 0 unless stated.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

ROW_BYTES = 656
PAGE = 64
D_QK = 576
D_V = 512
POISON = 0x7FFFFFFF


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor  # bf16 [T, H, 576] (CPU)
    kv: torch.Tensor  # uint8 [num_pages, 64, 656] (CPU)
    indices: torch.Tensor  # int32 [T, ld], ld >= topk (CPU)
    topk: int
    sm_scale: float
    topk_length: Optional[torch.Tensor] = None  # int32 [T]
    attn_sink: Optional[torch.Tensor] = None  # fp32 [H]
    block_table: Optional[torch.Tensor] = None  # int32 [B, max_pages]
    tokens_per_req: int = 1
    decode: bool = False
    meta: dict = dataclasses.field(default_factory=dict)
    # dual-cache form: a second index list into a second cache (same row format)
    extra_kv: Optional[torch.Tensor] = None  # uint8 [num_pages2, 64, 656]
    extra_indices: Optional[torch.Tensor] = None  # int32 [T, ld2]
    extra_topk: int = 0
    extra_topk_length: Optional[torch.Tensor] = None  # int32 [T]
    extra_block_table: Optional[torch.Tensor] = None  # int32 [B, max_pages2]
    kv_format: str = "e4m3"  # code bytes of every cache: "e4m3" or "int8"
    layout: str = "rope64"  # "rope64", or "nope": q is [T, H, 512] and row bytes [528:656) are padding

    @property
    def dual(self):
        return self.extra_kv is not None

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def num_pages(self):
        return self.kv.shape[0]


def pow2_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Exponent e with 2^e = 2^ceil(log2(amax/448)), computed exactly via frexp."""
    v = np.asarray(amax, dtype=np.float64) / 448.0
    m, e = np.frexp(np.where(v > 0, v, 1.0))
    e = e - (m == 0.5).astype(e.dtype)
    return np.where(v > 0, e, 0)


def make_cache(rng: np.random.Generator, num_pages: int, chunk_rows: int = 65536, kv_format: str = "e4m3",
               scales: str = "pow2", layout: str = "rope64") -> torch.Tensor:
    """A paged cache ``[num_pages, 64, 656]`` of uint8 rows (see module docstring).

    ``kv_format="int8"``: the same row layout with signed int8 codes, per-128
    ``scale = amax / 127`` (fp32, not a power of two) and ``code =
    rint(x / scale)`` clipped to [-127, 127].  ``scales="any"`` (e4m3 only):
    ``scale = amax / 448`` as stored, not rounded to a power of two (GLM NSA
    stores arbitrary fp32 scales).  ``layout="nope"``: bytes ``[528:656)``
    are padding filled with 0xFF (a NaN pattern as bf16), never to be read."""
    n_rows = num_pages * PAGE
    out = np.empty((n_rows, ROW_BYTES), dtype=np.uint8)
    for lo in range(0, n_rows, chunk_rows):
        hi = min(n_rows, lo + chunk_rows)
        n = hi - lo
        x = rng.standard_normal((n, 512), dtype=np.float32)
        amax = np.abs(x.reshape(n, 4, 128)).max(axis=2)
        if kv_format == "int8":
            scale = (np.maximum(amax, np.float32(1e-30)) / np.float32(127.0)).astype(np.float32)  # [n, 4]
            y = (x.reshape(n, 4, 128) / scale[:, :, None]).reshape(n, 512)
            codes = np.clip(np.rint(y), -127, 127).astype(np.int8).view(np.uint8)
        elif scales == "any":
            scale = (np.maximum(amax, np.float32(1e-30)) / np.float32(448.0)).astype(np.float32)
            y = (x.reshape(n, 4, 128) / scale[:, :, None]).reshape(n, 512)
            y = np.clip(y, -448.0, 448.0)
            codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        else:
            e = pow2_scale_exponent(amax)
            scale = np.ldexp(np.float32(1.0), e).astype(np.float32)  # [n, 4]
            y = (x.reshape(n, 4, 128) / scale[:, :, None]).reshape(n, 512)
            y = np.clip(y, -448.0, 448.0)
            codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        rope = rng.standard_normal((n, 64), dtype=np.float32)
        rope_bits = torch.from_numpy(rope).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
        out[lo:hi, 0:512] = codes
        out[lo:hi, 512:528] = scale.astype("<f4").view(np.uint8).reshape(n, 16)
        out[lo:hi, 528:656] = rope_bits.reshape(n, 128) if layout == "rope64" else 0xFF
    return torch.from_numpy(out.reshape(num_pages, PAGE, ROW_BYTES))


def unique_rows(rng: np.random.Generator, T: int, K: int, N: int) -> np.ndarray:
    """``T`` rows of ``K`` distinct integers drawn uniformly from ``[0, N)``."""
    assert K <= N
    if 2 * K > N:
        keys = rng.random((T, N))
        return np.argsort(keys, axis=1)[:, :K].astype(np.int64)
    out = rng.integers(0, N, size=(T, K), dtype=np.int64)
    for _ in range(1000):
        order = np.argsort(out, axis=1, kind="stable")
        srt = np.take_along_axis(out, order, axis=1)
        d = np.zeros_like(srt, dtype=bool)
        d[:, 1:] = srt[:, 1:] == srt[:, :-1]
        if not d.any():
            return out
        dup = np.zeros_like(d)
        np.put_along_axis(dup, order, d, axis=1)
        out[dup] = rng.integers(0, N, size=int(dup.sum()), dtype=np.int64)
    raise RuntimeError("unique_rows did not converge")


def _bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)


def make_prefill(name, T, H, ctx, topk, seed=0, sink="normal", ld=None, ragged=False,
                 neg_prob=0.0, sm_scale=None, kv_format="e4m3", scales="pow2", layout="rope64") -> Workload:
    """Flat-addressed prefill: one context of ``ctx`` rows, ``topk`` unique ids per row.

    ``ragged``: topk_length ~ U{1..topk} per row and entries past it set to -1.
    ``ld``: index row stride (columns ``topk..ld`` hold a poison value).
    ``neg_prob``: each entry independently replaced by -1 with this probability.
    """
    rng = np.random.default_rng(seed)
    assert ctx % PAGE == 0
    kv = make_cache(rng, ctx // PAGE, kv_format=kv_format, scales=scales, layout=layout)
    d_qk = D_QK if layout == "rope64" else D_V
    q = _bf16(rng, (T, H, d_qk))
    ld = topk if ld is None else ld
    idx = np.full((T, ld), POISON, dtype=np.int64)
    idx[:, :topk] = unique_rows(rng, T, topk, ctx)
    tl = None
    if ragged:
        lens = rng.integers(1, topk + 1, size=T)
        tl = torch.from_numpy(lens.astype(np.int32))
        cols = np.arange(topk)[None, :]
        idx[:, :topk] = np.where(cols < lens[:, None], idx[:, :topk], -1)
    if neg_prob > 0:
        drop = rng.random((T, topk)) < neg_prob
        idx[:, :topk] = np.where(drop, -1, idx[:, :topk])
    if sink == "normal":
        s = torch.from_numpy(rng.standard_normal(H).astype(np.float32))
    elif sink == "zeros":
        s = torch.zeros(H, dtype=torch.float32)
    else:
        s = None
    return Workload(
        name=name, q=q, kv=kv, indices=torch.from_numpy(idx.astype(np.int32)), topk=topk,
        sm_scale=(1.0 / math.sqrt(d_qk)) if sm_scale is None else sm_scale,
        topk_length=tl, attn_sink=s, kv_format=kv_format, layout=layout,
        meta=dict(T=T, H=H, ctx=ctx, topk=topk, ld=ld, seed=seed, ragged=ragged,
                  neg_prob=neg_prob, sink=sink, kv_format=kv_format))


def make_decode(name, n_req, tokens_per_req, H, ctx_per_req, topk, seed=0, sink="normal",
                kv_format="e4m3", layout="rope64") -> Workload:
    """Paged decode: ``n_req`` requests, each its own context of ``ctx_per_req``
    logical positions mapped through a block table that is one shuffled
    permutation of all pages; ``topk`` unique logical ids per query token."""
    rng = np.random.default_rng(seed)
    assert ctx_per_req % PAGE == 0
    pages_per_req = ctx_per_req // PAGE
    num_pages = n_req * pages_per_req
    kv = make_cache(rng, num_pages, kv_format=kv_format, layout=layout)
    T = n_req * tokens_per_req
    d_qk = D_QK if layout == "rope64" else D_V
    q = _bf16(rng, (T, H, d_qk))
    bt = rng.permutation(num_pages).reshape(n_req, pages_per_req)
    idx = unique_rows(rng, T, topk, ctx_per_req)
    if sink == "normal":
        s = torch.from_numpy(rng.standard_normal(H).astype(np.float32))
    elif sink == "zeros":
        s = torch.zeros(H, dtype=torch.float32)
    else:
        s = None
    return Workload(
        name=name, q=q, kv=kv, indices=torch.from_numpy(idx.astype(np.int32)), topk=topk,
        sm_scale=1.0 / math.sqrt(d_qk), attn_sink=s,
        block_table=torch.from_numpy(bt.astype(np.int32)), tokens_per_req=tokens_per_req,
        decode=True, kv_format=kv_format, layout=layout,
        meta=dict(n_req=n_req, tokens_per_req=tokens_per_req, H=H, ctx_per_req=ctx_per_req,
                  topk=topk, seed=seed, sink=sink))


def _ragged_lengths(rng, T, topk, idx):
    """topk_length ~ U{0..topk} with the entries past it set to -1 (in place)."""
    lens = rng.integers(0, topk + 1, size=T)
    cols = np.arange(topk)[None, :]
    idx[:, :topk] = np.where(cols < lens[:, None], idx[:, :topk], -1)
    return torch.from_numpy(lens.astype(np.int32))


def make_dual_prefill(name, T, H, ctx, topk, extra_ctx, extra_topk, seed=0, sink="normal",
                      ragged=False, kv_format="e4m3") -> Workload:
    """Dual-cache prefill: a flat first list of ``topk`` unique ids into a cache
    of ``ctx`` rows and a flat second list of ``extra_topk`` unique ids into a
    second cache of ``extra_ctx`` rows.  ``ragged``: both lists get
    topk_length ~ U{0..width} (so either can be empty for a token)."""
    wl = make_prefill(name, T, H, ctx, topk, seed=seed, sink=sink, kv_format=kv_format)
    rng = np.random.default_rng(seed + 7919)
    assert extra_ctx % PAGE == 0
    wl.extra_kv = make_cache(rng, extra_ctx // PAGE, kv_format=kv_format)
    idx2 = unique_rows(rng, T, extra_topk, extra_ctx)
    if ragged:
        idx1 = wl.indices.numpy().astype(np.int64)
        wl.topk_length = _ragged_lengths(rng, T, topk, idx1)
        wl.indices = torch.from_numpy(idx1.astype(np.int32))
        wl.extra_topk_length = _ragged_lengths(rng, T, extra_topk, idx2)
    wl.extra_indices = torch.from_numpy(idx2.astype(np.int32))
    wl.extra_topk = extra_topk
    wl.meta.update(extra_ctx=extra_ctx, extra_topk=extra_topk, ragged=ragged)
    return wl


def make_dual_decode(name, n_req, tokens_per_req, H, ctx_per_req, topk, extra_ctx_per_req, extra_topk,
                     seed=0, sink="normal", kv_format="e4m3") -> Workload:
    """Dual-cache decode: the paged decode of ``make_decode`` plus, per
    request, a second paged cache of ``extra_ctx_per_req`` logical positions
    (its own shuffled block table) and ``extra_topk`` unique logical ids."""
    wl = make_decode(name, n_req, tokens_per_req, H, ctx_per_req, topk, seed=seed, sink=sink, kv_format=kv_format)
    rng = np.random.default_rng(seed + 7919)
    assert extra_ctx_per_req % PAGE == 0
    pages2 = extra_ctx_per_req // PAGE
    wl.extra_kv = make_cache(rng, n_req * pages2, kv_format=kv_format)
    wl.extra_block_table = torch.from_numpy(rng.permutation(n_req * pages2).reshape(n_req, pages2).astype(np.int32))
    wl.extra_indices = torch.from_numpy(unique_rows(rng, wl.T, extra_topk, extra_ctx_per_req).astype(np.int32))
    wl.extra_topk = extra_topk
    wl.meta.update(extra_ctx_per_req=extra_ctx_per_req, extra_topk=extra_topk)
    return wl


# The five workloads, named by what they are.
def tiny_prefill(seed=0):
    return make_prefill("tiny_prefill_T4_H8_ctx256_k64", T=4, H=8, ctx=256, topk=64,
                        seed=seed, sink="zeros")


def prefill_16k(topk=512, seed=0, T=1024):
    return make_prefill(f"prefill_T{T}_H64_ctx16384_k{topk}", T=T, H=64, ctx=16384,
                        topk=topk, seed=seed)


def fewhead_prefill(seed=0, T=8192):
    return make_prefill(f"fewhead_prefill_T{T}_H8_ctx32768_k640_ld1024_ragged", T=T, H=8,
                        ctx=32768, topk=640, seed=seed, ld=1024, ragged=True)


def batched_decode(seed=0, n_req=64):
    return make_decode(f"decode_{n_req}req_x2_H64_ctx32768_k2048_paged", n_req=n_req,
                       tokens_per_req=2, H=64, ctx_per_req=32768, topk=2048, seed=seed)


def large_prefill(seed=0, T=4096):
    return make_prefill(f"large_prefill_T{T}_H128_ctx131072_k2048_neg0.1", T=T, H=128,
                        ctx=131072, topk=2048, seed=seed, neg_prob=0.1)


def dual_decode(seed=0, n_req=64):
    """The dual-cache decode shape "topk 1024 + 2176": 64 requests x 2 tokens,
    H=64, a 32768-position main cache and an 8192-position second cache per
    request, both paged."""
    return make_dual_decode(f"dual_decode_{n_req}req_x2_H64_ctx32768_k1024+ctx8192_k2176_paged", n_req=n_req,
                            tokens_per_req=2, H=64, ctx_per_req=32768, topk=1024, extra_ctx_per_req=8192,
                            extra_topk=2176, seed=seed)


def prefill_16k_int8(topk=1024, seed=0, T=1024):
    """The 16k-footprint prefill on an INT8 cache (the AppMana releases page
    times "int8 width 1024" at this footprint)."""
    return make_prefill(f"prefill_T{T}_H64_ctx16384_k{topk}_int8", T=T, H=64, ctx=16384, topk=topk, seed=seed,
                        kv_format="int8")


WORKLOADS = {
    "tiny": tiny_prefill,
    "prefill16k_k512": lambda seed=0: prefill_16k(512, seed),
    "prefill16k_k1024": lambda seed=0: prefill_16k(1024, seed),
    "fewhead": fewhead_prefill,
    "decode": batched_decode,
    "large": large_prefill,
    "dual_decode": dual_decode,
    "prefill16k_int8": prefill_16k_int8,
}
