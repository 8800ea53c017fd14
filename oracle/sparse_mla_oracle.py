"""Plain CPU oracle for sparse MLA attention forward (prefill and decode).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA library (no kernels, headers, tables or helpers);
the only thing both sides share is the seeded input generator, which holds
none of the arithmetic below.

Everything is numpy float64 and written as the plain definition of the result,
one token at a time, so that it can be checked against the pages by eye:

* Row layout (656 bytes, FP8 "nope" + per-128 fp32 scales + bf16 rope):
  FlashInfer PR #4802 "Refactor Sparse MLA SM120", review note on
  ``decode_dsv3_2_kernel.cuh`` (the per-token KV layout comment:
  ``[0:512)`` e4m3, ``[512:528)`` 4 x FP32 scale, one per 128-element tile,
  ``[528:656)`` 64 x BF16 rope; "DSv3.2 stores power-of-2 FP32 scales").
* Paged cache with page block 64 (``page_block_size != 64`` is rejected):
  same PR, commit note on dispatch-miss diagnostics.
* Index rows with -1 padding, a row stride taken from the tensor, last dim
  contiguous: same PR, commit note on taking the index row stride from the
  tensor.
* ``topk_length`` and the per-head ``attn_sink``: vLLM PR #57673
  "[Perf][DSv4.1] Native-head Triton sparse MLA for SM90 few-head prefill",
  Test Result section ("combined topk 640, attn_sink + topk_length").
* V shares the latent with K and ``d_v == d_nope == 512``: FlashInfer PR
  #4802, Summary (the "rope writeback overrun at D_V==D_NOPE" fix).
* Split-K decode merged with an LSE-weighted combine: AppMana
  forks-flash-mla-ampere-dsv4 releases, "decode H6: warp-wide combine";
  FlashInfer PR #4802, "Runner and CUDA graphs" (decode split-K scratch).

Readings where the pages are silent (each one is listed with its reason in
the design notes of the repository):

* sink: ``attn_sink[h]`` is a logit in the same (scaled) units as the scores;
  it adds ``exp(sink[h])`` to the softmax denominator only (a key with a zero
  value vector).  A missing sink means ``-inf`` (no sink).
* LSE: natural log of the scaled scores, sink excluded.
* A slot is valid iff ``j < clamp(topk_length[t], 0, topk)`` and the index is
  in range (``0 <= idx < rows`` for flat addressing; for paged addressing the
  logical page must lie inside the block-table row and the physical page
  inside the cache).  Anything else (-1 or out of range) is masked like -1.
* No valid slot: ``out = 0`` and ``lse = -inf``.
* e4m3 is OCP E4M3FN: bias 7, no infinities, ``S.1111.111`` is NaN.

Pins (``tests/test_oracle.py``): the e4m3 / bf16 / fp32 decoders against
torch's own dtype conversions over every code; a hand-derived closed-form
example in ``tests/golden/``; dense attention via
``torch.nn.functional.scaled_dot_product_attention`` when the index set covers
the whole context; the sink as an extra key through the same library routine;
one valid index; identical rows; permutation invariance; paged == flat after a
page shuffle; truncation == -1 padding; the split/merge algebra against the
one-shot result; the dual-cache form against the one-list form (two caches
stacked into one with the second list's ids shifted, an empty second list,
the two lists swapped, and one list split in two over the same cache); the
int8 decoder against torch's int8 view over every byte and SDPA on an int8
cache.  Every function below has at least one of these pins.
"""
from __future__ import annotations

import numpy as np

# Shape constants of the 656-byte row (FlashInfer PR #4802, KV layout note).
ROW_BYTES = 656
D_NOPE = 512
D_ROPE = 64
D_QK = D_NOPE + D_ROPE  # 576
D_V = D_NOPE  # 512: V is the nope part of the same latent row
SCALE_BLOCK = 128
PAGE_BLOCK = 64
_SCALE_OFF = 512
_ROPE_OFF = 528


# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------
def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode OCP E4M3FN bytes to float64.

    Sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent field 0
    is subnormal (m/8 * 2^-6); ``x.1111.111`` is NaN; there is no infinity.
    """
    b = np.asarray(codes).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def int8_to_f64(codes: np.ndarray) -> np.ndarray:
    """Signed int8 codes (two's complement bytes) to float64."""
    return np.asarray(codes, dtype=np.uint8).view(np.int8).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the top half of an IEEE binary32: widen the bits and reinterpret."""
    u = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f32_le_bytes_to_f64(b: np.ndarray) -> np.ndarray:
    """Little-endian IEEE binary32 from groups of 4 bytes (last axis)."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint8))
    return b.view("<f4").astype(np.float64)


# ----------------------------------------------------------------------------
# Row decoding (the dequantisation step)
# ----------------------------------------------------------------------------
def decode_rows(rows: np.ndarray, kv_format: str = "e4m3", layout: str = "rope64") -> np.ndarray:
    """Dequantise latent rows: uint8 ``[n, 656]`` -> float64 ``[n, 576]``.

    ``k[i] = code(byte[i]) * scale[i // 128]`` for ``i < 512`` and
    ``k[512 + i] = bf16(rope[i])`` for ``i < 64`` (FlashInfer PR #4802, KV
    layout note).  V of the same row is ``k[:512]``.  ``code`` is e4m3, or
    for ``kv_format="int8"`` a signed byte: the AppMana releases page names
    INT8 latent-cache kernels without a byte layout, read here as the same
    row with int8 codes in place of e4m3.  ``layout="nope"`` (GLM53_NOPE,
    FlashInfer PR #4802 review note on the KV layout comment): no rope,
    ``[528:656)`` is padding and is not read; the result is ``[n, 512]``.
    """
    rows = np.asarray(rows, dtype=np.uint8)
    assert rows.ndim == 2 and rows.shape[1] == ROW_BYTES, rows.shape
    assert kv_format in ("e4m3", "int8"), kv_format
    n = rows.shape[0]
    nope = (int8_to_f64 if kv_format == "int8" else e4m3_to_f64)(rows[:, :D_NOPE])
    scales = f32_le_bytes_to_f64(rows[:, _SCALE_OFF:_ROPE_OFF]).reshape(n, D_NOPE // SCALE_BLOCK)
    nope = nope * np.repeat(scales, SCALE_BLOCK, axis=1)
    if layout == "nope":
        return nope
    assert layout == "rope64", layout
    rope_bits = np.ascontiguousarray(rows[:, _ROPE_OFF:ROW_BYTES]).view("<u2")
    rope = bf16_bits_to_f64(rope_bits)
    return np.concatenate([nope, rope], axis=1)


# ----------------------------------------------------------------------------
# Index handling (validity + address translation)
# ----------------------------------------------------------------------------
def resolve_rows(indices, topk, num_pages, topk_length=None, block_table=None,
                 tokens_per_req=1, tokens=None):
    """Physical cache row for every slot ``(t, j)``, ``j < topk``; -1 if invalid.

    ``indices`` may be wider than ``topk`` (a view into a wider buffer); only
    the first ``topk`` columns are read.  Flat addressing: row = idx, valid iff
    ``0 <= idx < num_pages * 64``.  Paged addressing: request
    ``r = t // tokens_per_req``, logical page ``idx // 64`` must be inside the
    block-table row, and ``row = block_table[r, idx // 64] * 64 + idx % 64``
    with the physical page inside the cache.
    """
    idx = np.asarray(indices)[:, :topk].astype(np.int64)
    T = idx.shape[0]
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    idx = idx[sel]
    if topk_length is None:
        lens = np.full(sel.shape[0], topk, dtype=np.int64)
    else:
        lens = np.clip(np.asarray(topk_length).astype(np.int64)[sel], 0, topk)
    j = np.arange(topk)[None, :]
    in_len = j < lens[:, None]
    rows = np.full(idx.shape, -1, dtype=np.int64)
    if block_table is None:
        ok = in_len & (idx >= 0) & (idx < num_pages * PAGE_BLOCK)
        rows[ok] = idx[ok]
        return rows
    bt = np.asarray(block_table).astype(np.int64)
    req = sel // int(tokens_per_req)
    lpage = np.where(idx >= 0, idx // PAGE_BLOCK, -1)
    ok = in_len & (idx >= 0) & (lpage < bt.shape[1]) & (req[:, None] < bt.shape[0])
    safe_lp = np.where(ok, lpage, 0)
    safe_req = np.broadcast_to(np.where(req < bt.shape[0], req, 0)[:, None], idx.shape)
    ppage = bt[safe_req, safe_lp]
    ok &= (ppage >= 0) & (ppage < num_pages)
    rows[ok] = ppage[ok] * PAGE_BLOCK + idx[ok] % PAGE_BLOCK
    return rows


# ----------------------------------------------------------------------------
# Attention for one token
# ----------------------------------------------------------------------------
def attend_one(q_t, K, sm_scale, sink=None):
    """Sink softmax attention of one token over its gathered rows.

    ``q_t``: ``[H, d_qk]`` float64; ``K``: ``[n, d_qk]`` dequantised rows
    (``V = K[:, :512]``); ``sink``: ``[H]`` logits or None.
    Returns ``(out [H, 512], lse [H])`` with

        s_j  = sm_scale * <q_h, k_j>
        m    = max_j s_j,   l = sum_j exp(s_j - m),   lse = m + log l
        out  = sum_j exp(s_j - m) v_j / (l + exp(sink_h - m))
    """
    H = q_t.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, D_V)), np.full(H, -np.inf)
    s = sm_scale * (q_t @ K.T)  # [H, n]
    m = s.max(axis=1)
    p = np.exp(s - m[:, None])
    l = p.sum(axis=1)
    lse = m + np.log(l)
    denom = l if sink is None else l + np.exp(np.asarray(sink, dtype=np.float64) - m)
    out = (p @ K[:, :D_V]) / denom[:, None]
    return out, lse


def sparse_mla_forward(q, kv_cache, indices, topk, sm_scale, topk_length=None,
                       attn_sink=None, block_table=None, tokens_per_req=1,
                       tokens=None, q_selected=False, kv_format="e4m3", layout="rope64"):
    """Sparse MLA forward for the selected tokens (all tokens by default).

    ``q``: float64 ``[T, H, 576]`` (bf16 values widened exactly), or only the
    rows of ``tokens`` in that order when ``q_selected``;
    ``kv_cache``: uint8 ``[num_pages, 64, 656]`` (or ``[rows, 656]``);
    ``indices``: int ``[T, >= topk]``.  Returns float64 ``out [n_sel, H, 512]``
    and ``lse [n_sel, H]`` (natural log, sink excluded).
    """
    kv = np.asarray(kv_cache, dtype=np.uint8).reshape(-1, ROW_BYTES)
    num_pages = kv.shape[0] // PAGE_BLOCK
    q = np.asarray(q, dtype=np.float64)
    T = np.asarray(indices).shape[0]
    _, H, D = q.shape
    assert D == (D_QK if layout == "rope64" else D_NOPE)
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    if q_selected:
        assert q.shape[0] == sel.shape[0]
    rows = resolve_rows(indices, topk, num_pages, topk_length, block_table,
                        tokens_per_req, sel)
    out = np.zeros((sel.shape[0], H, D_V))
    lse = np.zeros((sel.shape[0], H))
    sink = None if attn_sink is None else np.asarray(attn_sink, dtype=np.float64)
    for i, t in enumerate(sel):
        r = rows[i]
        K = decode_rows(kv[r[r >= 0]], kv_format, layout)
        out[i], lse[i] = attend_one(q[i] if q_selected else q[t], K, sm_scale, sink)
    return out, lse


def sparse_mla_forward_dual(q, kv_cache, indices, topk, extra_kv_cache, extra_indices, extra_topk,
                            sm_scale, topk_length=None, extra_topk_length=None, attn_sink=None,
                            block_table=None, extra_block_table=None, tokens_per_req=1,
                            tokens=None, q_selected=False, kv_format="e4m3", layout="rope64"):
    """Dual-cache form: one sink softmax per token over the valid slots of two
    index lists, the first resolved in ``kv_cache`` and the second in
    ``extra_kv_cache`` (FlashInfer PR #4802: the DSv4 secondary cache with its
    own index row stride; dual-cache decode-form calls that must not ignore
    the secondary cache; the "topk=1024+2176 dual" decode shape).

    Each list follows the slot rules of ``resolve_rows`` in its own cache and
    with its own ``topk`` / ``topk_length`` / block table (``tokens_per_req``
    is shared).  The candidate set is the concatenation of both lists' valid
    rows, and the sink enters the denominator once.
    """
    kv1 = np.asarray(kv_cache, dtype=np.uint8).reshape(-1, ROW_BYTES)
    kv2 = np.asarray(extra_kv_cache, dtype=np.uint8).reshape(-1, ROW_BYTES)
    q = np.asarray(q, dtype=np.float64)
    T = np.asarray(indices).shape[0]
    _, H, D = q.shape
    assert D == (D_QK if layout == "rope64" else D_NOPE) and np.asarray(extra_indices).shape[0] == T
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    if q_selected:
        assert q.shape[0] == sel.shape[0]
    rows1 = resolve_rows(indices, topk, kv1.shape[0] // PAGE_BLOCK, topk_length, block_table,
                         tokens_per_req, sel)
    rows2 = resolve_rows(extra_indices, extra_topk, kv2.shape[0] // PAGE_BLOCK, extra_topk_length,
                         extra_block_table, tokens_per_req, sel)
    out = np.zeros((sel.shape[0], H, D_V))
    lse = np.zeros((sel.shape[0], H))
    sink = None if attn_sink is None else np.asarray(attn_sink, dtype=np.float64)
    for i, t in enumerate(sel):
        r1, r2 = rows1[i], rows2[i]
        K = np.concatenate([decode_rows(kv1[r1[r1 >= 0]], kv_format, layout),
                            decode_rows(kv2[r2[r2 >= 0]], kv_format, layout)], axis=0)
        out[i], lse[i] = attend_one(q[i] if q_selected else q[t], K, sm_scale, sink)
    return out, lse


# ----------------------------------------------------------------------------
# Split-K decode: partial results and the LSE-weighted merge
# ----------------------------------------------------------------------------
def split_partials(q_t, K, sm_scale, bounds):
    """Sink-free partial results over contiguous chunks of the gathered rows.

    ``bounds``: list of ``(lo, hi)`` row ranges.  Each chunk returns its own
    normalised output ``o_s`` and ``lse_s`` (``-inf`` and zeros when empty).
    """
    parts = []
    for lo, hi in bounds:
        parts.append(attend_one(q_t, K[lo:hi], sm_scale, None))
    return parts


def merge_partials(parts, sink=None):
    """LSE-weighted merge of split partials, then the sink.

    ``lse = log sum_s exp(lse_s)``; ``o = sum_s exp(lse_s - lse) o_s``;
    with a sink the result is scaled by ``exp(lse) / (exp(lse) + exp(sink))``.
    Splits with ``lse_s = -inf`` weigh 0; if all are empty, out = 0 and
    lse = -inf.
    """
    lses = np.stack([p[1] for p in parts])  # [S, H]
    outs = np.stack([p[0] for p in parts])  # [S, H, 512]
    mx = lses.max(axis=0)
    H = lses.shape[1]
    out = np.zeros((H, D_V))
    lse = np.full(H, -np.inf)
    live = np.isfinite(mx)
    if live.any():
        w = np.exp(lses[:, live] - mx[live])
        tot = w.sum(axis=0)
        lse[live] = mx[live] + np.log(tot)
        out[live] = (w[:, :, None] * outs[:, live]).sum(axis=0) / tot[:, None]
        if sink is not None:
            sk = np.asarray(sink, dtype=np.float64)[live]
            out[live] *= (1.0 / (1.0 + np.exp(sk - lse[live])))[:, None]
    return out, lse
