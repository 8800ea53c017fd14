"""Pins of the CPU oracle against things other than itself (CPU only).

Each pin is a library routine (torch dtype conversions, scaled_dot_product_attention,
logsumexp), a hand-derived closed form (tests/golden/), a mathematical invariant
(permutation, identical rows, paged == flat), or brute force on tiny inputs.
The last test plants mistakes into copies of the oracle functions and checks that
the pins catch each of them.
"""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle.sparse_mla_oracle as O
from sparse_mla_attention_03_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------------------- helpers
def build_row(codes=None, scales=(1.0, 1.0, 1.0, 1.0), rope_bits=None):
    """One 656-byte row assembled byte by byte (struct for the fp32 scales)."""
    r = np.zeros(656, dtype=np.uint8)
    for i, c in (codes or {}).items():
        r[int(i)] = c
    r[512:528] = np.frombuffer(struct.pack("<4f", *scales), dtype=np.uint8)
    for i, bits in (rope_bits or {}).items():
        r[528 + 2 * int(i)] = bits & 0xFF
        r[528 + 2 * int(i) + 1] = (bits >> 8) & 0xFF
    return r


def dequant_via_torch(kv_rows):
    """Dequantise with torch's own dtype conversions (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(kv_rows))
    codes = t[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    sc = t[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    rope = t[:, 528:656].contiguous().view(torch.bfloat16).to(torch.float64)
    nope = codes * sc.repeat_interleave(128, dim=1)
    return torch.cat([nope, rope], dim=1)


def q_f64(wl):
    return wl.q.to(torch.float64).numpy()


def sdpa_dense(q, K, sm_scale, sink=None):
    """Reference dense attention for one token via torch SDPA in float64.

    The sink is modelled as one extra key whose logit equals sink[h] (an additive
    mask on a zero key) and whose value is zero."""
    H = q.shape[0]
    qt = torch.from_numpy(q).reshape(1, H, 1, 576)
    Kt = torch.as_tensor(K).reshape(1, 1, -1, 576).expand(1, H, -1, 576)
    Vt = torch.as_tensor(K[:, :512]).reshape(1, 1, -1, 512).expand(1, H, -1, 512)
    mask = None
    if sink is not None:
        Kt = torch.cat([Kt, torch.zeros(1, H, 1, 576, dtype=torch.float64)], dim=2)
        Vt = torch.cat([Vt, torch.zeros(1, H, 1, 512, dtype=torch.float64)], dim=2)
        mask = torch.zeros(1, H, 1, Kt.shape[2], dtype=torch.float64)
        mask[0, :, 0, -1] = torch.as_tensor(sink, dtype=torch.float64)
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask, scale=sm_scale)
    scores = (qt @ torch.as_tensor(K).T.reshape(1, 1, 576, -1)).reshape(H, -1) * sm_scale
    lse = torch.logsumexp(scores, dim=1)
    return out.reshape(H, 512).numpy(), lse.numpy()


def tiny_dense_workload(seed=3, H=4, ctx=256):
    """A full-coverage case: every context row is selected, in a random order."""
    rng = np.random.default_rng(seed)
    wl = inputs.make_prefill("dense", T=3, H=H, ctx=ctx, topk=ctx, seed=seed, sink=None)
    perm = np.stack([rng.permutation(ctx) for _ in range(3)]).astype(np.int32)
    wl.indices = torch.from_numpy(perm)
    return wl


# ----------------------------------------------------------------------------- pins
def check_e4m3(e4m3_to_f64=O.e4m3_to_f64):
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_to_f64(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    fin = ~np.isnan(lib)
    assert np.array_equal(ours[fin], lib[fin])
    assert np.array_equal(np.signbit(ours[fin]), np.signbit(lib[fin]))
    # closed forms
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    assert ours[0x08] == 2.0 ** -6 and ours[0xB8] == -1.0 and ours[0x40] == 2.0


def test_e4m3_exhaustive_and_closed_forms():
    check_e4m3()


def test_bf16_and_f32_decoders():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=20000, dtype=np.uint16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ours = O.bf16_bits_to_f64(bits)
    fin = ~np.isnan(lib)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[fin], lib[fin])
    vals = [1.0, -2.5, 2.0 ** -7, 3.4e38, 1e-40]
    raw = np.frombuffer(struct.pack("<5f", *vals), dtype=np.uint8)
    got = O.f32_le_bytes_to_f64(raw)
    want = np.array(struct.unpack("<5f", struct.pack("<5f", *vals)))
    assert np.array_equal(got, want)


def check_decode_rows(decode_rows=O.decode_rows):
    wl = inputs.make_prefill("dq", T=1, H=1, ctx=128, topk=8, seed=11)
    rows = wl.kv.numpy().reshape(-1, 656)
    ours = decode_rows(rows)
    lib = dequant_via_torch(rows).numpy()
    assert np.array_equal(ours, lib)
    # a row built byte by byte: code 0x38 at nope[130] with scale[1] = 0.125; rope[3] = -1.5
    r = build_row({130: 0x38, 5: 0xC0}, scales=(2.0, 0.125, 1.0, 1.0), rope_bits={3: 0xBFC0})
    k = decode_rows(r[None, :])[0]
    assert k[130] == 0.125 and k[5] == -4.0 and k[512 + 3] == -1.5
    assert np.count_nonzero(k) == 3


def test_decode_rows_vs_torch_and_by_hand():
    check_decode_rows()


def check_golden(attend=None):
    with open(os.path.join(HERE, "golden", "hand_closed_forms.json")) as f:
        g = json.load(f)
    for ex in g["examples"]:
        rows = np.stack([build_row({int(k): v for k, v in r["codes"].items()}, r["scales"],
                                   {int(k): v for k, v in r["rope"].items()}) for r in ex["rows"]])
        H = ex["H"]
        q = np.zeros((1, H, 576))
        for h, qd in enumerate(ex["q"]):
            for d, v in qd.items():
                q[0, h, int(d)] = v
        kv = np.zeros((64, 656), dtype=np.uint8)
        kv[: rows.shape[0]] = rows
        idx = np.full((1, 4), -1, dtype=np.int32)
        idx[0, : rows.shape[0]] = np.arange(rows.shape[0])
        for case in ex["cases"]:
            out, lse = O.sparse_mla_forward(q, kv.reshape(1, 64, 656), idx, 4, ex["sm_scale"],
                                            attn_sink=case["sink"])
            for h in range(H):
                want = np.zeros(512)
                for d, v in case["out"][h].items():
                    want[int(d)] = v
                np.testing.assert_allclose(out[0, h], want, rtol=0, atol=1e-15)
                assert abs(lse[0, h] - case["lse"][h]) < 1e-14


def test_hand_derived_closed_forms():
    check_golden()


def check_dense_vs_sdpa(forward=O.sparse_mla_forward, with_sink=False):
    wl = tiny_dense_workload()
    sink = np.array([0.3, -1.2, 2.0, 0.0]) if with_sink else None
    out, lse = forward(q_f64(wl), wl.kv.numpy(), wl.indices.numpy(), wl.topk, wl.sm_scale,
                       attn_sink=sink)
    K = dequant_via_torch(wl.kv.numpy().reshape(-1, 656)).numpy()
    for t in range(wl.T):
        ro, rl = sdpa_dense(q_f64(wl)[t], K, wl.sm_scale, sink)
        np.testing.assert_allclose(out[t], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], rl, rtol=0, atol=1e-12)


def test_dense_coverage_equals_sdpa():
    check_dense_vs_sdpa(with_sink=False)


def test_sink_equals_extra_key_in_sdpa():
    check_dense_vs_sdpa(with_sink=True)


def test_single_valid_index():
    wl = inputs.make_prefill("one", T=2, H=4, ctx=128, topk=16, seed=5, sink="normal")
    idx = np.full((2, 16), -1, dtype=np.int32)
    idx[0, 7] = 42
    idx[1, 0] = 99
    q = q_f64(wl)
    sink = wl.attn_sink.numpy().astype(np.float64)
    out, lse = O.sparse_mla_forward(q, wl.kv.numpy(), idx, 16, wl.sm_scale)
    outs, lses = O.sparse_mla_forward(q, wl.kv.numpy(), idx, 16, wl.sm_scale, attn_sink=sink)
    K = dequant_via_torch(wl.kv.numpy().reshape(-1, 656)).numpy()
    for t, row in ((0, 42), (1, 99)):
        s = wl.sm_scale * (q[t] @ K[row])
        np.testing.assert_allclose(out[t], np.broadcast_to(K[row, :512], (4, 512)), atol=1e-14)
        np.testing.assert_allclose(lse[t], s, atol=1e-12)
        sig = 1.0 / (1.0 + np.exp(sink - s))
        np.testing.assert_allclose(outs[t], sig[:, None] * K[row, :512][None, :], atol=1e-13)


def test_identical_rows_give_row_and_log_n():
    wl = inputs.make_prefill("same", T=1, H=3, ctx=64, topk=5, seed=6, sink=None)
    kv = wl.kv.numpy().copy().reshape(-1, 656)
    for r in range(1, 5):
        kv[r] = kv[0]
    idx = np.array([[0, 1, 2, 3, 4]], dtype=np.int32)
    out, lse = O.sparse_mla_forward(q_f64(wl), kv.reshape(1, 64, 656), idx, 5, wl.sm_scale)
    out1, lse1 = O.sparse_mla_forward(q_f64(wl), kv.reshape(1, 64, 656), idx[:, :1], 1, wl.sm_scale)
    np.testing.assert_allclose(out, out1, atol=1e-14)
    np.testing.assert_allclose(lse, lse1 + math.log(5), atol=1e-12)


def test_permutation_invariance_including_padding():
    wl = inputs.make_prefill("perm", T=3, H=4, ctx=512, topk=64, seed=8, neg_prob=0.25)
    rng = np.random.default_rng(1)
    idx = wl.indices.numpy()
    perm = np.stack([rng.permutation(64) for _ in range(3)])
    idx_p = np.take_along_axis(idx, perm, axis=1)
    a = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), idx, 64, wl.sm_scale, attn_sink=wl.attn_sink.numpy())
    b = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), idx_p, 64, wl.sm_scale, attn_sink=wl.attn_sink.numpy())
    np.testing.assert_allclose(a[0], b[0], atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], atol=1e-12)


def test_truncation_equals_padding_and_clamps():
    wl = inputs.make_prefill("trunc", T=4, H=2, ctx=256, topk=32, seed=9)
    idx = wl.indices.numpy()
    tl = np.array([5, 0, 40, -3], dtype=np.int32)
    pad = idx.copy()
    for t, n in enumerate(np.clip(tl, 0, 32)):
        pad[t, n:] = -1
    a = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), idx, 32, wl.sm_scale, topk_length=tl)
    b = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), pad, 32, wl.sm_scale)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert np.all(a[1][1] == -np.inf) and np.all(a[0][1] == 0) and np.all(a[1][3] == -np.inf)


def test_paged_equals_flat_after_page_shuffle():
    rng = np.random.default_rng(4)
    wl = inputs.make_prefill("paged", T=4, H=2, ctx=1024, topk=48, seed=12)
    kv = wl.kv.numpy()  # 16 pages, request view = logical order
    n_pages = kv.shape[0]
    # two requests of two tokens, each with its own 8 logical pages
    perm = rng.permutation(n_pages)
    phys = np.empty_like(kv)
    phys[perm] = kv  # logical page p lives at physical page perm[p]
    bt = perm.reshape(2, 8).astype(np.int32)
    logical = np.stack([rng.choice(512, 48, replace=False) for _ in range(4)]).astype(np.int32)
    out_p, lse_p = O.sparse_mla_forward(q_f64(wl), phys, logical, 48, wl.sm_scale,
                                        block_table=bt, tokens_per_req=2)
    flat = logical.copy()
    flat[2:] += 512  # request 1's logical pages are logical pages 8..15
    out_f, lse_f = O.sparse_mla_forward(q_f64(wl), kv, flat, 48, wl.sm_scale)
    np.testing.assert_array_equal(out_p, out_f)
    np.testing.assert_array_equal(lse_p, lse_f)
    # a logical page beyond the block-table row is masked like -1
    bad = logical.copy()
    bad[0, 0] = 8 * 64 + 3
    rows = O.resolve_rows(bad, 48, n_pages, block_table=bt, tokens_per_req=2)
    assert rows[0, 0] == -1 and rows[0, 1] == perm[logical[0, 1] // 64] * 64 + logical[0, 1] % 64


def test_out_of_range_is_masked_like_padding():
    wl = inputs.make_prefill("oor", T=2, H=2, ctx=128, topk=8, seed=13)
    idx = wl.indices.numpy().copy()
    bad = idx.copy()
    bad[0, 2] = 128
    bad[1, 5] = -7
    pad = idx.copy()
    pad[0, 2] = -1
    pad[1, 5] = -1
    a = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), bad, 8, wl.sm_scale)
    b = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), pad, 8, wl.sm_scale)
    np.testing.assert_array_equal(a[0], b[0])


def test_empty_row():
    wl = inputs.make_prefill("empty", T=1, H=3, ctx=64, topk=4, seed=14)
    idx = np.full((1, 4), -1, dtype=np.int32)
    out, lse = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), idx, 4, wl.sm_scale,
                                    attn_sink=wl.attn_sink.numpy())
    assert np.all(out == 0) and np.all(lse == -np.inf)


def check_split_merge(merge=O.merge_partials):
    wl = inputs.make_prefill("split", T=1, H=4, ctx=512, topk=200, seed=15)
    q = q_f64(wl)[0]
    K = O.decode_rows(wl.kv.numpy().reshape(-1, 656)[wl.indices.numpy()[0]])
    sink = wl.attn_sink.numpy().astype(np.float64)
    ref = O.attend_one(q, K, wl.sm_scale, sink)
    for bounds in ([(0, 200)], [(0, 64), (64, 128), (128, 200)], [(0, 100), (100, 100), (100, 200)],
                   [(i, min(200, i + 7)) for i in range(0, 200, 7)] + [(200, 200)]):
        parts = O.split_partials(q, K, wl.sm_scale, bounds)
        out, lse = merge(parts, sink)
        np.testing.assert_allclose(out, ref[0], atol=1e-13)
        np.testing.assert_allclose(lse, ref[1], atol=1e-12)
    empty = merge(O.split_partials(q, K[:0], wl.sm_scale, [(0, 0), (0, 0)]), sink)
    assert np.all(empty[0] == 0) and np.all(empty[1] == -np.inf)


def test_split_merge_equals_one_shot():
    check_split_merge()


# ----------------------------------------------------------------------------- planted mistakes
def _bad_e4m3_bias(codes):
    b = np.asarray(codes).astype(np.int64)
    e = (b >> 3) & 0xF
    m = (b & 7) / 8.0
    v = np.where(e == 0, m * 2.0 ** -7, (1 + m) * np.exp2(e - 8.0))
    return np.where(b & 0x80, -v, v)


def _bad_decode_scale_index(rows):
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    nope = O.e4m3_to_f64(rows[:, :512])
    sc = O.f32_le_bytes_to_f64(rows[:, 512:528]).reshape(n, 4)
    nope = nope * np.tile(sc, (1, 128))  # wrong: i % 4 instead of i // 128
    rope = O.bf16_bits_to_f64(np.ascontiguousarray(rows[:, 528:]).view("<u2"))
    return np.concatenate([nope, rope], axis=1)


def _bad_decode_rope_order(rows):
    k = O.decode_rows(rows)
    k[:, 512:] = k[:, 512:][:, ::-1]
    return k


def _bad_merge_sink_twice(parts, sink=None):
    out, lse = O.merge_partials(parts, sink)
    if sink is not None:
        out = out * (1.0 / (1.0 + np.exp(np.asarray(sink) - lse)))[:, None]
    return out, lse


def _bad_merge_plain_average(parts, sink=None):
    outs = np.stack([p[0] for p in parts])
    out, lse = O.merge_partials(parts, sink)
    return outs.mean(axis=0), lse


def test_planted_mistakes_are_caught(monkeypatch):
    with pytest.raises(AssertionError):
        check_e4m3(_bad_e4m3_bias)
    with pytest.raises(AssertionError):
        check_decode_rows(_bad_decode_scale_index)
    with pytest.raises(AssertionError):
        check_decode_rows(_bad_decode_rope_order)
    with pytest.raises(AssertionError):
        check_split_merge(_bad_merge_sink_twice)
    with pytest.raises(AssertionError):
        check_split_merge(_bad_merge_plain_average)

    def bad_attend_sink_in_numerator(q_t, K, sm_scale, sink=None):
        out, lse = orig_attend(q_t, K, sm_scale, None)
        if sink is not None:
            out = out + np.exp(np.asarray(sink))[:, None] * 1e-3
        return out, lse

    def bad_attend_no_scale(q_t, K, sm_scale, sink=None):
        return orig_attend(q_t, K, 1.0, sink)

    def bad_attend_lse_with_sink(q_t, K, sm_scale, sink=None):
        out, lse = orig_attend(q_t, K, sm_scale, sink)
        if sink is not None:
            lse = np.logaddexp(lse, sink)
        return out, lse

    def bad_attend_transposed_v(q_t, K, sm_scale, sink=None):
        out, lse = orig_attend(q_t, K, sm_scale, sink)
        return out[:, ::-1].copy(), lse

    orig_attend = O.attend_one
    for bad, with_sink in ((bad_attend_no_scale, False), (bad_attend_transposed_v, False),
                           (bad_attend_sink_in_numerator, True), (bad_attend_lse_with_sink, True)):
        monkeypatch.setattr(O, "attend_one", bad)
        with pytest.raises(AssertionError):
            check_dense_vs_sdpa(O.sparse_mla_forward, with_sink=with_sink)
            check_golden()
        monkeypatch.setattr(O, "attend_one", orig_attend)


# ----------------------------------------------------------------------------- dual-cache form
def _dual_case(seed=21):
    return inputs.make_dual_prefill("dualpin", T=5, H=3, ctx=256, topk=70, extra_ctx=192, extra_topk=45,
                                    seed=seed, ragged=True)


def _call_dual(fwd, wl, kv=None, extra_kv=None, **kw):
    args = dict(topk_length=None if wl.topk_length is None else wl.topk_length.numpy(),
                extra_topk_length=None if wl.extra_topk_length is None else wl.extra_topk_length.numpy(),
                attn_sink=wl.attn_sink.numpy(), extra_block_table=None if wl.extra_block_table is None
                else wl.extra_block_table.numpy(), block_table=None if wl.block_table is None
                else wl.block_table.numpy(), tokens_per_req=wl.tokens_per_req)
    args.update(kw)
    return fwd(q_f64(wl), wl.kv.numpy() if kv is None else kv, wl.indices.numpy(), wl.topk,
               wl.extra_kv.numpy() if extra_kv is None else extra_kv, wl.extra_indices.numpy(), wl.extra_topk,
               wl.sm_scale, **args)


def check_dual(fwd=None):
    """The dual-cache form against the one-list form and a library routine."""
    fwd = fwd or O.sparse_mla_forward_dual
    wl = _dual_case()
    out, lse = _call_dual(fwd, wl)
    l1, l2 = wl.topk_length.numpy(), wl.extra_topk_length.numpy()
    # (a) both caches stacked into one cache, the second list's ids shifted past
    # the first cache's rows, the lengths written as -1 padding
    kv1 = wl.kv.numpy().reshape(-1, 656)
    kv2 = wl.extra_kv.numpy().reshape(-1, 656)
    stack = np.concatenate([kv1, kv2])
    i1 = wl.indices.numpy().astype(np.int64)
    i1 = np.where(np.arange(wl.topk)[None, :] < l1[:, None], i1, -1)
    i2 = wl.extra_indices.numpy().astype(np.int64)
    i2 = np.where(np.arange(wl.extra_topk)[None, :] < l2[:, None], i2 + kv1.shape[0], -1)
    one = np.concatenate([i1, i2], axis=1).astype(np.int32)
    out_s, lse_s = O.sparse_mla_forward(q_f64(wl), stack, one, one.shape[1], wl.sm_scale,
                                        attn_sink=wl.attn_sink.numpy())
    np.testing.assert_allclose(out, out_s, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_s, rtol=1e-12, atol=1e-12)
    # (b) an empty second list is the one-list form over the first list
    out_e, lse_e = _call_dual(fwd, wl, extra_topk_length=np.zeros(wl.T, dtype=np.int32))
    out_1, lse_1 = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), wl.indices.numpy(), wl.topk, wl.sm_scale,
                                        topk_length=l1, attn_sink=wl.attn_sink.numpy())
    np.testing.assert_allclose(out_e, out_1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_e, lse_1, rtol=1e-12, atol=1e-12)
    # (c) swapping the two lists (with their caches) changes nothing
    out_w, lse_w = fwd(q_f64(wl), wl.extra_kv.numpy(), wl.extra_indices.numpy(), wl.extra_topk, wl.kv.numpy(),
                       wl.indices.numpy(), wl.topk, wl.sm_scale, topk_length=l2, extra_topk_length=l1,
                       attn_sink=wl.attn_sink.numpy())
    np.testing.assert_allclose(out_w, out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse_w, lse, rtol=1e-12, atol=1e-12)
    # (d) one cache, its rows split between the two lists: dense attention
    # over the whole context through torch SDPA, with the sink as an extra key
    dense = tiny_dense_workload(seed=5, H=3, ctx=128)
    sink = np.array([0.3, -1.2, 2.0])
    kvd = dense.kv.numpy()
    perm = dense.indices.numpy()
    od, ld = fwd(q_f64(dense), kvd, perm[:, :50], 50, kvd, perm[:, 50:], 78, dense.sm_scale, attn_sink=sink)
    K = dequant_via_torch(kvd.reshape(-1, 656)).numpy()
    for t in range(dense.T):
        ref_o, ref_l = sdpa_dense(q_f64(dense)[t], K, dense.sm_scale, sink)
        np.testing.assert_allclose(od[t], ref_o, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(ld[t], ref_l, rtol=1e-12, atol=1e-12)
    # (e) a paged second list equals the flat list of its physical rows
    wd = inputs.make_dual_decode("dualpaged", n_req=2, tokens_per_req=2, H=2, ctx_per_req=256, topk=40,
                                 extra_ctx_per_req=128, extra_topk=30, seed=8)
    op, lp = _call_dual(fwd, wd)
    bt2 = wd.extra_block_table.numpy().astype(np.int64)
    li = wd.extra_indices.numpy().astype(np.int64)
    req = (np.arange(wd.T) // wd.tokens_per_req)[:, None]
    phys = (bt2[req, li // 64] * 64 + li % 64).astype(np.int32)
    of, lf = fwd(q_f64(wd), wd.kv.numpy(), wd.indices.numpy(), wd.topk, wd.extra_kv.numpy(), phys, wd.extra_topk,
                 wd.sm_scale, attn_sink=wd.attn_sink.numpy(), block_table=wd.block_table.numpy(),
                 tokens_per_req=wd.tokens_per_req)
    np.testing.assert_array_equal(op, of)
    np.testing.assert_array_equal(lp, lf)


def test_dual_cache_form_against_one_list_and_sdpa():
    check_dual()


def test_dual_cache_planted_mistakes_are_caught():
    def second_list_in_first_cache(q, kv, i1, k1, kv2, i2, k2, sm_scale, **kw):
        return O.sparse_mla_forward_dual(q, kv, i1, k1, kv, i2, k2, sm_scale, **kw)

    def two_softmaxes_averaged(q, kv, i1, k1, kv2, i2, k2, sm_scale, topk_length=None, extra_topk_length=None,
                               attn_sink=None, block_table=None, extra_block_table=None, tokens_per_req=1):
        a = O.sparse_mla_forward(q, kv, i1, k1, sm_scale, topk_length=topk_length, attn_sink=attn_sink,
                                 block_table=block_table, tokens_per_req=tokens_per_req)
        b = O.sparse_mla_forward(q, kv2, i2, k2, sm_scale, topk_length=extra_topk_length, attn_sink=attn_sink,
                                 block_table=extra_block_table, tokens_per_req=tokens_per_req)
        return 0.5 * (a[0] + b[0]), np.logaddexp(a[1], b[1])

    def second_length_ignored(q, kv, i1, k1, kv2, i2, k2, sm_scale, extra_topk_length=None, **kw):
        return O.sparse_mla_forward_dual(q, kv, i1, k1, kv2, i2, k2, sm_scale, **kw)

    for bad in (second_list_in_first_cache, two_softmaxes_averaged, second_length_ignored):
        with pytest.raises(AssertionError):
            check_dual(bad)


# ----------------------------------------------------------------------------- int8 cache format
def dequant_int8_via_torch(kv_rows):
    """int8 codes through torch's own int8 view (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(kv_rows))
    codes = t[:, :512].contiguous().view(torch.int8).to(torch.float64)
    sc = t[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    rope = t[:, 528:656].contiguous().view(torch.bfloat16).to(torch.float64)
    return torch.cat([codes * sc.repeat_interleave(128, dim=1), rope], dim=1)


def check_int8(int8_to_f64=O.int8_to_f64, decode_rows=O.decode_rows):
    codes = np.arange(256, dtype=np.uint8)
    ours = int8_to_f64(codes)
    lib = torch.from_numpy(codes).view(torch.int8).to(torch.float64).numpy()
    assert np.array_equal(ours, lib)
    assert ours[0x7F] == 127 and ours[0x80] == -128 and ours[0xFF] == -1 and ours[0x01] == 1
    wl = inputs.make_prefill("dq8", T=1, H=1, ctx=128, topk=8, seed=11, kv_format="int8")
    rows = wl.kv.numpy().reshape(-1, 656)
    assert np.array_equal(decode_rows(rows, "int8"), dequant_int8_via_torch(rows).numpy())
    # by hand: code 0xFE (-2) at nope[300] with scale[2] = 0.75 -> -1.5
    r = build_row({300: 0xFE}, scales=(1.0, 1.0, 0.75, 1.0))
    k = decode_rows(r[None, :], "int8")[0]
    assert k[300] == -1.5 and np.count_nonzero(k) == 1


def test_int8_decoder_and_rows():
    check_int8()


def test_int8_dense_coverage_equals_sdpa():
    rng = np.random.default_rng(9)
    wl = inputs.make_prefill("dense8", T=3, H=4, ctx=256, topk=256, seed=9, sink=None, kv_format="int8")
    wl.indices = torch.from_numpy(np.stack([rng.permutation(256) for _ in range(3)]).astype(np.int32))
    sink = np.array([0.3, -1.2, 2.0, 0.0])
    out, lse = O.sparse_mla_forward(q_f64(wl), wl.kv.numpy(), wl.indices.numpy(), 256, wl.sm_scale,
                                    attn_sink=sink, kv_format="int8")
    K = dequant_int8_via_torch(wl.kv.numpy().reshape(-1, 656)).numpy()
    for t in range(wl.T):
        ro, rl = sdpa_dense(q_f64(wl)[t], K, wl.sm_scale, sink)
        np.testing.assert_allclose(out[t], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], rl, rtol=0, atol=1e-12)


def test_int8_planted_mistakes_are_caught():
    def unsigned(codes):
        return np.asarray(codes, dtype=np.uint8).astype(np.float64)

    def offset_binary(codes):
        return np.asarray(codes, dtype=np.uint8).astype(np.float64) - 128.0

    for bad in (unsigned, offset_binary):
        with pytest.raises(AssertionError):
            check_int8(int8_to_f64=bad)
    # the row decoder reading int8 rows as e4m3 fails the row pin
    with pytest.raises(AssertionError):
        check_int8(decode_rows=lambda rows, fmt: O.decode_rows(rows, "e4m3"))


# ----------------------------------------------------------------------------- no-rope layout (GLM53_NOPE)
def check_nope(forward=O.sparse_mla_forward):
    wl = inputs.make_prefill("nopepin", T=4, H=3, ctx=256, topk=90, seed=31, ragged=True, layout="nope")
    sink = np.array([0.5, -0.4, 1.0])
    out, lse = forward(q_f64(wl), wl.kv.numpy(), wl.indices.numpy(), wl.topk, wl.sm_scale,
                       topk_length=wl.topk_length.numpy(), attn_sink=sink, layout="nope")
    # the 0xFF padding (NaN as bf16) is never read
    assert np.isfinite(out).all() and not np.isnan(lse).any()
    # equals the rope layout with a zero q rope and zero rope bytes
    kv = wl.kv.numpy().copy()
    kv[..., 528:656] = 0
    q576 = np.concatenate([q_f64(wl), np.zeros((wl.T, wl.H, 64))], axis=2)
    out_r, lse_r = O.sparse_mla_forward(q576, kv, wl.indices.numpy(), wl.topk, wl.sm_scale,
                                        topk_length=wl.topk_length.numpy(), attn_sink=sink)
    np.testing.assert_allclose(out, out_r, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_r, rtol=1e-12, atol=1e-12)
    # dense coverage against SDPA over 512-dim keys
    rng = np.random.default_rng(4)
    dn = inputs.make_prefill("nopedense", T=2, H=3, ctx=128, topk=128, seed=41, sink=None, layout="nope")
    dn.indices = torch.from_numpy(np.stack([rng.permutation(128) for _ in range(2)]).astype(np.int32))
    od, ld = forward(q_f64(dn), dn.kv.numpy(), dn.indices.numpy(), 128, dn.sm_scale, attn_sink=sink,
                     layout="nope")
    K = dequant_via_torch(dn.kv.numpy().reshape(-1, 656)).numpy()[:, :512]
    for t in range(dn.T):
        qt = torch.from_numpy(q_f64(dn)[t]).reshape(1, 3, 1, 512)
        Kt = torch.as_tensor(K).reshape(1, 1, -1, 512).expand(1, 3, -1, 512)
        Kt = torch.cat([Kt, torch.zeros(1, 3, 1, 512, dtype=torch.float64)], dim=2)
        mask = torch.zeros(1, 3, 1, Kt.shape[2], dtype=torch.float64)
        mask[0, :, 0, -1] = torch.as_tensor(sink)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Kt, attn_mask=mask, scale=dn.sm_scale)
        np.testing.assert_allclose(od[t], ref.reshape(3, 512).numpy(), rtol=0, atol=1e-12)
        sc = (qt.reshape(3, 512) @ torch.as_tensor(K).T) * dn.sm_scale
        np.testing.assert_allclose(ld[t], torch.logsumexp(sc, dim=1).numpy(), rtol=0, atol=1e-12)


def test_nope_layout_pins():
    check_nope()


def test_nope_planted_mistake_reads_padding():
    orig = O.decode_rows

    def reads_padding(rows, kv_format="e4m3", layout="rope64"):
        k = orig(rows, kv_format, "rope64")
        return k[:, :512] + 0.0 * k[:, 512:].sum(axis=1, keepdims=True) if layout == "nope" else k

    def forward(*a, **kw):
        O.decode_rows = reads_padding
        try:
            return O.sparse_mla_forward(*a, **kw)
        finally:
            O.decode_rows = orig

    with pytest.raises(AssertionError):
        check_nope(forward)
