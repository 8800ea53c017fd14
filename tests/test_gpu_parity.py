"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases run the oracle on every token (several 64-row tiles plus a ragged
tail); the full-size workloads run the oracle on a seeded sample of tokens.
Index handling is compared bit for bit through sparse_mla_resolve_rows.
"""
import numpy as np
import pytest
import torch

import oracle.sparse_mla_oracle as O
from sparse_mla_attention_03_gb300 import binding, inputs
from tests.helpers import assert_close, oracle_dual_for, oracle_for, sample_tokens_by_quarter, to_dev

pytestmark = pytest.mark.gpu


def run_prefill(wl, **kw):
    d = to_dev(wl)
    return binding.sparse_mla_prefill(d["q"], d["kv"], d["indices"], wl.sm_scale, topk=wl.topk,
                                      topk_length=d["topk_length"], attn_sink=d["attn_sink"],
                                      block_table=d["block_table"], tokens_per_req=wl.tokens_per_req,
                                      kv_format=wl.kv_format, layout=wl.layout, **kw)


def run_decode(wl, num_splits=0, **kw):
    d = to_dev(wl)
    return binding.sparse_mla_decode(d["q"], d["kv"], d["indices"], wl.sm_scale, topk=wl.topk,
                                     topk_length=d["topk_length"], attn_sink=d["attn_sink"],
                                     block_table=d["block_table"], tokens_per_req=wl.tokens_per_req,
                                     num_splits=num_splits, kv_format=wl.kv_format, layout=wl.layout, **kw)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    binding.get_error_word()  # clear
    yield


# ----------------------------------------------------------------------------- small, full oracle
def test_tiny_workload_prefill_and_decode():
    wl = inputs.tiny_prefill()
    ref = oracle_for(wl)
    out, lse = run_prefill(wl)
    torch.cuda.synchronize()
    assert_close(out, lse, *ref, tag="tiny prefill")
    for s in (0, 1, 2):
        out, lse = run_decode(wl, num_splits=s)
        assert_close(out, lse, *ref, tag=f"tiny decode S={s}")
    assert binding.get_error_word() == 0


@pytest.mark.parametrize("H", [1, 5, 8, 16, 24, 64, 128])
@pytest.mark.parametrize("sink", ["normal", None])
def test_small_prefill_heads(H, sink):
    wl = inputs.make_prefill(f"small_H{H}", T=5, H=H, ctx=2048, topk=200, seed=H, sink=sink,
                             neg_prob=0.15)
    ref = oracle_for(wl)
    out, lse = run_prefill(wl)
    assert_close(out, lse, *ref, tag=f"H={H} sink={sink}")


@pytest.mark.parametrize("H", [8, 64])
def test_ragged_topk_length_and_strided_index_view(H):
    wl = inputs.make_prefill("ragged", T=7, H=H, ctx=4096, topk=320, seed=21, ld=512, ragged=True)
    wl.topk_length[0] = 0
    wl.topk_length[1] = 1
    wl.topk_length[2] = 320
    wl.topk_length[3] = 65
    ref = oracle_for(wl)
    out, lse = run_prefill(wl)
    assert_close(out, lse, *ref, tag="ragged")
    lse_h = lse.cpu().numpy()
    assert np.all(np.isneginf(lse_h[0])) and np.all(out[0].float().cpu().numpy() == 0)


@pytest.mark.parametrize("H", [8, 64])
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8, 32])
def test_decode_split_invariance_paged(H, S):
    wl = inputs.make_decode("dec_small", n_req=3, tokens_per_req=2, H=H, ctx_per_req=4096, topk=2048,
                            seed=31 + S)
    ref = oracle_for(wl)
    out, lse = run_decode(wl, num_splits=S)
    assert_close(out, lse, *ref, tag=f"decode H={H} S={S}")


@pytest.mark.parametrize("H,S", [(64, 0), (64, 5), (16, 0), (8, 3)])
def test_paged_decode_ragged_lengths_and_padding(H, S):
    # paged decode, 3 tokens per request, ragged topk_length (including 0 and
    # the full width), -1 entries inside the valid range, one out-of-range
    # logical page (masked and flagged)
    wl = inputs.make_decode("decrag", n_req=3, tokens_per_req=3, H=H, ctx_per_req=4096, topk=700, seed=301 + S)
    rng = np.random.default_rng(302)
    lens = rng.integers(0, 701, size=wl.T)
    lens[0], lens[1] = 0, 700
    wl.topk_length = torch.from_numpy(lens.astype(np.int32))
    idx = wl.indices.clone()
    idx[2, 5:40] = -1
    idx[3, 7] = 4096 + 64  # logical page 65 is outside the 64-column block-table row
    wl.indices = idx
    wl.topk_length[3] = 700
    out, lse = run_decode(wl, num_splits=S)
    assert_close(out, lse, *oracle_for(wl), tag=f"decode_ragged_H{H}_S{S}")
    assert binding.get_error_word() & binding.ERRF_INDEX_RANGE


def test_noncontiguous_views_written_in_place():
    # q[:, :8] / out[:, :8] views into width-64 buffers; index rows from a width-1024 buffer
    wl = inputs.make_prefill("views", T=6, H=8, ctx=2048, topk=192, seed=41, ld=1024)
    d = to_dev(wl)
    qbuf = torch.randn(6, 64, 576, device="cuda").to(torch.bfloat16)
    qbuf[:, :8] = d["q"]
    obuf = torch.full((6, 64, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((6, 64), 7.0, dtype=torch.float32, device="cuda")
    out, lse = binding.sparse_mla_prefill(qbuf[:, :8], d["kv"], d["indices"], wl.sm_scale, topk=192,
                                          attn_sink=d["attn_sink"], out=obuf[:, :8], lse=lbuf[:, :8])
    assert out.data_ptr() == obuf.data_ptr()
    ref = oracle_for(wl)
    assert_close(obuf[:, :8], lbuf[:, :8], *ref, tag="views")
    assert torch.all(obuf[:, 8:] == 7.0) and torch.all(lbuf[:, 8:] == 7.0)


@pytest.mark.parametrize("pad", [4, 8])
def test_tc_out_rows_with_padding(pad):
    # out rows padded by 4 or 8 elements (rows 8- or 16-byte aligned) of a
    # wider buffer, written in place; the padding is left untouched
    wl = inputs.make_prefill("outpad", T=5, H=64, ctx=2048, topk=320, seed=291 + pad, ragged=True)
    d = to_dev(wl)
    row = 64 * 512 + pad
    flat = torch.full((5 * row,), 3.0, dtype=torch.bfloat16, device="cuda")
    out = flat.as_strided((5, 64, 512), (row, 512, 1))
    o, lse = binding.sparse_mla_prefill(d["q"], d["kv"], d["indices"], wl.sm_scale, topk=wl.topk,
                                        topk_length=d["topk_length"], attn_sink=d["attn_sink"], out=out)
    assert o.data_ptr() == flat.data_ptr()
    assert_close(out, lse, *oracle_for(wl), tag=f"outpad{pad}")
    pads = flat.view(5, row)[:, 64 * 512:]
    assert torch.all(pads == 3.0)


def test_single_valid_index_and_empty_rows():
    wl = inputs.make_prefill("single", T=4, H=16, ctx=1024, topk=128, seed=51)
    idx = torch.full((4, 128), -1, dtype=torch.int32)
    idx[0, 77] = 5
    idx[1, 0] = 1023
    wl.indices = idx  # rows 2, 3 have no valid slot
    ref = oracle_for(wl)
    out, lse = run_prefill(wl)
    assert_close(out, lse, *ref, tag="single")
    out, lse = run_decode(wl, num_splits=2)
    assert_close(out, lse, *ref, tag="single decode")


def test_index_resolution_bit_exact_flat_and_paged():
    wl = inputs.make_prefill("res", T=9, H=8, ctx=1024, topk=96, seed=61, ld=130, ragged=True)
    idx = wl.indices.clone()
    idx[0, :4] = torch.tensor([1024, -5, 0x7FFFFFFF, 1023], dtype=torch.int32)
    wl.topk_length[0] = 96
    d = to_dev(wl)
    rows = binding.sparse_mla_resolve_rows(d["q"], d["kv"], idx.cuda(), topk=96,
                                           topk_length=d["topk_length"]).cpu().numpy()
    want = O.resolve_rows(idx.numpy(), 96, wl.num_pages, wl.topk_length.numpy())
    np.testing.assert_array_equal(rows, want)
    assert binding.get_error_word() & binding.ERRF_INDEX_RANGE
    dec = inputs.make_decode("resp", n_req=4, tokens_per_req=2, H=8, ctx_per_req=1024, topk=64, seed=62)
    didx = dec.indices.clone()
    didx[1, 3] = 1024  # logical page 16 is outside the 16-column block-table row
    dd = to_dev(dec)
    rows = binding.sparse_mla_resolve_rows(dd["q"], dd["kv"], didx.cuda(), block_table=dd["block_table"],
                                           tokens_per_req=2).cpu().numpy()
    want = O.resolve_rows(didx.numpy(), 64, dec.num_pages, block_table=dec.block_table.numpy(),
                          tokens_per_req=2)
    np.testing.assert_array_equal(rows, want)
    assert binding.get_error_word() & binding.ERRF_INDEX_RANGE


def test_two_streams_match_one_stream():
    wa = inputs.make_prefill("sa", T=16, H=8, ctx=2048, topk=256, seed=71)
    wb = inputs.make_prefill("sb", T=16, H=64, ctx=2048, topk=256, seed=72)
    ref_a, ref_b = run_prefill(wa), run_prefill(wb)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    da, db = to_dev(wa), to_dev(wb)
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        oa = binding.sparse_mla_prefill(da["q"], da["kv"], da["indices"], wa.sm_scale, attn_sink=da["attn_sink"])
    with torch.cuda.stream(s2):
        ob = binding.sparse_mla_prefill(db["q"], db["kv"], db["indices"], wb.sm_scale, attn_sink=db["attn_sink"])
    torch.cuda.synchronize()
    assert torch.equal(oa[0], ref_a[0]) and torch.equal(oa[1], ref_a[1])
    assert torch.equal(ob[0], ref_b[0]) and torch.equal(ob[1], ref_b[1])


def test_zero_tokens():
    wl = inputs.make_prefill("z", T=1, H=8, ctx=64, topk=8, seed=81)
    d = to_dev(wl)
    q0 = d["q"][:0]
    out, lse = binding.sparse_mla_prefill(q0, d["kv"], d["indices"][:0], wl.sm_scale)
    assert out.shape == (0, 8, 512)
    out, lse = binding.sparse_mla_decode(q0, d["kv"], d["indices"][:0], wl.sm_scale)
    assert lse.shape == (0, 8)


def test_deterministic_repeat():
    wl = inputs.make_prefill("det", T=8, H=64, ctx=4096, topk=512, seed=91)
    a = run_prefill(wl)
    b = run_prefill(wl)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ----------------------------------------------------------------------------- bounded waits
@pytest.mark.parametrize("mode", ["prefill", "decode_split3"])
def test_wait_limit_runs_out_and_the_context_stays_usable(mode):
    # With the test hook on, the tcgen05 kernel's producers gather nothing, so
    # the MMA issue's first wait is never completed.  With a 2 ms wait limit
    # the call ends with SMLA_ERRF_TIMEOUT in the error word instead of
    # hanging, and the next call on the same stream, hook off and default
    # limit, is correct.
    wl = inputs.make_prefill("waitlim", T=2, H=64, ctx=2048, topk=512, seed=311)
    call = run_prefill if mode == "prefill" else (lambda w: run_decode(w, num_splits=3))
    prev = binding.set_wait_limit_ns(2_000_000)
    binding.set_test_stall(True)
    try:
        call(wl)
        flags = binding.get_error_word()
    finally:
        binding.set_test_stall(False)
        binding.set_wait_limit_ns(prev)
    assert flags & binding.ERRF_TIMEOUT
    out, lse = call(wl)
    assert_close(out, lse, *oracle_for(wl), tag=f"{mode} after a timed-out call")
    assert binding.get_error_word() == 0


# ----------------------------------------------------------------------------- split choice, L2 guard
def test_decode_split_choice_beyond_l2_and_guard_limited_count():
    # H=128, 64 tokens, topk 2048, a 344 MB paged cache: the rows of each token
    # are gathered by two CTAs (two head groups).  The automatic choice is the
    # planner's for this device; on an L2 too small for those CTAs' rows the
    # L2-footprint guard would take more splits.  Both counts are correct.
    wl = inputs.make_decode("guard", n_req=32, tokens_per_req=2, H=128, ctx_per_req=16384, topk=2048, seed=321)
    props = torch.cuda.get_device_properties(0)
    sms, l2 = props.multi_processor_count, props.L2_cache_size
    auto = binding.decode_num_splits(wl.T, wl.H, wl.topk)
    assert auto == binding.plan_num_splits(wl.T, wl.H, wl.topk, 0, sms, l2)
    small_l2 = 3 * 16 * 64 * 656  # fits two splits' streamed rows, not one split's
    guarded = binding.plan_num_splits(wl.T, wl.H, wl.topk, 0, sms, small_l2)
    assert guarded > binding.plan_num_splits(wl.T, wl.H, wl.topk, 0, sms, 10 ** 15)
    ref = oracle_for(wl)
    for s_ in sorted({0, guarded}):
        out, lse = run_decode(wl, num_splits=s_)
        assert_close(out, lse, *ref, tag=f"beyond-L2 H=128 decode S={s_ or auto}")
    assert binding.get_error_word() == 0


# ----------------------------------------------------------------------------- size limits
@pytest.mark.parametrize("H,S", [(128, 0), (128, 64), (8, 64)])
def test_maximum_heads_splits_and_topk(H, S):
    # the largest head count, 64 splits (the maximum) and a 16384-slot index
    # list (256 chunks of 64) over a paged 32768-position context, with a
    # ragged topk_length so that some splits are empty
    wl = inputs.make_decode("maxsize", n_req=2, tokens_per_req=2, H=H, ctx_per_req=32768, topk=16384, seed=331 + S)
    wl.topk_length = torch.tensor([16384, 1, 9000, 0], dtype=torch.int32)
    eff = binding.decode_num_splits(wl.T, wl.H, wl.topk, S)
    assert S == 0 or eff == S
    out, lse = run_decode(wl, num_splits=S)
    assert_close(out, lse, *oracle_for(wl), tag=f"max H={H} S={S or eff} topk=16384")
    assert binding.get_error_word() == 0


# ----------------------------------------------------------------------------- caches beyond L2
# A cache larger than a quarter of the device's L2 (at least 32 MB on GB300)
# runs the tcgen05 kernel's early-load / L2-prefetch variant; these cases cover
# it with the full oracle on every token.
@pytest.mark.parametrize("H", [64, 128])
def test_cache_beyond_l2_prefill(H):
    wl = inputs.make_prefill("bigcache", T=5, H=H, ctx=65536, topk=704, seed=31, ragged=True, neg_prob=0.05)
    assert wl.kv.numel() >= 40 << 20
    out, lse = run_prefill(wl)
    assert_close(out, lse, *oracle_for(wl), tag=f"bigcache_prefill_H{H}")
    assert binding.get_error_word() == 0


@pytest.mark.parametrize("S", [1, 3])
def test_cache_beyond_l2_paged_decode(S):
    wl = inputs.make_decode("bigcache_dec", n_req=4, tokens_per_req=2, H=64, ctx_per_req=16384, topk=1024, seed=37)
    assert wl.kv.numel() >= 40 << 20
    out, lse = run_decode(wl, num_splits=S)
    assert_close(out, lse, *oracle_for(wl), tag=f"bigcache_decode_S{S}")
    assert binding.get_error_word() == 0


@pytest.mark.parametrize("H", [8, 64])
def test_q_heads_zero_subnormal_and_large(H):
    # the q prescale: an all-zero head, a head of bf16 subnormals (the
    # exponent-field shortcut falls back to the float maximum) and large heads
    wl = inputs.make_prefill("qext", T=3, H=H, ctx=1024, topk=200, seed=281)
    q = wl.q.clone()
    q[:, 0] = 0
    q[:, 1] = (q[:, 1].float() * 1e-39).to(torch.bfloat16)
    q[:, 2] = (q[:, 2].float() * 30.0).to(torch.bfloat16)
    q[:, H - 1] = (q[:, H - 1].float() * 1e-3).to(torch.bfloat16)
    wl.q = q
    out, lse = run_prefill(wl)
    assert_close(out, lse, *oracle_for(wl), tag=f"q_extreme_H{H}")
    assert binding.get_error_word() == 0


def test_q_heads_spanning_past_the_exact_range():
    # one q prescale per token (tcgen05 kernel): a head 2^24 times the others
    # pushes them down by about 2^-12 in f16, so their elements below about
    # 2^-2 become f16 subnormals and lose bits; the ordinary heads must still
    # meet the tolerances.  The large head's lse (about 1e7) is beyond what
    # fp32 resolves to 1e-3, so only its out is compared.
    wl = inputs.make_prefill("qspan", T=4, H=64, ctx=2048, topk=256, seed=283)
    big = 3
    q = wl.q.clone()
    q[:, big] = (q[:, big].float() * 2.0 ** 24).to(torch.bfloat16)
    wl.q = q
    out, lse = run_prefill(wl)
    ref_out, ref_lse = oracle_for(wl)
    keep = [h for h in range(wl.H) if h != big]
    assert_close(out[:, keep], lse[:, keep], ref_out[:, keep], ref_lse[:, keep], tag="q_span_2^24")
    o = out[:, big].float().cpu().numpy().astype(np.float64)
    assert np.abs(o - ref_out[:, big]).max() <= 2e-2
    assert binding.get_error_word() == 0


# ----------------------------------------------------------------------------- dual-cache form
def run_dual(wl, decode=False, num_splits=0):
    d = to_dev(wl)
    kw = dict(topk=wl.topk, topk_length=d["topk_length"], extra_topk=wl.extra_topk,
              extra_topk_length=d["extra_topk_length"], attn_sink=d["attn_sink"], block_table=d["block_table"],
              extra_block_table=d["extra_block_table"], tokens_per_req=wl.tokens_per_req, kv_format=wl.kv_format,
              layout=wl.layout)
    if decode:
        return binding.sparse_mla_decode_dual(d["q"], d["kv"], d["indices"], d["extra_kv"], d["extra_indices"],
                                              wl.sm_scale, num_splits=num_splits, **kw)
    return binding.sparse_mla_prefill_dual(d["q"], d["kv"], d["indices"], d["extra_kv"], d["extra_indices"],
                                           wl.sm_scale, **kw)


# topk 200 pads the first list to 256 combined slots, so 128-row tiles of the
# tcgen05 kernel and 64-row tiles of the warp-MMA kernel both meet padding,
# the list boundary and a ragged tail
@pytest.mark.parametrize("H", [8, 16, 64, 128])
def test_dual_prefill_ragged(H):
    wl = inputs.make_dual_prefill("dualp", T=7, H=H, ctx=2048, topk=200, extra_ctx=1024, extra_topk=150,
                                  seed=101 + H, ragged=True)
    wl.topk_length[0], wl.extra_topk_length[0] = 0, 150   # second list only
    wl.topk_length[1], wl.extra_topk_length[1] = 200, 0   # first list only
    wl.topk_length[2], wl.extra_topk_length[2] = 0, 0     # nothing: out 0, lse -inf
    out, lse = run_dual(wl)
    assert_close(out, lse, *oracle_dual_for(wl), tag=f"dual_prefill_H{H}")
    assert binding.get_error_word() == 0


@pytest.mark.parametrize("H,S", [(64, 0), (64, 1), (64, 3), (64, 8), (8, 0), (8, 5)])
def test_dual_decode_paged(H, S):
    wl = inputs.make_dual_decode("duald", n_req=3, tokens_per_req=2, H=H, ctx_per_req=4096, topk=300,
                                 extra_ctx_per_req=2048, extra_topk=217, seed=131 + S)
    out, lse = run_dual(wl, decode=True, num_splits=S)
    assert_close(out, lse, *oracle_dual_for(wl), tag=f"dual_decode_H{H}_S{S}")
    assert binding.get_error_word() == 0


def test_dual_cache_beyond_l2():
    # 43 MB + 10.7 MB of caches: the early-load / L2-prefetch variant
    wl = inputs.make_dual_prefill("dualbig", T=4, H=64, ctx=65536, topk=384, extra_ctx=16384, extra_topk=320,
                                  seed=151, ragged=True)
    out, lse = run_dual(wl)
    assert_close(out, lse, *oracle_dual_for(wl), tag="dual_bigcache")
    assert binding.get_error_word() == 0


def test_dual_index_resolution_bit_exact():
    wl = inputs.make_dual_decode("dualres", n_req=3, tokens_per_req=2, H=8, ctx_per_req=1024, topk=100,
                                 extra_ctx_per_req=512, extra_topk=70, seed=161)
    wl.topk_length = torch.tensor([100, 37, 0, 64, 99, 1], dtype=torch.int32)
    wl.extra_topk_length = torch.tensor([70, 0, 12, 70, 69, 33], dtype=torch.int32)
    i2 = wl.extra_indices.clone()
    i2[0, :3] = torch.tensor([512, -7, 0x7FFFFFFF], dtype=torch.int32)  # out of the 8-page table row
    wl.extra_indices = i2
    d = to_dev(wl)
    rows = binding.sparse_mla_resolve_rows_dual(
        d["q"], d["kv"], d["indices"], d["extra_kv"], d["extra_indices"], topk=wl.topk,
        topk_length=d["topk_length"], extra_topk=wl.extra_topk, extra_topk_length=d["extra_topk_length"],
        block_table=d["block_table"], extra_block_table=d["extra_block_table"], tokens_per_req=2).cpu().numpy()
    r1 = O.resolve_rows(wl.indices.numpy(), 100, wl.num_pages, wl.topk_length.numpy(),
                        wl.block_table.numpy(), 2)
    r2 = O.resolve_rows(wl.extra_indices.numpy(), 70, wl.extra_kv.shape[0], wl.extra_topk_length.numpy(),
                        wl.extra_block_table.numpy(), 2)
    base = binding.dual_width(100, 70) - 70
    assert base == 128 and rows.shape == (6, 198)
    want = np.full((6, 198), -1, dtype=np.int64)
    want[:, :100] = r1
    want[:, base:] = np.where(r2 >= 0, r2 + wl.num_pages * 64, -1)
    np.testing.assert_array_equal(rows, want)
    assert binding.get_error_word() & binding.ERRF_INDEX_RANGE


@pytest.mark.parametrize("H", [8, 64])
def test_empty_first_cache(H):
    # a cache with no pages (a null pointer): every index of the first list is
    # padding or out of range, so only the second list contributes
    wl = inputs.make_dual_prefill("dualempty", T=4, H=H, ctx=256, topk=96, extra_ctx=1024, extra_topk=200,
                                  seed=181)
    wl.kv = torch.empty((0, 64, 656), dtype=torch.uint8)
    idx = wl.indices.clone()
    idx[:, ::2] = -1
    wl.indices = idx
    out, lse = run_dual(wl)
    assert_close(out, lse, *oracle_dual_for(wl), tag=f"dual_empty_first_H{H}")
    assert binding.get_error_word() & binding.ERRF_INDEX_RANGE  # the other indices are out of range


def test_dual_rejects_bad_extra():
    wl = inputs.make_dual_prefill("dualbad", T=2, H=8, ctx=256, topk=64, extra_ctx=128, extra_topk=32, seed=171)
    d = to_dev(wl)
    with pytest.raises(ValueError):
        binding.sparse_mla_prefill_dual(d["q"], d["kv"], d["indices"], d["extra_kv"][:, :32], d["extra_indices"],
                                        wl.sm_scale)
    with pytest.raises(binding.SparseMLAError):
        binding.sparse_mla_prefill_dual(d["q"], d["kv"], d["indices"], d["extra_kv"], d["extra_indices"],
                                        wl.sm_scale, extra_topk=0)


# ----------------------------------------------------------------------------- caches beyond the whole L2
# A cache larger than the device's L2 itself runs the tcgen05 kernel's third
# load policy (256-byte row reads, 128-dim groups released in pairs); these
# cover its four instantiations (e4m3 / int8, one list / two) with the full
# oracle on every token.
@pytest.mark.parametrize("fmt", ["e4m3", "int8"])
@pytest.mark.parametrize("dual", [False, True])
def test_cache_beyond_whole_l2(fmt, dual):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    if dual:
        wl = inputs.make_dual_decode("huge_dual", n_req=2, tokens_per_req=2, H=64, ctx_per_req=131072, topk=1024,
                                     extra_ctx_per_req=4096, extra_topk=320, seed=353, kv_format=fmt)
        cache = wl.kv.numel() + wl.extra_kv.numel()
        assert cache > l2, (cache, l2)
        out, lse = run_dual(wl, decode=True)
        ref = oracle_dual_for(wl)
    else:
        wl = inputs.make_decode("huge", n_req=2, tokens_per_req=2, H=64, ctx_per_req=131072, topk=1536, seed=351,
                                kv_format=fmt)
        wl.topk_length = torch.tensor([1536, 700, 1, 1200], dtype=torch.int32)
        assert wl.kv.numel() > l2, (wl.kv.numel(), l2)
        out, lse = run_decode(wl, num_splits=0)
        ref = oracle_for(wl)
    assert_close(out, lse, *ref, tag=f"beyond_whole_L2_{fmt}_{'dual' if dual else 'one'}")
    assert binding.get_error_word() == 0


# ----------------------------------------------------------------------------- int8 cache format
@pytest.mark.parametrize("H", [1, 8, 16, 64, 128])
def test_int8_prefill_ragged(H):
    wl = inputs.make_prefill("i8p", T=6, H=H, ctx=2048, topk=300, seed=201 + H, ragged=True, kv_format="int8")
    out, lse = run_prefill(wl)
    assert_close(out, lse, *oracle_for(wl), tag=f"int8_prefill_H{H}")
    assert binding.get_error_word() == 0


@pytest.mark.parametrize("H,S", [(64, 0), (64, 3), (8, 0), (8, 4)])
def test_int8_decode_paged(H, S):
    wl = inputs.make_decode("i8d", n_req=3, tokens_per_req=2, H=H, ctx_per_req=4096, topk=512, seed=211 + S,
                            kv_format="int8")
    out, lse = run_decode(wl, num_splits=S)
    assert_close(out, lse, *oracle_for(wl), tag=f"int8_decode_H{H}_S{S}")
    assert binding.get_error_word() == 0


def test_int8_dual_and_beyond_l2():
    wl = inputs.make_dual_prefill("i8dual", T=4, H=64, ctx=65536, topk=320, extra_ctx=2048, extra_topk=200,
                                  seed=221, ragged=True, kv_format="int8")
    out, lse = run_dual(wl)
    assert_close(out, lse, *oracle_dual_for(wl), tag="int8_dual_bigcache")
    assert binding.get_error_word() == 0


def test_int8_differs_from_e4m3_reading():
    # the same bytes read in the two formats give different results: the
    # format field reaches the kernels
    wl = inputs.make_prefill("i8fmt", T=2, H=8, ctx=256, topk=64, seed=231, kv_format="int8")
    a, _ = run_prefill(wl)
    wl.kv_format = "e4m3"
    b, _ = run_prefill(wl)
    diff = (a.float() - b.float()).abs()  # codes 0x7F / 0xFF are NaN when read as e4m3
    assert torch.isnan(diff).any() or diff.max().item() > 1e-2


# ----------------------------------------------------------------------------- other row layouts
# GLM53_NOPE: no rope, q is [T, H, 512], row bytes [528, 656) are padding
# (filled with 0xFF, a NaN pattern as bf16, by the generator: reading them
# would poison the result)
@pytest.mark.parametrize("H", [8, 16, 64, 128])
def test_nope_prefill_ragged(H):
    wl = inputs.make_prefill("nopep", T=6, H=H, ctx=2048, topk=300, seed=241 + H, ragged=True, layout="nope")
    out, lse = run_prefill(wl)
    assert_close(out, lse, *oracle_for(wl), tag=f"nope_prefill_H{H}")
    assert binding.get_error_word() == 0


@pytest.mark.parametrize("H,S", [(64, 0), (64, 3), (8, 2)])
def test_nope_decode_paged(H, S):
    wl = inputs.make_decode("noped", n_req=3, tokens_per_req=2, H=H, ctx_per_req=4096, topk=512, seed=251 + S,
                            layout="nope", kv_format="int8" if S == 3 else "e4m3")
    out, lse = run_decode(wl, num_splits=S)
    assert_close(out, lse, *oracle_for(wl), tag=f"nope_decode_H{H}_S{S}")
    assert binding.get_error_word() == 0


def test_nope_dual_beyond_l2():
    wl = inputs.make_dual_prefill("nopedual", T=4, H=64, ctx=65536, topk=256, extra_ctx=1024, extra_topk=128,
                                  seed=261, ragged=True)
    # rebuild both caches and q in the no-rope layout
    nope = inputs.make_prefill("nopedual", T=4, H=64, ctx=65536, topk=256, seed=261, layout="nope")
    wl.q, wl.kv, wl.layout, wl.sm_scale = nope.q, nope.kv, "nope", nope.sm_scale
    wl.extra_kv = inputs.make_prefill("nopex", T=1, H=1, ctx=1024, topk=8, seed=262, layout="nope").kv
    out, lse = run_dual(wl)
    assert_close(out, lse, *oracle_dual_for(wl), tag="nope_dual")
    assert binding.get_error_word() == 0


# GLM_NSA: arbitrary (not power-of-two) fp32 scales on e4m3 codes
@pytest.mark.parametrize("H", [8, 64])
def test_arbitrary_scales(H):
    wl = inputs.make_prefill("nsa", T=6, H=H, ctx=2048, topk=384, seed=271 + H, ragged=True, scales="any")
    out, lse = run_prefill(wl)
    assert_close(out, lse, *oracle_for(wl), tag=f"arbitrary_scales_H{H}")
    assert binding.get_error_word() == 0


# ----------------------------------------------------------------------------- full-size workloads
# Each full-size workload runs in the benchmark's launch configuration (the
# automatic split count for decode); the oracle then checks a seeded sample of
# at least 256 query tokens, drawn evenly from the four quarters of the token
# range so that CTAs of every wave are covered, plus the first and last token.
# Workloads with fewer tokens than that are checked on every token.
FULL = {  # name: (generator, kind, query tokens)
    "prefill16k_k512": (lambda: inputs.prefill_16k(512), "prefill", 1024),
    "prefill16k_k1024": (lambda: inputs.prefill_16k(1024), "prefill", 1024),
    "fewhead": (inputs.fewhead_prefill, "prefill", 8192),
    "decode": (inputs.batched_decode, "decode", 128),
    "large": (inputs.large_prefill, "prefill", 4096),
    "dual_decode": (inputs.dual_decode, "dual_decode", 128),
    "prefill16k_int8_k1024": (inputs.prefill_16k_int8, "prefill", 1024),
}
FULL_SAMPLE = 256


@pytest.mark.parametrize("name", list(FULL),
                         ids=[f"{k}-{min(v[2], FULL_SAMPLE)}plus-of-{v[2]}-tokens" if v[2] > FULL_SAMPLE
                              else f"{k}-all-{v[2]}-tokens" for k, v in FULL.items()])
def test_full_size_workload_sampled(name):
    make, kind, n_tokens = FULL[name]
    wl = make()
    assert wl.T == n_tokens
    if kind == "dual_decode":
        out, lse = run_dual(wl, decode=True)
    else:
        out, lse = (run_prefill(wl) if kind == "prefill" else run_decode(wl))
    toks = sample_tokens_by_quarter(wl.T, FULL_SAMPLE, seed=5, must=(0, wl.T - 1))
    assert len(toks) >= min(FULL_SAMPLE, wl.T)
    for q in range(4):  # every quarter of the token range is represented
        assert np.any((toks >= q * wl.T // 4) & (toks < (q + 1) * wl.T // 4))
    ref = oracle_dual_for(wl, tokens=toks) if wl.dual else oracle_for(wl, tokens=toks)
    tt = torch.as_tensor(toks, device=out.device)
    assert_close(out[tt], lse[tt], *ref, tag=f"{name} ({len(toks)} of {wl.T} tokens)")
    assert torch.isfinite(out).all()
    assert binding.get_error_word() == 0
