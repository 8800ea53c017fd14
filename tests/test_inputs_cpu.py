"""The seeded input generator: the row format it writes and the shapes of the
workloads (host-only checks; the arithmetic is pinned in test_oracle.py)."""
import numpy as np
import torch

from sparse_mla_attention_03_gb300 import inputs


def _rows(kv):
    return kv.numpy().reshape(-1, 656)


def test_e4m3_rows_have_no_nan_codes_and_power_of_two_scales():
    wl = inputs.make_prefill("gen", T=2, H=4, ctx=256, topk=32, seed=1)
    r = _rows(wl.kv)
    assert not np.any((r[:, :512] & 0x7F) == 0x7F)  # satfinite: no NaN codes
    sc = np.ascontiguousarray(r[:, 512:528]).view("<f4")
    m, e = np.frexp(sc)
    assert np.all(m == 0.5) and np.all(sc > 0)  # powers of two


def test_arbitrary_scales_and_int8_codes():
    r = _rows(inputs.make_prefill("gen", T=2, H=4, ctx=256, topk=32, seed=2, scales="any").kv)
    sc = np.ascontiguousarray(r[:, 512:528]).view("<f4")
    assert np.any(np.frexp(sc)[0] != 0.5)  # not all powers of two
    r8 = _rows(inputs.make_prefill("gen", T=2, H=4, ctx=256, topk=32, seed=3, kv_format="int8").kv)
    codes = r8[:, :512].view(np.int8)
    assert codes.min() >= -127 and codes.max() <= 127
    assert np.any(codes == 127) or np.any(codes == -127)  # each block's max maps to +-127


def test_nope_layout_pads_the_rope_bytes():
    wl = inputs.make_prefill("gen", T=2, H=4, ctx=128, topk=16, seed=4, layout="nope")
    assert wl.q.shape[2] == 512 and np.all(_rows(wl.kv)[:, 528:] == 0xFF)


def test_indices_unique_and_in_range():
    wl = inputs.make_prefill("gen", T=5, H=4, ctx=1024, topk=300, seed=5, ld=400)
    idx = wl.indices.numpy()
    assert np.all(idx[:, 300:] == inputs.POISON)
    for row in idx[:, :300]:
        assert len(set(row.tolist())) == 300 and row.min() >= 0 and row.max() < 1024


def test_dual_generators():
    wl = inputs.make_dual_prefill("gen", T=4, H=8, ctx=256, topk=70, extra_ctx=128, extra_topk=40, seed=6,
                                  ragged=True)
    assert wl.dual and wl.extra_indices.shape == (4, 40) and wl.extra_kv.shape == (2, 64, 656)
    for lens, idx, k in ((wl.topk_length, wl.indices, 70), (wl.extra_topk_length, wl.extra_indices, 40)):
        lens, idx = lens.numpy(), idx.numpy()
        assert np.all((lens >= 0) & (lens <= k))
        cols = np.arange(k)[None, :]
        assert np.all(idx[cols >= lens[:, None]] == -1) and np.all(idx[cols < lens[:, None]] >= 0)
    wd = inputs.make_dual_decode("gen", n_req=2, tokens_per_req=2, H=8, ctx_per_req=256, topk=40,
                                 extra_ctx_per_req=128, extra_topk=30, seed=7)
    bt2 = wd.extra_block_table.numpy()
    assert sorted(bt2.ravel().tolist()) == list(range(wd.extra_kv.shape[0]))  # a permutation of the pages
    assert torch.all(wd.extra_indices < 128)
