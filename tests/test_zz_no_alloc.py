"""The decode entry point that allocates nothing (sparse_mla_decode_noalloc).

Some callers cannot allocate device memory -- a host engine that owns all
device memory through its own pool and hands a library only tensors and a
stream, or a latency-critical path that cannot take an allocation's implicit
synchronisation.  For them the library keeps the decode's split partials in a
fixed array compiled into it.  This file checks, through the C ABI, that two
calls in a row give the same results as the workspace-taking
sparse_mla_decode (within the parity tolerances of the other tests), and that
a request too large for the array is refused with a clear error.  It is named
so that pytest collects it last.
"""
import pytest
import torch

from sparse_mla_attention_03_gb300 import binding, inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu


def _dev(wl):
    return {k: (None if getattr(wl, k) is None else getattr(wl, k).cuda())
            for k in ("q", "kv", "indices", "topk_length", "attn_sink", "block_table")}


def _both(wl, num_splits):
    d = _dev(wl)
    kw = dict(topk=wl.topk, topk_length=d["topk_length"], attn_sink=d["attn_sink"],
              block_table=d["block_table"], tokens_per_req=wl.tokens_per_req, num_splits=num_splits)
    ref = binding.sparse_mla_decode(d["q"], d["kv"], d["indices"], wl.sm_scale, **kw)
    out = torch.empty_like(ref[0])
    lse = torch.empty_like(ref[1])
    got = binding.sparse_mla_decode_noalloc(d["q"], d["kv"], d["indices"], wl.sm_scale, out=out, lse=lse, **kw)
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_decode_matches_workspace_decode_twice(cuda_lib):
    a = inputs.make_decode("noalloc_a", n_req=8, tokens_per_req=2, H=64, ctx_per_req=8192, topk=1024, seed=7)
    b = inputs.make_prefill("noalloc_b", T=12, H=8, ctx=4096, topk=640, seed=8, ragged=True)
    for wl, s in ((a, 4), (b, 3)):  # two calls in a row, different shapes and contents
        ref, got = _both(wl, s)
        assert_close(got[0], got[1], ref[0].double().cpu().numpy(), ref[1].double().cpu().numpy(),
                     tag=f"noalloc {wl.name}")


def test_noalloc_single_split_needs_no_scratch(cuda_lib):
    # one split writes the outputs directly: a size whose partials would not
    # fit the built-in array still runs, and matches the workspace decode
    wl = inputs.make_prefill("noalloc_s1", T=512, H=64, ctx=2048, topk=2048, seed=10)
    assert binding.decode_workspace_size(wl.T, wl.H, wl.topk, 1) > binding.noalloc_scratch_bytes()
    ref, got = _both(wl, 1)
    assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])


def test_noalloc_rejects_requests_beyond_the_array(cuda_lib):
    wl = inputs.make_prefill("noalloc_big", T=512, H=64, ctx=2048, topk=2048, seed=9, sink=None)
    need = binding.decode_workspace_size(wl.T, wl.H, wl.topk, 8)
    assert need > binding.noalloc_scratch_bytes()
    d = _dev(wl)
    with pytest.raises(binding.SparseMLAError) as ei:
        binding.sparse_mla_decode_noalloc(d["q"], d["kv"], d["indices"], wl.sm_scale, num_splits=8)
    assert ei.value.code == binding.SMLA_ERR_INVALID
    assert "scratch" in str(ei.value)


def test_noalloc_automatic_split_count(cuda_lib):
    # num_splits = 0: the automatic choice (here more than one split, so the
    # partials go through the built-in array) -- lowered to fit the array if
    # it ever needed more; on 152 SMs the automatic choice stays well within it
    wl = inputs.make_decode("noalloc_auto", n_req=16, tokens_per_req=2, H=128, ctx_per_req=8192, topk=2048, seed=11)
    s = binding.decode_num_splits(wl.T, wl.H, wl.topk, 0)
    assert s > 1 and binding.decode_workspace_size(wl.T, wl.H, wl.topk, 0) <= binding.noalloc_scratch_bytes()
    for _ in range(2):
        ref, got = _both(wl, 0)
        assert_close(got[0], got[1], ref[0].double().cpu().numpy(), ref[1].double().cpu().numpy(),
                     tag="noalloc automatic splits")
