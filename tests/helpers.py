"""Shared test helpers: device transfer, oracle calls on sampled tokens, tolerances."""
import numpy as np
import torch

import oracle.sparse_mla_oracle as O

# Tolerances on out (bf16) and lse (fp32) against the fp64 oracle.
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def to_dev(wl, device="cuda"):
    d = {}
    for k in ("q", "kv", "indices", "topk_length", "attn_sink", "block_table", "extra_kv", "extra_indices",
              "extra_topk_length", "extra_block_table"):
        v = getattr(wl, k)
        d[k] = None if v is None else v.to(device)
    return d


def oracle_dual_for(wl, tokens=None):
    """The dual-cache oracle on all tokens, or on ``tokens`` only."""
    sel = None if tokens is None else np.asarray(tokens)
    q = wl.q.to(torch.float64).numpy() if sel is None else wl.q[torch.as_tensor(sel)].to(torch.float64).numpy()
    np_ = lambda x: None if x is None else x.numpy()
    return O.sparse_mla_forward_dual(
        q, wl.kv.numpy(), wl.indices.numpy(), wl.topk, wl.extra_kv.numpy(), wl.extra_indices.numpy(),
        wl.extra_topk, wl.sm_scale, topk_length=np_(wl.topk_length), extra_topk_length=np_(wl.extra_topk_length),
        attn_sink=None if wl.attn_sink is None else wl.attn_sink.numpy().astype(np.float64),
        block_table=np_(wl.block_table), extra_block_table=np_(wl.extra_block_table),
        tokens_per_req=wl.tokens_per_req, tokens=sel, q_selected=sel is not None, kv_format=wl.kv_format,
        layout=wl.layout)


def oracle_for(wl, tokens=None, indices=None, topk=None, topk_length="wl", attn_sink="wl"):
    q = wl.q.to(torch.float64).numpy() if tokens is None else wl.q[torch.as_tensor(tokens)].to(torch.float64).numpy()
    idx = (wl.indices if indices is None else indices).numpy()
    tl = wl.topk_length if topk_length == "wl" else topk_length
    sk = wl.attn_sink if attn_sink == "wl" else attn_sink
    bt = None if wl.block_table is None else wl.block_table.numpy()
    sel = None if tokens is None else np.asarray(tokens)
    return O.sparse_mla_forward(q, wl.kv.numpy(), idx, topk or wl.topk, wl.sm_scale,
                                topk_length=None if tl is None else tl.numpy(),
                                attn_sink=None if sk is None else sk.numpy().astype(np.float64),
                                block_table=bt, tokens_per_req=wl.tokens_per_req, tokens=sel,
                                q_selected=sel is not None, kv_format=wl.kv_format, layout=wl.layout)


def assert_close(out_gpu, lse_gpu, out_ref, lse_ref, tag=""):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    assert o.shape == out_ref.shape, (o.shape, out_ref.shape)
    assert np.isfinite(o).all(), f"{tag}: non-finite outputs"
    err = np.abs(o - out_ref)
    assert err.max() <= OUT_MAX_ABS, f"{tag}: out max_abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{tag}: out mean_abs {err.mean():.3e}"
    ninf_g, ninf_r = np.isneginf(l), np.isneginf(lse_ref)
    assert np.array_equal(ninf_g, ninf_r), f"{tag}: -inf LSE pattern differs"
    if (~ninf_r).any():
        le = np.abs(l[~ninf_r] - lse_ref[~ninf_r])
        assert le.max() <= LSE_ABS, f"{tag}: lse max_abs {le.max():.3e}"
    return float(err.max()), float(err.mean())


def sample_tokens_by_quarter(T, n, seed=0, must=()):
    """A seeded sample of about ``n`` distinct tokens of ``range(T)``: n/4 from
    each quarter of the range (all of them when T <= n), plus ``must``."""
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    pick = set(int(x) for x in must if 0 <= x < T)
    bounds = [q * T // 4 for q in range(5)]
    for q in range(4):
        lo, hi = bounds[q], bounds[q + 1]
        pick.update(int(x) for x in lo + rng.choice(hi - lo, size=min(n // 4, hi - lo), replace=False))
    return np.array(sorted(pick))
