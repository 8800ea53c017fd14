"""Thin ctypes binding over libsparse_mla.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor shapes/dtypes/devices, fills the ``smla_args`` struct of
``include/sparse_mla.h`` with raw device pointers and strides, and passes the
current torch stream.  PyTorch only provides device memory and streams.  If
the library is missing, every call raises ``SparseMLAError``: there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsparse_mla.so")
D_QK, D_V, ROW_BYTES, PAGE = 576, 512, 656, 64

SMLA_OK, SMLA_ERR_INVALID, SMLA_ERR_UNSUPPORTED, SMLA_ERR_CUDA, SMLA_ERR_DEVICE = range(5)
KV_FORMATS = {"e4m3": 0, "int8": 1}  # SMLA_KV_E4M3, SMLA_KV_INT8
LAYOUTS = {"rope64": 0, "nope": 1}  # SMLA_LAYOUT_ROPE64, SMLA_LAYOUT_NOPE
ERRF_INDEX_RANGE, ERRF_TIMEOUT, ERRF_SCALE_RANGE = 1, 2, 4


class SparseMLAError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"sparse_mla error {code}: {msg}")
        self.code = code


class SmlaArgs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_stride_t", ctypes.c_int64),
        ("kv", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64),
        ("bt_rows", ctypes.c_int32), ("bt_cols", ctypes.c_int32),
        ("tokens_per_req", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("indices", ctypes.c_void_p), ("idx_stride_t", ctypes.c_int64),
        ("topk_length", ctypes.c_void_p), ("attn_sink", ctypes.c_void_p),
        ("sm_scale", ctypes.c_float), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
        ("kv_format", ctypes.c_int32),
        ("out", ctypes.c_void_p), ("out_stride_t", ctypes.c_int64),
        ("lse", ctypes.c_void_p), ("lse_stride_t", ctypes.c_int64),
        ("layout", ctypes.c_int32), ("reserved1", ctypes.c_int32),
    ]


class SmlaExtraArgs(ctypes.Structure):
    """The second list and cache of the dual-cache form (``smla_extra_args``)."""
    _fields_ = [
        ("kv", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64),
        ("bt_rows", ctypes.c_int32), ("bt_cols", ctypes.c_int32),
        ("topk", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("indices", ctypes.c_void_p), ("idx_stride_t", ctypes.c_int64),
        ("topk_length", ctypes.c_void_p),
    ]


# (name, restype, argtypes) for every symbol of include/sparse_mla.h
_P = ctypes.POINTER(SmlaArgs)
_X = ctypes.POINTER(SmlaExtraArgs)
SYMBOLS = {
    "sparse_mla_prefill": (ctypes.c_int, [_P, ctypes.c_void_p]),
    "sparse_mla_decode": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "sparse_mla_decode_workspace_size": (ctypes.c_size_t, [ctypes.c_int32] * 4),
    "sparse_mla_decode_num_splits": (ctypes.c_int32, [ctypes.c_int32] * 4),
    "sparse_mla_plan_num_splits": (ctypes.c_int32, [ctypes.c_int32] * 5 + [ctypes.c_int64]),
    "sparse_mla_resolve_rows": (ctypes.c_int, [_P, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
    "sparse_mla_decode_noalloc": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_void_p]),
    "sparse_mla_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "sparse_mla_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "sparse_mla_set_test_stall": (ctypes.c_int32, [ctypes.c_int32]),
    "sparse_mla_get_error_word": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "sparse_mla_last_error": (ctypes.c_char_p, []),
    "sparse_mla_abi_version": (ctypes.c_int32, []),
    "sparse_mla_dual_width": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32]),
    "sparse_mla_prefill_dual": (ctypes.c_int, [_P, _X, ctypes.c_void_p]),
    "sparse_mla_decode_dual": (ctypes.c_int, [_P, _X, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                              ctypes.c_void_p]),
    "sparse_mla_resolve_rows_dual": (ctypes.c_int, [_P, _X, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]),
}

_lib = None
_lock = threading.Lock()


def load(path: Optional[str] = None):
    """Load libsparse_mla.so (raises SparseMLAError if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise SparseMLAError(-1, f"{p} is not built; run sparse_mla_attention_03_gb300.build.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SYMBOLS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _check(rc):
    if rc != SMLA_OK:
        msg = load().sparse_mla_last_error().decode(errors="replace")
        raise SparseMLAError(rc, msg)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def make_args(q, kv, indices, topk, sm_scale, out, lse, topk_length=None, attn_sink=None,
              block_table=None, tokens_per_req=1, kv_format="e4m3", layout="rope64") -> SmlaArgs:
    """Validate tensor layouts and build the C struct (no data is touched)."""
    T, H = q.shape[0], q.shape[1]
    dev = q.device

    def on_dev(x, name, dtype):
        if x is None:
            return
        if x.device != dev:
            raise ValueError(f"{name} is on {x.device}, q is on {dev}")
        if x.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {x.dtype}")

    on_dev(q, "q", torch.bfloat16)
    on_dev(kv, "kv", torch.uint8)
    on_dev(indices, "indices", torch.int32)
    on_dev(out, "out", torch.bfloat16)
    on_dev(lse, "lse", torch.float32)
    on_dev(topk_length, "topk_length", torch.int32)
    on_dev(attn_sink, "attn_sink", torch.float32)
    on_dev(block_table, "block_table", torch.int32)
    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(LAYOUTS)}, got {layout!r}")
    d_qk = D_QK if layout == "rope64" else D_V
    if q.dim() != 3 or q.shape[2] != d_qk or q.stride(2) != 1 or q.stride(1) != d_qk:
        raise ValueError(f"q must be [T, H, {d_qk}] with head stride {d_qk} and unit last stride")
    if kv.dim() != 3 or tuple(kv.shape[1:]) != (PAGE, ROW_BYTES) or not kv.is_contiguous():
        raise ValueError("kv must be a contiguous [num_pages, 64, 656] uint8 tensor")
    if indices.dim() != 2 or indices.shape[0] != T or indices.stride(1) != 1 or indices.shape[1] < topk:
        raise ValueError("indices must be [T, >= topk] with a contiguous last dimension")
    if out.shape != (T, H, D_V) or out.stride(2) != 1 or out.stride(1) != D_V:
        raise ValueError("out must be [T, H, 512] with head stride 512 and unit last stride")
    if lse.shape != (T, H) or lse.stride(1) != 1:
        raise ValueError("lse must be [T, H] with unit last stride")
    if topk_length is not None and (topk_length.shape != (T,) or topk_length.stride(0) != 1):
        raise ValueError("topk_length must be a contiguous [T] tensor")
    if attn_sink is not None and (attn_sink.shape != (H,) or attn_sink.stride(0) != 1):
        raise ValueError("attn_sink must be a contiguous [H] tensor")
    a = SmlaArgs()
    a.q, a.q_stride_t = q.data_ptr(), q.stride(0)
    a.kv, a.num_pages = kv.data_ptr(), kv.shape[0]
    if block_table is not None:
        if block_table.dim() != 2 or block_table.stride(1) != 1:
            raise ValueError("block_table must be [B, max_pages] with a contiguous last dimension")
        a.block_table = block_table.data_ptr()
        a.bt_stride = block_table.stride(0)
        a.bt_rows, a.bt_cols = block_table.shape
        a.tokens_per_req = int(tokens_per_req)
    a.topk = int(topk)
    a.indices, a.idx_stride_t = indices.data_ptr(), indices.stride(0)
    a.topk_length = _ptr(topk_length)
    a.attn_sink = _ptr(attn_sink)
    a.sm_scale = float(sm_scale)
    a.T, a.H = T, H
    a.out, a.out_stride_t = out.data_ptr(), out.stride(0)
    a.lse, a.lse_stride_t = lse.data_ptr(), lse.stride(0)
    if kv_format not in KV_FORMATS:
        raise ValueError(f"kv_format must be one of {sorted(KV_FORMATS)}, got {kv_format!r}")
    a.kv_format = KV_FORMATS[kv_format]
    a.layout = LAYOUTS[layout]
    return a


def _outputs(q, out, lse):
    T, H = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    return out, lse


def sparse_mla_prefill(q, kv, indices, sm_scale, topk=None, topk_length=None, attn_sink=None,
                       block_table=None, tokens_per_req=1, out=None, lse=None, stream=None,
                       kv_format="e4m3", layout="rope64"):
    """Sparse MLA prefill; returns ``(out bf16 [T,H,512], lse fp32 [T,H])``."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    out, lse = _outputs(q, out, lse)
    a = make_args(q, kv, indices, topk, sm_scale, out, lse, topk_length, attn_sink, block_table,
                  tokens_per_req, kv_format, layout)
    _check(lib.sparse_mla_prefill(ctypes.byref(a), _stream_handle(stream)))
    return out, lse


def decode_workspace_size(T, H, topk, num_splits=0) -> int:
    return int(load().sparse_mla_decode_workspace_size(T, H, topk, num_splits))


def decode_num_splits(T, H, topk, num_splits=0) -> int:
    return int(load().sparse_mla_decode_num_splits(T, H, topk, num_splits))


def plan_num_splits(T, H, topk, num_splits, num_sms, l2_bytes) -> int:
    """The split count for a device with ``num_sms`` SMs and ``l2_bytes`` of L2 (host only)."""
    return int(load().sparse_mla_plan_num_splits(T, H, topk, num_splits, num_sms, l2_bytes))


def sparse_mla_decode(q, kv, indices, sm_scale, topk=None, topk_length=None, attn_sink=None,
                      block_table=None, tokens_per_req=1, num_splits=0, workspace=None, out=None,
                      lse=None, stream=None,
                       kv_format="e4m3", layout="rope64"):
    """Split-K sparse MLA decode plus combine; returns ``(out, lse)``.

    ``workspace``: a uint8 CUDA tensor of at least ``decode_workspace_size``
    bytes (allocated here through torch when omitted)."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    out, lse = _outputs(q, out, lse)
    a = make_args(q, kv, indices, topk, sm_scale, out, lse, topk_length, attn_sink, block_table,
                  tokens_per_req, kv_format, layout)
    need = decode_workspace_size(q.shape[0], q.shape[1], topk, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.sparse_mla_decode(ctypes.byref(a), int(num_splits), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream_handle(stream)))
    return out, lse


def noalloc_scratch_bytes() -> int:
    """Size of the no-alloc decode's built-in array, read from the library."""
    return int(load().sparse_mla_noalloc_scratch_bytes())


def set_wait_limit_ns(ns: int) -> int:
    """Limit of every bounded in-kernel wait of later calls; returns the previous one."""
    return int(load().sparse_mla_set_wait_limit_ns(int(ns)))


def set_test_stall(on: bool) -> bool:
    """Test hook: the tcgen05 kernel's producers gather nothing (its waits run out); returns the previous setting."""
    return bool(load().sparse_mla_set_test_stall(1 if on else 0))



def sparse_mla_decode_noalloc(q, kv, indices, sm_scale, topk=None, topk_length=None, attn_sink=None,
                              block_table=None, tokens_per_req=1, num_splits=0, out=None, lse=None,
                              stream=None,
                       kv_format="e4m3", layout="rope64"):
    """Split-K decode whose partials live in the library's built-in scratch
    array: for callers that cannot allocate device memory.  ``out``/``lse``
    must be passed to allocate nothing here either."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    out, lse = _outputs(q, out, lse)
    a = make_args(q, kv, indices, topk, sm_scale, out, lse, topk_length, attn_sink, block_table,
                  tokens_per_req, kv_format, layout)
    _check(lib.sparse_mla_decode_noalloc(ctypes.byref(a), int(num_splits), _stream_handle(stream)))
    return out, lse


def sparse_mla_resolve_rows(q, kv, indices, topk=None, topk_length=None, block_table=None,
                            tokens_per_req=1, stream=None,
                       kv_format="e4m3", layout="rope64"):
    """Physical cache row per slot (int32 [T, topk], -1 = invalid), from the device."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    T, H = q.shape[0], q.shape[1]
    out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    rows = torch.empty((T, topk), dtype=torch.int32, device=q.device)
    a = make_args(q, kv, indices, topk, 1.0, out, lse, topk_length, None, block_table, tokens_per_req,
                  kv_format, layout)
    _check(lib.sparse_mla_resolve_rows(ctypes.byref(a), rows.data_ptr(), topk, _stream_handle(stream)))
    return rows


def get_error_word(stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(load().sparse_mla_get_error_word(_stream_handle(stream), ctypes.byref(v)))
    return int(v.value)


# ----------------------------------------------------------------------------- dual-cache form
def make_extra(q, kv, indices, topk=None, topk_length=None, block_table=None) -> SmlaExtraArgs:
    """Validate the second list / cache of the dual-cache form and build its struct."""
    T = q.shape[0]
    dev = q.device
    topk = indices.shape[1] if topk is None else topk
    for x, name, dtype in ((kv, "extra kv", torch.uint8), (indices, "extra indices", torch.int32),
                           (topk_length, "extra topk_length", torch.int32),
                           (block_table, "extra block_table", torch.int32)):
        if x is None:
            continue
        if x.device != dev:
            raise ValueError(f"{name} is on {x.device}, q is on {dev}")
        if x.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if kv.dim() != 3 or tuple(kv.shape[1:]) != (PAGE, ROW_BYTES) or not kv.is_contiguous():
        raise ValueError("extra kv must be a contiguous [num_pages, 64, 656] uint8 tensor")
    if indices.dim() != 2 or indices.shape[0] != T or indices.stride(1) != 1 or indices.shape[1] < topk:
        raise ValueError("extra indices must be [T, >= topk] with a contiguous last dimension")
    if topk_length is not None and (topk_length.shape != (T,) or topk_length.stride(0) != 1):
        raise ValueError("extra topk_length must be a contiguous [T] tensor")
    x = SmlaExtraArgs()
    x.kv, x.num_pages = kv.data_ptr(), kv.shape[0]
    if block_table is not None:
        if block_table.dim() != 2 or block_table.stride(1) != 1:
            raise ValueError("extra block_table must be [B, max_pages] with a contiguous last dimension")
        x.block_table = block_table.data_ptr()
        x.bt_stride = block_table.stride(0)
        x.bt_rows, x.bt_cols = block_table.shape
    x.topk = int(topk)
    x.indices, x.idx_stride_t = indices.data_ptr(), indices.stride(0)
    x.topk_length = _ptr(topk_length)
    return x


def dual_width(topk, extra_topk) -> int:
    """Combined slots per token of the dual-cache form."""
    return int(load().sparse_mla_dual_width(int(topk), int(extra_topk)))


def sparse_mla_prefill_dual(q, kv, indices, extra_kv, extra_indices, sm_scale, topk=None, topk_length=None,
                            extra_topk=None, extra_topk_length=None, attn_sink=None, block_table=None,
                            extra_block_table=None, tokens_per_req=1, out=None, lse=None, stream=None,
                       kv_format="e4m3", layout="rope64"):
    """One softmax over two index lists into two caches; returns ``(out, lse)``."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    out, lse = _outputs(q, out, lse)
    a = make_args(q, kv, indices, topk, sm_scale, out, lse, topk_length, attn_sink, block_table,
                  tokens_per_req, kv_format, layout)
    a.tokens_per_req = int(tokens_per_req)
    x = make_extra(q, extra_kv, extra_indices, extra_topk, extra_topk_length, extra_block_table)
    _check(lib.sparse_mla_prefill_dual(ctypes.byref(a), ctypes.byref(x), _stream_handle(stream)))
    return out, lse


def sparse_mla_decode_dual(q, kv, indices, extra_kv, extra_indices, sm_scale, topk=None, topk_length=None,
                           extra_topk=None, extra_topk_length=None, attn_sink=None, block_table=None,
                           extra_block_table=None, tokens_per_req=1, num_splits=0, workspace=None,
                           out=None, lse=None, stream=None,
                       kv_format="e4m3", layout="rope64"):
    """Split-K decode of the dual-cache form plus combine; returns ``(out, lse)``."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    out, lse = _outputs(q, out, lse)
    a = make_args(q, kv, indices, topk, sm_scale, out, lse, topk_length, attn_sink, block_table,
                  tokens_per_req, kv_format, layout)
    a.tokens_per_req = int(tokens_per_req)
    x = make_extra(q, extra_kv, extra_indices, extra_topk, extra_topk_length, extra_block_table)
    need = decode_workspace_size(q.shape[0], q.shape[1], dual_width(topk, x.topk), num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(lib.sparse_mla_decode_dual(ctypes.byref(a), ctypes.byref(x), int(num_splits), workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(), _stream_handle(stream)))
    return out, lse


def sparse_mla_resolve_rows_dual(q, kv, indices, extra_kv, extra_indices, topk=None, topk_length=None,
                                 extra_topk=None, extra_topk_length=None, block_table=None,
                                 extra_block_table=None, tokens_per_req=1, stream=None,
                       kv_format="e4m3", layout="rope64"):
    """Row per combined slot (int32 [T, width]); second-cache rows are offset
    by the first cache's row count; -1 = invalid or padding."""
    lib = load()
    topk = indices.shape[1] if topk is None else topk
    T, H = q.shape[0], q.shape[1]
    out = torch.empty((T, H, D_V), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    a = make_args(q, kv, indices, topk, 1.0, out, lse, topk_length, None, block_table, tokens_per_req,
                  kv_format, layout)
    a.tokens_per_req = int(tokens_per_req)
    x = make_extra(q, extra_kv, extra_indices, extra_topk, extra_topk_length, extra_block_table)
    width = dual_width(topk, x.topk)
    rows = torch.empty((T, width), dtype=torch.int32, device=q.device)
    _check(lib.sparse_mla_resolve_rows_dual(ctypes.byref(a), ctypes.byref(x), rows.data_ptr(), width,
                                            _stream_handle(stream)))
    return rows
