"""GB300-native sparse MLA attention forward (prefill and decode).

The compute path is the C-ABI library ``libsparse_mla.so`` (hand-written sm_103a
CUDA, declared in ``include/sparse_mla.h``); ``binding`` is a thin ctypes layer
over it.  Importing this package does not load the library; the first call does,
and fails loudly if it is missing.
"""
from .binding import (  # noqa: F401
    SparseMLAError, decode_workspace_size, load, sparse_mla_decode, sparse_mla_prefill,
    sparse_mla_resolve_rows,
)
