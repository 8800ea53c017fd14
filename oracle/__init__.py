"""CPU oracle (test infrastructure only; see sparse_mla_oracle's header)."""
from .sparse_mla_oracle import (  # noqa: F401
    D_NOPE, D_QK, D_ROPE, D_V, PAGE_BLOCK, ROW_BYTES, attend_one, bf16_bits_to_f64,
    decode_rows, e4m3_to_f64, f32_le_bytes_to_f64, merge_partials, resolve_rows,
    sparse_mla_forward, split_partials,
)
