"""CPU float64 oracle (test infrastructure; never used by the product path)."""
from .mla_oracle import (  # noqa: F401
    E4M3_TABLE, UE8M0_TABLE, attend, bf16_bits_to_float, combine, dequantize_rows,
    e4m3_to_float, sparse_mla_decode, split_partials, split_ranges, ue8m0_to_float,
    weighted_deviation,
)
