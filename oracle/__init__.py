"""Float64 CPU oracle for sparse-MLA decode.

TEST INFRASTRUCTURE ONLY.  This package is the independent checker that the
CUDA path is compared against.  Only the test suite, the package smoke check
and the benchmark's CPU-baseline leg may import it; the library itself never
does, and it shares no code, tables or constants with the CUDA sources.

See ``smla_oracle`` for what is computed and which passage each step follows.
"""
from .smla_oracle import (  # noqa: F401
    E4M3_TABLE,
    PAGE_SIZE,
    bf16_bits_to_f64,
    dequant_entries,
    decode,
    decode_row,
    e4m3_decode,
    merge_partials,
    partial_row,
    plan_cost,
    plan_num_splits,
    row_entries,
    ue8m0_scale,
)
