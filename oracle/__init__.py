"""Scalar CPU oracle for the W12 format and the skinny GEMM (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and it never touches them.
"""
from .oracle import (  # noqa: F401
    build,
    lib_path,
    encode,
    blob_header,
    decode,
    decode_rows,
    decode_q8,
    gemm,
    gemm_rows,
    abs_gemm,
    row_ebase,
    num_tiles,
    b_row_bytes,
    round_bf16,
    i8_quantize,
    gemm_i8,
    abs_gemm_i8,
    silu_mul,
    TILE_ROWS,
    TILE_COLS,
)
