"""Test infrastructure only: the float64 CPU oracle for absorbed-form MLA split-KV decode.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (the C-ABI library and its Python binding)
never imports, calls or links anything here, and this package imports nothing from
the product path.
"""
from .mla_ref import (  # noqa: F401
    LATENT_DIM,
    ROPE_DIM,
    CACHE_DIM,
    decode_bf16,
    decode_e4m3,
    decode_e2m1,
    nvfp4_page_bytes,
    dequant_pages,
    gather_tokens,
    visible_len,
    window_range,
    mla_decode_ref,
    mla_decode_one,
    mla_partial_ref,
    combine_ref,
    mla_decode_split_ref,
    forced_split_ranges,
    E4M3_TABLE,
    E2M1_TABLE,
    next_power_of_2,
    cdiv,
    tilegym_split_heuristic,
    workspace_bytes_formula,
)
