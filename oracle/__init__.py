"""fp64 CPU oracle for exact ring attention -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never does, and
this package imports nothing from it.
"""
from .oracle import (  # noqa: F401
    KIND_FULL,
    KIND_LOCAL,
    KIND_SKIP,
    build_oracle,
    merge,
    naive_fwd,
    naive_fwd_rows,
    ring_fwd,
    ring_visits,
    partial,
    bwd,
    bwd_dq_rows,
    bwd_dkdv_rows,
    bwd_bf16_rounding_model,
    naive_fwd_blocked,
    naive_fwd_gqa,
    naive_fwd_rows_gqa,
    bwd_gqa,
    ring_step_bytes,
    ring_total_bytes,
    kv_cache_bytes_per_token,
    score_matrix_elements,
    attention_flops,
)
