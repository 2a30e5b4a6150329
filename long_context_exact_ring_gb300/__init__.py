"""Exact ring attention for one GB300 (sm_103a): a C-ABI CUDA library
(libringattn.so, include/ring_attn.h) and its thin Python binding.

    from long_context_exact_ring_gb300 import ring_attn_fwd, ring_attn_bwd
    o, lse = ring_attn_fwd(q, k, v, P=4, causal=True)
    dq, dk, dv = ring_attn_bwd(q, k, v, o, lse, dO, P=4, causal=True)

Torch is used for device memory and streams only; every step runs in the
library's kernels.  Build the library with
``python -m long_context_exact_ring_gb300.build``.
"""
from ._binding import (  # noqa: F401
    EXPORTED,
    LIB_PATH,
    RA_ERR_CUDA,
    RA_ERR_DEVICE_TIMEOUT,
    RA_ERR_INVALID_ARG,
    RA_ERR_UNSUPPORTED,
    RA_OK,
    RingAttnError,
    attn_merge_partials,
    bwd_workspace_size,
    check_status,
    load_library,
    profile_enable,
    profile_read,
    profile_reset,
    ring_attn_bwd,
    ring_attn_bwd_noalloc,
    NOALLOC_SCRATCH_BYTES,
    ring_attn_fwd,
    ring_attn_fwd_emulated,
    emulated_workspace_size,
    ring_attn_fwd_f32,
    fwd_f32_workspace_size,
    ring_attn_fwd_ulysses_emulated,
    ulysses_workspace_size,
    ring_schedule,
    set_wait_limit_ns,
    status_string,
    trace_visits,
)
