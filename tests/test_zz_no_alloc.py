"""ring_attn_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (a host framework that owns every device allocation through
its own pool, or a path where cudaMalloc / cudaFree would block or
synchronize the device).  The library's fixed static scratch replaces the
caller's workspace.

Called here directly through the C ABI, twice in a row (the scratch keeps
the previous call's contents, so the second call checks that what must
start at zero is cleared), and compared with ring_attn_bwd -- which takes a
caller-owned workspace -- within the gradient tolerance of the other tests.
This file is collected last so a failure here comes after every other test.
"""
import ctypes

import pytest
import torch

import workloads
from _parity import assert_grad_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


def _noalloc(lib, q, k, v, o, lse, do, dq, dk, dv, P, causal, scale):
    B, H, S, d = q.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.ring_attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr(), B, H, S, d, P, int(causal), ctypes.c_float(scale),
                                     ctypes.c_void_p(stream))


@pytest.mark.parametrize("S,P,causal", [(1024, 4, True), (1200, 3, False)])
def test_noalloc_matches_workspace_entry_point_twice(ra, S, P, causal):
    lib = ra.load_library()
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=1, H=2, S=S, P=P, causal=causal, seed=21,
                         keep_fp32=False)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    sc = inp["scale"]
    o, lse = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    ref = ra.ring_attn_bwd(q, k, v, o, lse, do, P, causal, sc)
    assert ra.check_status() == ra.RA_OK
    for call in range(2):
        outs = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = _noalloc(lib, q, k, v, o, lse, do, *outs, P, causal, sc)
        assert rc == ra.RA_OK, f"call {call}: {ra.status_string(rc)}"
        assert ra.check_status() == ra.RA_OK
        for got, want, name in zip(outs, ref, ("dQ", "dK", "dV")):
            assert_grad_close(f64(got), f64(want), f"{name} (call {call})")


def test_noalloc_rejects_shapes_beyond_the_scratch(ra):
    lib = ra.load_library()
    # 64 heads x 4096 tokens at d = 128 needs ~136 MB of workspace > 64 MiB;
    # the call returns before touching any pointer.
    fake = 1 << 20
    rc = lib.ring_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                   1, 64, 4096, 128, 4, 1, ctypes.c_float(0.088), None)
    assert rc == ra.RA_ERR_UNSUPPORTED
    assert ra.bwd_workspace_size(1, 64, 4096, 128) > ra.NOALLOC_SCRATCH_BYTES
    assert ra.bwd_workspace_size(1, 32, 4096, 128) > ra.NOALLOC_SCRATCH_BYTES
    assert ra.bwd_workspace_size(1, 16, 8064, 128) <= ra.NOALLOC_SCRATCH_BYTES
