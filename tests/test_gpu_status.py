"""Bounded waits: a valid run under a tiny wait limit either completes or
ends early with RA_ERR_DEVICE_TIMEOUT -- it never hangs -- and the library
stays usable afterwards.  Nothing here faults the GPU: the kernels run on
valid inputs and only their time limit is shortened."""
import pytest
import torch

import oracle
import workloads
from _parity import assert_o_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


def test_tiny_wait_limit_reports_or_completes(ra):
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=1, H=4, S=8192, P=4, seed=2)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    assert ra.check_status() == 0
    try:
        ra.set_wait_limit_ns(1)
        o, lse = ra.ring_attn_fwd(q, k, v, 4, True, inp["scale"])
        st_fwd = ra.check_status()
        ra.ring_attn_bwd(q, k, v, o, lse, do, 4, True, inp["scale"])
        st_bwd = ra.check_status()
    finally:
        ra.set_wait_limit_ns(0)
    assert st_fwd in (ra.RA_OK, ra.RA_ERR_DEVICE_TIMEOUT)
    assert st_bwd in (ra.RA_OK, ra.RA_ERR_DEVICE_TIMEOUT)
    # with the default limit a fresh run is correct again
    o, lse = ra.ring_attn_fwd(q, k, v, 4, True, inp["scale"])
    assert ra.check_status() == ra.RA_OK
    rows = workloads.sample_rows(1, 4, 8192, 4, n_random=32, heads=[0, 3]).numpy()
    o_ref, _ = oracle.naive_fwd_rows(f64(q), f64(k), f64(v), True, inp["scale"], rows)
    assert_o_close(f64(o).reshape(-1, 128)[rows], o_ref)
