"""The ring protocol emulated with P logical ranks on one GPU
(ring_attn_fwd_emulated): per-step partials on the compute stream, K/V
rotation to the next rank on a copy stream, LSE merge of every step.
Compared with the oracle's literal ring (fp64) and with the fused
forward, with the rotation overlapped and serialized."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


CASES = [
    # B, H, S,    d,   P, causal
    (1, 2, 1024, 128, 4, True),
    (1, 2, 1024, 128, 4, False),
    (2, 2, 768, 64, 3, True),
    (1, 2, 1000, 128, 8, True),     # C = 125: chunks shorter than a tile
    (1, 1, 512, 128, 1, True),      # P = 1: no rotation
    (1, 2, 2048, 128, 2, False),
]


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("B,H,S,d,P,causal", CASES)
def test_emulated_ring_matches_oracle(ra, B, H, S, d, P, causal, overlap):
    inp = workloads.make(workloads.FWD_CAUSAL_32K, B=B, H=H, S=S, d=d, P=P, causal=causal,
                         seed=500 + S + P, keep_fp32=False)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = ra.ring_attn_fwd_emulated(q, k, v, P, causal, inp["scale"], overlap=overlap)
    assert ra.check_status() == ra.RA_OK
    o_ref, lse_ref, _ = oracle.ring_fwd(f64(q), f64(k), f64(v), P, causal, inp["scale"])
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)
    # and the fused ring on the same inputs
    o2, lse2 = ra.ring_attn_fwd(q, k, v, P, causal, inp["scale"])
    assert (o.float() - o2.float()).abs().max().item() <= 2e-2
    assert (lse - lse2).abs().max().item() <= 1e-4


def test_emulated_ring_repeat_and_inputs_untouched(ra):
    # the receive buffers rotate copies; the caller's K and V stay as given,
    # and a second call on the same workspace gives the same result
    inp = workloads.make(workloads.FWD_CAUSAL_32K, H=2, S=2048, P=4, seed=77, keep_fp32=False)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    k0, v0 = k.clone(), v.clone()
    ws = torch.empty(ra.emulated_workspace_size(1, 2, 2048, 128), dtype=torch.uint8, device="cuda")
    a = ra.ring_attn_fwd_emulated(q, k, v, 4, True, inp["scale"], workspace=ws)
    b = ra.ring_attn_fwd_emulated(q, k, v, 4, True, inp["scale"], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(k, k0) and torch.equal(v, v0)


@pytest.mark.slow
def test_emulated_ring_128k_sampled(ra):
    w = workloads.FWD_CAUSAL_128K
    inp = workloads.make(w, keep_fp32=False)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = ra.ring_attn_fwd_emulated(q, k, v, w.P, True, inp["scale"])
    o2, lse2 = ra.ring_attn_fwd(q, k, v, w.P, True, inp["scale"])
    assert ra.check_status() == ra.RA_OK
    assert (o.float() - o2.float()).abs().max().item() <= 2e-2
    assert (lse - lse2).abs().max().item() <= 1e-4
    local = workloads.sample_rows(1, 1, w.S, w.P, n_random=32).numpy()
    for h in (0, w.H - 1):
        o_ref, lse_ref = oracle.naive_fwd_rows(f64(q[0:1, h:h + 1]), f64(k[0:1, h:h + 1]),
                                               f64(v[0:1, h:h + 1]), True, inp["scale"], local)
        assert_o_close(f64(o[0, h])[local], o_ref)
        assert_lse_close(f64(lse[0, h])[local], lse_ref)
