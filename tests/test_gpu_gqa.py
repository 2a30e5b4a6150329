"""Grouped-query attention on the GPU against the oracle (MHA on K/V
repeated for each query head's group; shared K/V gradients summed over the
group).  Whole tensors at small shapes; sampled rows at the 128K grouped
shape (32 query heads over 8 key/value heads)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import assert_grad_close, assert_lse_close, assert_o_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


CASES = [
    # B, H, H_kv, S,   d,   P, causal
    (1, 4, 2, 1024, 128, 4, True),
    (1, 4, 1, 1024, 128, 4, False),     # multi-query
    (2, 6, 3, 768, 64, 3, True),
    (1, 8, 2, 1000, 128, 4, True),      # ragged chunk tails
    (1, 4, 4, 512, 128, 2, True),       # one member per group: plain multi-head
]


@pytest.mark.parametrize("B,H,Hkv,S,d,P,causal", CASES)
def test_gqa_fwd_bwd_whole_tensor(ra, B, H, Hkv, S, d, P, causal):
    inp = workloads.make(workloads.FWDBWD_GQA_128K, B=B, H=H, H_kv=Hkv, S=S, d=d, P=P,
                         causal=causal, seed=400 + S + H + Hkv, keep_fp32=False)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    assert k.shape[1] == Hkv
    sc = inp["scale"]
    o, lse = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, o, lse, do, P, causal, sc)
    assert ra.check_status() == ra.RA_OK
    assert dk.shape == k.shape and dv.shape == v.shape
    o_ref, lse_ref = oracle.naive_fwd_gqa(f64(q), f64(k), f64(v), causal, sc)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)
    dq_r, dk_r, dv_r = oracle.bwd_gqa(f64(q), f64(k), f64(v), f64(do), causal, sc)
    assert_grad_close(f64(dq), dq_r, "dQ")
    assert_grad_close(f64(dk), dk_r, "dK")
    assert_grad_close(f64(dv), dv_r, "dV")


def test_gqa_group_equals_repeated_heads_on_gpu(ra):
    # The grouped call equals the multi-head call on explicitly repeated K/V,
    # with dK/dV summed over each group.
    inp = workloads.make(workloads.FWDBWD_GQA_128K, H=8, H_kv=2, S=1024, seed=17, keep_fp32=False)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    sc, P = inp["scale"], inp["P"]
    o, lse = ra.ring_attn_fwd(q, k, v, P, True, sc)
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, o, lse, do, P, True, sc)
    kr, vr = (x.repeat_interleave(4, dim=1).contiguous() for x in (k, v))
    o2, lse2 = ra.ring_attn_fwd(q, kr, vr, P, True, sc)
    dq2, dk2, dv2 = ra.ring_attn_bwd(q, kr, vr, o2, lse2, do, P, True, sc)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert (dq.float() - dq2.float()).abs().max().item() <= 1e-2
    dk2s = dk2.float().view(1, 2, 4, 1024, 128).sum(2)
    dv2s = dv2.float().view(1, 2, 4, 1024, 128).sum(2)
    assert (dk.float() - dk2s).abs().max().item() <= 5e-2
    assert (dv.float() - dv2s).abs().max().item() <= 5e-2


@pytest.mark.slow
def test_gqa_128k_sampled(ra):
    w = workloads.FWDBWD_GQA_128K
    inp = workloads.make(w, keep_fp32=False)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    sc, P, S, H, Hkv = inp["scale"], inp["P"], inp["S"], inp["H"], inp["H_kv"]
    o, lse = ra.ring_attn_fwd(q, k, v, P, True, sc)
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, o, lse, do, P, True, sc)
    assert ra.check_status() == ra.RA_OK
    local = workloads.sample_rows(1, 1, S, P, n_random=48).numpy()
    G = H // Hkv
    for h in (0, G, H - 1):
        hk = h // G
        qh, dh = f64(q[0:1, h:h + 1]), f64(do[0:1, h:h + 1])
        kh, vh = f64(k[0:1, hk:hk + 1]), f64(v[0:1, hk:hk + 1])
        o_ref, lse_ref = oracle.naive_fwd_rows(qh, kh, vh, True, sc, local)
        assert_o_close(f64(o[0, h])[local], o_ref, f"O head {h}")
        assert_lse_close(f64(lse[0, h])[local], lse_ref, f"LSE head {h}")
        dq_r, _ = oracle.bwd_dq_rows(qh, kh, vh, dh, True, sc, local)
        assert_grad_close(f64(dq[0, h])[local], dq_r, f"dQ head {h}")
    # sum over keys of dV = sum over the group's query rows of dO; of dK = 0
    dv_sum = dv.float().sum(dim=2)
    do_sum = do.float().view(1, Hkv, G, S, 128).sum(dim=(2, 3))
    ref = do.float().abs().sum(dim=2).max().item() * G
    assert (dv_sum - do_sum).abs().max().item() <= 1e-2 * ref
    assert dk.float().sum(dim=2).abs().max().item() <= 1e-2 * ref
