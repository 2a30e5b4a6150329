"""The Ulysses layout path on one GPU (P logical ranks, two all-to-alls,
full-sequence attention per head group) against the oracle and against the
fused kernel run as a single chunk: every head's attention is computed by
the same kernel over the same keys in the same order, so the two must agree
bit for bit; the all-to-alls only move rows."""
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
    # B, H, H_kv, S,   d,   P, causal
    (1, 4, 4, 1024, 128, 4, True),
    (2, 4, 4, 768, 64, 2, False),
    (1, 8, 4, 1024, 128, 4, True),       # grouped-query, H_kv = P
    (1, 6, 3, 1200, 128, 3, True),       # ragged tiles, P = 3
    (2, 2, 2, 512, 64, 1, True),         # one rank: no exchange
]


@pytest.mark.parametrize("B,H,Hkv,S,d,P,causal", CASES)
def test_ulysses_equals_single_chunk_and_oracle(ra, B, H, Hkv, S, d, P, causal):
    inp = workloads.make(workloads.FWDBWD_GQA_128K, B=B, H=H, H_kv=Hkv, S=S, d=d, P=P,
                         causal=causal, seed=700 + S + H, keep_fp32=False)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    sc = inp["scale"]
    k0, v0 = k.clone(), v.clone()
    o_u, lse_u = ra.ring_attn_fwd_ulysses_emulated(q, k, v, P, causal, sc)
    o_1, lse_1 = ra.ring_attn_fwd(q, k, v, 1, causal, sc)
    o_r, lse_r = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    assert ra.check_status() == ra.RA_OK
    assert torch.equal(o_u, o_1) and torch.equal(lse_u, lse_1), "differs from the single-chunk call"
    assert torch.equal(k, k0) and torch.equal(v, v0), "inputs were modified"
    if Hkv == H:
        o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), causal, sc)
    else:
        o_ref, lse_ref = oracle.naive_fwd_gqa(f64(q), f64(k), f64(v), causal, sc)
    assert_o_close(f64(o_u), o_ref)
    assert_lse_close(f64(lse_u), lse_ref)
    # the ring with P chunks computes the same attention (order of keys differs)
    assert_o_close(f64(o_r), f64(o_u), "ring vs Ulysses")


def test_ulysses_needs_whole_heads_per_rank(ra):
    inp = workloads.make(workloads.FWDBWD_GQA_128K, B=1, H=8, H_kv=2, S=1024, P=4, seed=3,
                         keep_fp32=False)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    with pytest.raises(Exception) as e:       # 2 key/value heads cannot feed 4 ranks
        ra.ring_attn_fwd_ulysses_emulated(q, k, v, 4, True)
    assert "UNSUPPORTED" in str(e.value)


def test_ulysses_128k_sampled_rows(ra):
    # the 128K causal shape at P = 4 (32 heads, 8 per rank), sampled rows vs the oracle
    w = workloads.FWD_CAUSAL_128K
    inp = workloads.make(w, keep_fp32=False)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = ra.ring_attn_fwd_ulysses_emulated(q, k, v, inp["P"], inp["causal"], inp["scale"])
    assert ra.check_status() == ra.RA_OK
    rows = workloads.sample_rows(1, 1, inp["S"], inp["P"], n_random=64).numpy()
    for h in (0, 13, 31):
        qh, kh, vh = (f64(x[0:1, h:h + 1]) for x in (q, k, v))
        o_ref, lse_ref = oracle.naive_fwd_rows(qh, kh, vh, inp["causal"], inp["scale"], rows)
        assert_o_close(f64(o[0, h])[rows], o_ref.reshape(len(rows), -1), f"O head {h}")
        assert_lse_close(f64(lse[0, h])[rows], lse_ref.reshape(-1), f"LSE head {h}")
