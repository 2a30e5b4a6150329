"""Forward parity on the GPU: the CUDA path through the C ABI against the
fp64 oracle on identical seeded bf16 inputs.

Small shapes are compared element by element over whole tensors (several
tiles per chunk, ragged chunk tails, P = 1, causal and not, d = 64 and 128).
The 32K causal workload is compared over every element of every head; the
larger workloads run in the same launch configuration the benchmark times
and are compared on sampled rows (row 0, first/last rows of every chunk and
their neighbours, seeded random rows) of a few heads.
"""
import math

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


def _run(ra, inp):
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o, lse = ra.ring_attn_fwd(q, k, v, inp["P"], inp["causal"], inp["scale"])
    assert ra.check_status() == 0
    return q, k, v, o, lse


SMALL = [
    # B, H, S,    d,   P, causal
    (1, 2, 1024, 128, 4, True),
    (1, 2, 1024, 128, 4, False),
    (2, 3, 768, 64, 3, True),       # C = 256
    (1, 2, 1000, 128, 4, True),     # C = 250: ragged tiles in every chunk
    (1, 2, 1000, 64, 8, False),     # C = 125: chunks shorter than a tile
    (1, 1, 384, 128, 1, False),     # P = 1: plain attention
    (1, 1, 384, 128, 1, True),
    (1, 2, 640, 64, 5, True),       # C = 128: one query tile per chunk
    (1, 1, 200, 128, 8, True),      # C = 25
    (2, 2, 2048, 128, 8, False),
    (1, 1, 1, 64, 1, True),         # a single token
    (1, 1, 17, 128, 1, False),
]


@pytest.mark.parametrize("B,H,S,d,P,causal", SMALL)
def test_fwd_small_whole_tensor(ra, B, H, S, d, P, causal):
    inp = workloads.make(workloads.FWD_CAUSAL_32K, B=B, H=H, S=S, d=d, P=P, causal=causal,
                         seed=100 + S + d + P)
    q, k, v, o, lse = _run(ra, inp)
    o_ref, lse_ref, log = oracle.ring_fwd(f64(q), f64(k), f64(v), P, causal, inp["scale"])
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)


def test_fwd_tiny_workload(ra):
    w = workloads.TINY_F32
    inp = workloads.make(w)
    q, k, v, o, lse = _run(ra, inp)
    # the GPU takes the bf16 rounding of the fp32 draws; so does the oracle here
    o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), w.causal, w.scale)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)


def test_fwd_peaked_keys_small(ra):
    # every 64th key row x8: peaked rows that force the running max to move
    inp = workloads.make(workloads.FWD_PEAKED_64K, B=1, H=2, S=4096, P=8)
    q, k, v, o, lse = _run(ra, inp)
    o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), False, inp["scale"])
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)


def test_fwd_large_scores_rescale(ra):
    # scores that grow along the sequence make the running max rise tile
    # after tile, so the O rescale path runs on every tile
    B, H, S, d, P = 1, 1, 2048, 128, 4
    g = torch.Generator().manual_seed(5)
    q = torch.randn(B, H, S, d, generator=g)
    k = torch.randn(B, H, S, d, generator=g) * torch.linspace(0.1, 4.0, S).view(1, 1, S, 1)
    v = torch.randn(B, H, S, d, generator=g)
    q, k, v = (x.to(torch.bfloat16).cuda() for x in (q, k, v))
    for causal in (False, True):
        o, lse = ra.ring_attn_fwd(q, k, v, P, causal, 1.0 / math.sqrt(d))
        o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), causal, 1.0 / math.sqrt(d))
        assert_o_close(f64(o), o_ref)
        assert_lse_close(f64(lse), lse_ref)


def test_fwd_matches_unchunked_for_every_P(ra):
    # exactness: the ring result does not depend on P (beyond rounding)
    inp = workloads.make(workloads.FWD_CAUSAL_32K, B=1, H=2, S=2048, d=128, seed=9)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), True, inp["scale"])
    for P in (1, 2, 4, 8, 16):
        o, lse = ra.ring_attn_fwd(q, k, v, P, True, inp["scale"])
        assert_o_close(f64(o), o_ref, f"O P={P}")
        assert_lse_close(f64(lse), lse_ref, f"LSE P={P}")


def test_fwd_rejects_bad_shapes(ra):
    q = torch.zeros(1, 1, 256, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RingAttnError) as e:
        ra.ring_attn_fwd(q, q, q, 4, True)
    assert e.value.status == ra.RA_ERR_UNSUPPORTED
    q = torch.zeros(1, 1, 250, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RingAttnError) as e:
        ra.ring_attn_fwd(q, q, q, 4, True)
    assert e.value.status == ra.RA_ERR_INVALID_ARG


def test_fwd_empty_is_noop(ra):
    q = torch.zeros(1, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = ra.ring_attn_fwd(q, q, q, 4, True)
    assert o.numel() == 0 and lse.numel() == 0


def _sampled(ra, w, heads, n_random=192):
    inp = workloads.make(w, keep_fp32=False)
    q, k, v, o, lse = _run(ra, inp)
    B, H, S, P, d = inp["B"], inp["H"], inp["S"], inp["P"], inp["d"]
    local = workloads.sample_rows(1, 1, S, P, n_random=n_random).numpy()
    for bh in heads:
        b, h = divmod(bh, H)
        # the oracle sees one head at a time, widened to fp64
        qh, kh, vh = (f64(x[b:b + 1, h:h + 1]) for x in (q, k, v))
        o_ref, lse_ref = oracle.naive_fwd_rows(qh, kh, vh, inp["causal"], inp["scale"], local)
        assert_o_close(f64(o[b, h])[local], o_ref, f"O head {bh}")
        assert_lse_close(f64(lse[b, h])[local], lse_ref, f"LSE head {bh}")
    # no row anywhere may be non-finite
    assert torch.isfinite(lse).all() and torch.isfinite(o.float()).all()


@pytest.mark.slow
def test_fwd_causal_32k_whole_tensor(ra):
    # B=1, H=32, S=32768, d=128, P=4, causal: every element of O and LSE of
    # every head against the definition (row blocks, fp64, one head at a time)
    w = workloads.FWD_CAUSAL_32K
    inp = workloads.make(w, keep_fp32=False)
    q, k, v, o, lse = _run(ra, inp)
    for h in range(w.H):
        qh, kh, vh = (f64(x[0:1, h:h + 1]) for x in (q, k, v))
        o_ref, lse_ref = oracle.naive_fwd_blocked(qh, kh, vh, True, inp["scale"], block=512)
        assert_o_close(f64(o[0:1, h:h + 1]), o_ref, f"O head {h}")
        assert_lse_close(f64(lse[0:1, h:h + 1]), lse_ref, f"LSE head {h}")


@pytest.mark.slow
def test_fwd_causal_128k_sampled(ra):
    w = workloads.FWD_CAUSAL_128K
    _sampled(ra, w, heads=[0, w.B * w.H - 1], n_random=96)


@pytest.mark.slow
def test_fwd_peaked_64k_sampled(ra):
    w = workloads.FWD_PEAKED_64K
    _sampled(ra, w, heads=[0, w.B * w.H - 1], n_random=96)
