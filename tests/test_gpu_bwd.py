"""Backward parity on the GPU against the oracle's plain derivative.

Whole tensors at small shapes (several tiles, ragged chunk tails, causal and
not, d = 64 and 128) and at S = 4096.  At the full 128K causal size, in the
benchmark's launch configuration: sampled dQ, dK and dV rows of two heads
against the oracle element by element, every LSE row of those heads, plus
properties that hold at any size (sum_c dV_c = sum_r dO_r, sum_c dK_c = 0).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import assert_grad_close, assert_grad_close_model, assert_grad_max, assert_lse_close, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


def _fwd_bwd(ra, inp):
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    P, causal, sc = inp["P"], inp["causal"], inp["scale"]
    o, lse = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, o, lse, do, P, causal, sc)
    assert ra.check_status() == 0
    return q, k, v, do, o, lse, dq, dk, dv


SMALL = [
    # B, H, S,    d,   P, causal
    (1, 2, 1024, 128, 4, True),
    (1, 2, 1024, 128, 4, False),
    (2, 2, 768, 64, 3, True),
    (1, 2, 1000, 128, 4, True),     # ragged chunk tails (C = 250: rows read from global)
    (1, 2, 1200, 128, 4, True),     # ragged tails with C % 4 == 0 (C = 300: rows by TMA)
    (1, 1, 1200, 64, 3, False),     # C = 400
    (1, 1, 1000, 64, 8, False),     # chunks shorter than a tile
    (1, 1, 384, 128, 1, True),      # P = 1
    (1, 1, 200, 128, 8, True),
    (1, 1, 1, 128, 1, False),
]


@pytest.mark.parametrize("B,H,S,d,P,causal", SMALL)
def test_bwd_small_whole_tensor(ra, B, H, S, d, P, causal):
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=B, H=H, S=S, d=d, P=P, causal=causal,
                         seed=300 + S + d + P)
    q, k, v, do, o, lse, dq, dk, dv = _fwd_bwd(ra, inp)
    # the oracle differentiates the exact attention of the same bf16 inputs
    dq_r, dk_r, dv_r, _, _ = oracle.bwd(f64(q), f64(k), f64(v), f64(do), causal, inp["scale"])
    assert_grad_max(f64(dq), dq_r, "dQ")
    assert_grad_max(f64(dk), dk_r, "dK")
    assert_grad_max(f64(dv), dv_r, "dV")


def test_bwd_peaked_keys(ra):
    # stress input (keys c % 64 == 0 scaled x8, V ~ U(-1, 1)): gradients
    # reach ~20, and bf16 storage of O, P, dS and the outputs alone misses
    # the exact derivative by up to ~0.09; the bound adds that model error
    w = workloads.FWD_PEAKED_64K
    inp = workloads.make(w, B=1, H=2, S=2048, P=8, backward=True)
    q, k, v, do, o, lse, dq, dk, dv = _fwd_bwd(ra, inp)
    args = (f64(q), f64(k), f64(v), f64(do), False, inp["scale"])
    dq_r, dk_r, dv_r, _, _ = oracle.bwd(*args)
    mq, mk, mv = oracle.bwd_bf16_rounding_model(*args)
    assert_grad_close_model(f64(dq), dq_r, mq, "dQ")
    assert_grad_close_model(f64(dk), dk_r, mk, "dK")
    assert_grad_close_model(f64(dv), dv_r, mv, "dV")


def test_bwd_repeatable_workspace_reuse(ra):
    # the dQ accumulator is cleared by every call: two calls, same answer
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=1, H=2, S=1024, P=4, seed=8)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = ra.ring_attn_fwd(q, k, v, 4, True, inp["scale"])
    ws = torch.empty(ra.bwd_workspace_size(1, 2, 1024, 128), dtype=torch.uint8, device="cuda")
    ws.fill_(0x7f)
    a = ra.ring_attn_bwd(q, k, v, o, lse, do, 4, True, inp["scale"], workspace=ws)
    b = ra.ring_attn_bwd(q, k, v, o, lse, do, 4, True, inp["scale"], workspace=ws)
    for x, y in zip(a, b):
        assert (x.float() - y.float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("d,P,causal", [(128, 4, True), (64, 4, True), (128, 8, False)])
def test_bwd_s4096_whole_tensor(ra, d, P, causal):
    # the 128K fwd+bwd recipe at S = 4096 (P = 4, C = 1024: eight key tiles
    # per chunk), every element of dQ, dK and dV against the plain derivative;
    # d = 64 takes the other shared-memory plan (dS in a buffer of its own,
    # the whole dQ tile in the staging buffer); the non-causal case with
    # P = 8 has every key tile meet all eight query chunks
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=1, H=2, S=4096, d=d, P=P, causal=causal, seed=44)
    q, k, v, do, o, lse, dq, dk, dv = _fwd_bwd(ra, inp)
    dq_r, dk_r, dv_r, _, _ = oracle.bwd(f64(q), f64(k), f64(v), f64(do), causal, inp["scale"])
    assert_grad_max(f64(dq), dq_r, "dQ")
    assert_grad_max(f64(dk), dk_r, "dK")
    assert_grad_max(f64(dv), dv_r, "dV")


@pytest.mark.slow
def test_bwd_causal_128k_sampled_rows(ra):
    # The full fwd+bwd workload (B=1, H=32, S=131072, d=128, P=4, causal), in
    # the benchmark's launch configuration.  For heads 0 and H-1, at sampled
    # positions (0, S-1, the first and last rows of every chunk and their
    # neighbours, 48 seeded random ones), element by element:
    #   dQ rows      -- oracle.bwd_dq_rows (LSE_r and D_r per sampled row);
    #   dK, dV rows  -- oracle.bwd_dkdv_rows, which takes LSE_r and D_r of
    #                   every query row r >= c of the head from the definition;
    #   LSE          -- every row of the head, from the same pass.
    w = workloads.FWDBWD_CAUSAL_128K
    inp = workloads.make(w, keep_fp32=False)
    q, k, v, do, o, lse, dq, dk, dv = _fwd_bwd(ra, inp)
    H, S, d, P, sc = inp["H"], inp["S"], inp["d"], inp["P"], inp["scale"]
    local = workloads.sample_rows(1, 1, S, P, n_random=48).numpy()
    for bh in (0, H - 1):
        qh, kh, vh, dh = (f64(x[0:1, bh:bh + 1]) for x in (q, k, v, do))
        dq_r, _ = oracle.bwd_dq_rows(qh, kh, vh, dh, True, sc, local)
        assert_grad_max(f64(dq[0, bh])[local], dq_r, f"dQ head {bh}")
        dk_r, dv_r, lse_r, _ = oracle.bwd_dkdv_rows(qh, kh, vh, dh, True, sc, local, block=512)
        assert_grad_max(f64(dk[0, bh])[local], dk_r, f"dK head {bh}")
        assert_grad_max(f64(dv[0, bh])[local], dv_r, f"dV head {bh}")
        assert_lse_close(f64(lse[0, bh]), lse_r, f"LSE head {bh}")
    # properties over every head: rows of P sum to 1 and sum_c dS_rc = 0
    dv_sum = dv.float().sum(dim=2)
    do_sum = do.float().sum(dim=2)
    dk_sum = dk.float().sum(dim=2)
    scale_ref = do.float().abs().sum(dim=2).max().item()
    assert (dv_sum - do_sum).abs().max().item() <= 1e-2 * scale_ref
    assert dk_sum.abs().max().item() <= 1e-2 * scale_ref
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
