"""Strided row layouts on the GPU: [B, S, H, d] storage (the layout most
training code keeps), padded rows, and mixtures of layouts, passed as
views whose d-element rows are contiguous.

The layout only changes where rows are read and written, so the forward
outputs and dK / dV must be bit-identical to the contiguous call on the same
values.  dQ is summed by fp32 reduce-adds from many key tiles whose order
is not fixed even between two contiguous calls, so it is compared within
one bf16 rounding step of the contiguous result and against the oracle."""
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


def as_layout(x: torch.Tensor, layout: str) -> torch.Tensor:
    """The values of contiguous [B, heads, S, d] x as a view over storage in
    `layout`: bhsd (contiguous), bshd ([B, S, heads, d]), pad (rows of d + 8
    elements), bshd_pad ([B, S, heads, d + 16])."""
    B, Hh, S, d = x.shape
    if layout == "bhsd":
        return x.clone()
    if layout == "bshd":
        st = torch.empty((B, S, Hh, d), dtype=x.dtype, device=x.device)
        st.copy_(x.transpose(1, 2))
        return st.transpose(1, 2)
    if layout == "pad":
        st = torch.full((B, Hh, S, d + 8), float("nan"), dtype=x.dtype, device=x.device)
        st[..., :d].copy_(x)
        return st[..., :d]
    if layout == "bshd_pad":
        st = torch.full((B, S, Hh, d + 16), float("nan"), dtype=x.dtype, device=x.device)
        st[..., :d].copy_(x.transpose(1, 2))
        return st[..., :d].transpose(1, 2)
    raise ValueError(layout)


def empty_layout(like: torch.Tensor, layout: str) -> torch.Tensor:
    return as_layout(torch.zeros_like(like), layout).fill_(float("nan"))


def assert_dq_close(got, want):
    # dQ is a sum of fp32 partials, one per key tile, whose reduce order
    # differs between calls: the two results may differ by one bf16 rounding
    # step, plus the reordering error of the fp32 sum itself, which is what
    # remains for a sum near zero -- at most ~n eps32 sum |partial|, i.e.
    # 1024 partials of size <= 1 at the 128K shape: 1024 * 2^-24 = 2^-14
    g, w = got.float(), want.float()
    bound = 2.0 ** -7 * torch.maximum(g.abs(), w.abs()) + 2.0 ** -14
    bad = (g - w).abs() > bound
    assert not bool(bad.any()), f"dQ differs beyond one bf16 step at {int(bad.sum())} elements"


CASES = [
    # B, H, H_kv, S,   d,   P, causal, layout of q, k, v, o / grads
    (1, 4, 4, 1024, 128, 4, True, ("bshd", "bshd", "bshd", "bshd")),
    (2, 4, 4, 768, 64, 3, False, ("bshd", "bshd", "bshd", "bshd")),
    (1, 4, 4, 1200, 128, 3, True, ("bshd", "bhsd", "pad", "bshd_pad")),   # ragged chunk tails, mixed
    (1, 8, 2, 1024, 128, 4, True, ("bshd", "bshd", "bshd", "bshd")),       # grouped-query
    (2, 6, 3, 512, 64, 2, True, ("pad", "bshd_pad", "bshd", "bhsd")),
]


@pytest.mark.parametrize("B,H,Hkv,S,d,P,causal,lay", CASES)
def test_strided_equals_contiguous(ra, B, H, Hkv, S, d, P, causal, lay):
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=B, H=H, H_kv=Hkv, S=S, d=d, P=P,
                         causal=causal, seed=900 + S + H, keep_fp32=False)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    sc = inp["scale"]
    o_c, lse_c = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    dq_c, dk_c, dv_c = ra.ring_attn_bwd(q, k, v, o_c, lse_c, do, P, causal, sc)

    lq, lk, lv, lout = lay
    qs, ks, vs = as_layout(q, lq), as_layout(k, lk), as_layout(v, lv)
    os_ = empty_layout(q, lout)
    o_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, P, causal, sc, o=os_)
    assert o_s.data_ptr() == os_.data_ptr()
    dos = as_layout(do, lout)
    dq_s, dk_s, dv_s = ra.ring_attn_bwd(qs, ks, vs, o_s, lse_s, dos, P, causal, sc,
                                        dq=empty_layout(q, lout), dk=empty_layout(k, lout),
                                        dv=empty_layout(v, lout))
    assert ra.check_status() == ra.RA_OK
    assert torch.equal(o_s, o_c), "O differs from the contiguous call"
    assert torch.equal(lse_s, lse_c), "LSE differs from the contiguous call"
    assert torch.equal(dk_s, dk_c), "dK differs from the contiguous call"
    assert torch.equal(dv_s, dv_c), "dV differs from the contiguous call"
    assert_dq_close(dq_s, dq_c)
    if "pad" in lout:
        # the padding columns of the output storage were never written
        assert torch.isnan(os_._base[..., d:].float()).all()


def test_bshd_matches_oracle_and_keeps_layout(ra):
    B, H, S, d, P = 1, 2, 1024, 128, 4
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=B, H=H, S=S, d=d, P=P, seed=31,
                         keep_fp32=False)
    q, k, v, do = (as_layout(inp[x].cuda(), "bshd") for x in ("q", "k", "v", "do"))
    sc = inp["scale"]
    o, lse = ra.ring_attn_fwd(q, k, v, P, True, sc)
    assert o.stride() == q.stride(), "o should default to q's layout"
    dq, dk, dv = ra.ring_attn_bwd(q, k, v, o, lse, do, P, True, sc)
    assert dq.stride() == q.stride() and dk.stride() == k.stride()
    assert ra.check_status() == ra.RA_OK
    o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), True, sc)
    assert_o_close(f64(o), o_ref)
    assert_lse_close(f64(lse), lse_ref)
    dq_r, dk_r, dv_r, _, _ = oracle.bwd(f64(q), f64(k), f64(v), f64(do), True, sc)
    assert_grad_close(f64(dq), dq_r, "dQ")
    assert_grad_close(f64(dk), dk_r, "dK")
    assert_grad_close(f64(dv), dv_r, "dV")


def test_bad_row_stride_is_rejected(ra):
    # rows of d + 4 elements: the row stride is not a multiple of 16 bytes
    q = torch.zeros((1, 2, 256, 132), dtype=torch.bfloat16, device="cuda")[..., :128]
    with pytest.raises(Exception) as e:
        ra.ring_attn_fwd(q, q, q, 2, True, 0.1)
    assert "INVALID_ARG" in str(e.value)


@pytest.mark.slow
def test_bshd_full_size_four_dim_maps(ra):
    # B = 2 with [B, S, H, d] storage: batch and head cannot share a stride,
    # so every Q / K / V / dO load goes through the 4-D tensor maps -- at the
    # peaked workload's full size (2 x 16 heads x 65536 tokens, P = 8)
    w = workloads.FWD_PEAKED_64K
    inp = workloads.make(w, device="cuda", keep_fp32=False, backward=True)
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    P, causal, sc = inp["P"], inp["causal"], inp["scale"]
    o_c, lse_c = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    dq_c, dk_c, dv_c = ra.ring_attn_bwd(q, k, v, o_c, lse_c, do, P, causal, sc)
    qs, ks, vs, dos = (as_layout(x, "bshd") for x in (q, k, v, do))
    del q, k, v, do
    o_s, lse_s = ra.ring_attn_fwd(qs, ks, vs, P, causal, sc)
    dq_s, dk_s, dv_s = ra.ring_attn_bwd(qs, ks, vs, o_s, lse_s, dos, P, causal, sc)
    assert ra.check_status() == ra.RA_OK
    assert o_s.stride() == qs.stride()
    assert torch.equal(o_s, o_c) and torch.equal(lse_s, lse_c)
    assert torch.equal(dk_s, dk_c) and torch.equal(dv_s, dv_c)
    assert_dq_close(dq_s, dq_c)
