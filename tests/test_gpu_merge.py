"""attn_merge_partials on the GPU against the oracle's merge, including the
-inf identity rows, in-place use, and an end-to-end check that merging the
partials of two key halves reproduces whole attention."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


def _partials(B, H, S, d, seed):
    g = torch.Generator().manual_seed(seed)
    o_a = torch.randn(B, H, S, d, generator=g)
    o_b = torch.randn(B, H, S, d, generator=g)
    l_a = torch.randn(B, H, S, generator=g) * 5
    l_b = torch.randn(B, H, S, generator=g) * 5
    # identity rows: one side, the other side, both
    l_a[..., 0] = -float("inf"); o_a[..., 0, :] = 0
    l_b[..., 1] = -float("inf"); o_b[..., 1, :] = 0
    l_a[..., 2] = l_b[..., 2] = -float("inf"); o_a[..., 2, :] = 0; o_b[..., 2, :] = 0
    return o_a, l_a, o_b, l_b


@pytest.mark.parametrize("B,H,S,d", [(1, 2, 300, 128), (2, 3, 129, 64), (1, 1, 5, 3), (1, 4, 1000, 1)])
def test_merge_matches_oracle(ra, B, H, S, d):
    o_a, l_a, o_b, l_b = _partials(B, H, S, d, 7 + d)
    o_ref, l_ref = oracle.merge(f64(o_a), f64(l_a), f64(o_b), f64(l_b))
    o, l = ra.attn_merge_partials(*(x.cuda() for x in (o_a, l_a, o_b, l_b)))
    assert ra.check_status() == 0
    np.testing.assert_allclose(f64(o), o_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(f64(l), l_ref, rtol=0, atol=1e-5)
    # identity rows reproduce the other side exactly
    assert torch.equal(o[..., 0, :].cpu(), o_b[..., 0, :]) and torch.equal(l[..., 0].cpu(), l_b[..., 0])
    assert torch.equal(o[..., 1, :].cpu(), o_a[..., 1, :]) and torch.equal(l[..., 1].cpu(), l_a[..., 1])
    assert (o[..., 2, :] == 0).all() and torch.isneginf(l[..., 2]).all()


def test_merge_in_place(ra):
    o_a, l_a, o_b, l_b = _partials(1, 2, 257, 128, 3)
    o_ref, l_ref = oracle.merge(f64(o_a), f64(l_a), f64(o_b), f64(l_b))
    a, la = o_a.cuda(), l_a.cuda()
    ra.attn_merge_partials(a, la, o_b.cuda(), l_b.cuda(), o_out=a, lse_out=la)
    np.testing.assert_allclose(f64(a), o_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(f64(la), l_ref, atol=1e-5)


def test_merge_of_key_halves_is_whole_attention(ra):
    # Partials over two key halves (oracle, fp64 -> fp32) merged on the GPU
    # equal attention over all keys.
    inp = workloads.make(workloads.FWD_PEAKED_64K, B=1, H=2, S=512, P=2)
    q, k, v = (f64(inp[x]) for x in ("q", "k", "v"))
    S, d, sc = 512, inp["d"], inp["scale"]
    parts = []
    for c0 in (0, 256):
        o_p = np.empty((1, 2, S, d)); l_p = np.empty((1, 2, S))
        for h in range(2):
            o_p[0, h], l_p[0, h] = oracle.partial(q[0, h], 0, k[0, h, c0:c0 + 256],
                                                  v[0, h, c0:c0 + 256], c0, False, sc)
        parts.append((torch.from_numpy(o_p).float().cuda(), torch.from_numpy(l_p).float().cuda()))
    o, l = ra.attn_merge_partials(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    o_ref, l_ref = oracle.naive_fwd(q, k, v, False, sc)
    np.testing.assert_allclose(f64(o), o_ref, atol=2e-5)
    np.testing.assert_allclose(f64(l), l_ref, atol=2e-5)


def test_merge_large_rows(ra):
    # many rows: the grid-stride loop covers rows beyond one wave
    B, H, S, d = 2, 16, 8192, 128
    o_a, l_a, o_b, l_b = (x.cuda() for x in _partials(B, H, S, d, 11))
    o, l = ra.attn_merge_partials(o_a, l_a, o_b, l_b)
    rows = torch.randint(0, B * H * S, (512,), generator=torch.Generator().manual_seed(1))
    oa = f64(o_a.reshape(-1, d)[rows.cuda()]); ob = f64(o_b.reshape(-1, d)[rows.cuda()])
    la = f64(l_a.reshape(-1)[rows.cuda()]); lb = f64(l_b.reshape(-1)[rows.cuda()])
    o_ref, l_ref = oracle.merge(oa, la, ob, lb)
    np.testing.assert_allclose(f64(o.reshape(-1, d)[rows.cuda()]), o_ref, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(f64(l.reshape(-1)[rows.cuda()]), l_ref, atol=1e-5)
