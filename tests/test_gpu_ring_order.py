"""The ring order the kernels really follow, bit-exact against the oracle's
schedule ("Context Parallelism" guide, section 2, "How It Works": at ring
step t query chunk i meets KV chunk j = (i - t) mod P; causal attention
skips chunks j > i).

With recording on (ring_attn_trace_visits), every CTA's TMA producer writes
each chunk its tile stream enters, in order.  Forward CTAs (one per query
chunk and 256-row pair of query tiles) must list exactly the oracle's
non-skipped visits of their query chunk, with the tile counts of chunk-level
and diagonal-tile skipping; backward CTAs (one per key tile) must list the
inverse -- the query chunks that meet their key chunk, by ring step.
Recording is off in the timed path; the last test checks that it is off by
default and after it is turned off.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TILE = 128          # keys (forward) and queries (backward) per tile
FWD_ROWS = 256      # query rows per forward CTA
SENTINEL = -777


@pytest.fixture(scope="module")
def ra():
    import long_context_exact_ring_gb300 as m
    from long_context_exact_ring_gb300 import build
    build.build()
    return m


def _expected_fwd(P, causal, i):
    return [(t, j, kind) for t, j, kind in oracle.ring_visits(P, causal, i) if kind != oracle.KIND_SKIP]


def _expected_bwd(P, causal, j):
    # the inverse of the schedule: the query chunks i whose visit list holds
    # key chunk j, ordered by the ring step at which they meet it
    got = []
    for i in range(P):
        for t, jj, kind in oracle.ring_visits(P, causal, i):
            if jj == j and kind != oracle.KIND_SKIP:
                got.append((t, i, kind))
    return sorted(got)


def _slots(buf, P, n):
    return buf.view(-1, P + 1, 8)[:n].cpu().numpy()


CASES = [
    # P, C (chunk length), causal
    (1, 384, False), (1, 384, True),
    (2, 256, False), (2, 256, True),
    (3, 300, False), (3, 300, True),        # ragged tiles in every chunk
    (4, 512, False), (4, 512, True),
    (5, 200, False), (5, 200, True),
    (8, 128, False), (8, 128, True),
    (8, 100, True),                         # chunks shorter than a tile
    (16, 128, False), (16, 128, True),
]


@pytest.mark.parametrize("P,C,causal", CASES)
def test_forward_ring_order_bit_exact(ra, P, C, causal):
    B, H, d = 1, 2, 128
    S = P * C
    inp = workloads.make(workloads.FWD_CAUSAL_32K, B=B, H=H, S=S, d=d, P=P, causal=causal, seed=7)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    pairs = math.ceil(C / FWD_ROWS)
    grid = B * H * P * pairs
    buf = torch.full((grid * (P + 1) * 8,), SENTINEL, dtype=torch.int32, device="cuda")
    ra.trace_visits(buf)
    try:
        ra.ring_attn_fwd(q, k, v, P, causal)
        assert ra.check_status() == 0
    finally:
        ra.trace_visits(None)
    slots = _slots(buf, P, grid)
    T = math.ceil(C / TILE)
    seen = set()
    for x in range(grid):
        bh, i, q0, nvis, step, ntiles = slots[x, 0, :6]
        assert step == -1
        seen.add((int(bh), int(i), int(q0)))
        want = _expected_fwd(P, causal, int(i))
        got = [tuple(int(a) for a in slots[x, 1 + e, :3]) for e in range(nvis)]
        assert got == want, (x, got, want)
        q_end = min(q0 + FWD_ROWS, (i + 1) * C)
        total = 0
        for e, (t, j, kind) in enumerate(want):
            n_t, first, last = (int(a) for a in slots[x, 1 + e, 3:6])
            if kind == oracle.KIND_LOCAL and causal:
                n_want = math.ceil((q_end - i * C) / TILE)   # tiles holding keys <= the CTA's last row
            else:
                n_want = T
            assert n_t == n_want, (x, e, n_t, n_want)
            assert first == j * C and last == j * C + (n_t - 1) * TILE
            total += n_t
        assert total == ntiles
        # unused visit entries stay untouched
        assert (slots[x, 1 + nvis:] == SENTINEL).all()
    # every (head, query chunk, row pair) has exactly one CTA
    assert seen == {(bh, i, i * C + u * FWD_ROWS) for bh in range(B * H) for i in range(P) for u in range(pairs)}


@pytest.mark.parametrize("P,C,causal", CASES)
def test_backward_ring_order_bit_exact(ra, P, C, causal):
    B, H, d = 1, 2, 128
    S = P * C
    inp = workloads.make(workloads.FWDBWD_CAUSAL_128K, B=B, H=H, S=S, d=d, P=P, causal=causal, seed=8)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = ra.ring_attn_fwd(q, k, v, P, causal)
    T = math.ceil(C / TILE)
    grid = B * H * P * T
    buf = torch.full((grid * (P + 1) * 8,), SENTINEL, dtype=torch.int32, device="cuda")
    ra.trace_visits(buf)
    try:
        ra.ring_attn_bwd(q, k, v, o, lse, do, P, causal)
        assert ra.check_status() == 0
    finally:
        ra.trace_visits(None)
    slots = _slots(buf, P, grid)
    seen = set()
    for x in range(grid):
        bkv, j, kt, nvis, ntiles, group = (int(a) for a in slots[x, 0, :6])
        assert group == 1
        seen.add((bkv, j, kt))
        want = _expected_bwd(P, causal, j)
        got = [(int(slots[x, 1 + e, 1]), int(slots[x, 1 + e, 0]), int(slots[x, 1 + e, 2])) for e in range(nvis)]
        assert got == want, (x, got, want)
        total = 0
        for e, (t, i, kind) in enumerate(want):
            n_t, first, last = (int(a) for a in slots[x, 1 + e, 3:6])
            first_tile = kt if (causal and i == j) else 0   # query tiles wholly above the diagonal are skipped
            assert n_t == T - first_tile, (x, e, n_t)
            assert first == i * C + first_tile * TILE and last == i * C + (T - 1) * TILE
            total += n_t
        assert total == ntiles
        assert (slots[x, 1 + nvis:] == SENTINEL).all()
    assert seen == {(bkv, j, kt) for bkv in range(B * H) for j in range(P) for kt in range(T)}


def test_backward_ring_order_gqa(ra):
    # grouped-query: the key tile streams the same ring sequence for each of
    # the group's query heads; the record holds the first head's
    B, H, H_kv, d, P, C = 1, 4, 2, 128, 4, 256
    S = P * C
    inp = workloads.make(workloads.FWDBWD_GQA_128K, B=B, H=H, H_kv=H_kv, S=S, d=d, P=P, seed=9)
    q, k, v, do = (inp[x].cuda() for x in ("q", "k", "v", "do"))
    o, lse = ra.ring_attn_fwd(q, k, v, P, True)
    T = C // TILE
    grid = B * H_kv * P * T
    buf = torch.full((grid * (P + 1) * 8,), SENTINEL, dtype=torch.int32, device="cuda")
    ra.trace_visits(buf)
    try:
        ra.ring_attn_bwd(q, k, v, o, lse, do, P, True)
        assert ra.check_status() == 0
    finally:
        ra.trace_visits(None)
    slots = _slots(buf, P, grid)
    for x in range(grid):
        bkv, j, kt, nvis, ntiles, group = (int(a) for a in slots[x, 0, :6])
        assert group == H // H_kv
        want = _expected_bwd(P, True, j)
        got = [(int(slots[x, 1 + e, 1]), int(slots[x, 1 + e, 0]), int(slots[x, 1 + e, 2])) for e in range(nvis)]
        assert got == want
        per_head = sum(int(slots[x, 1 + e, 3]) for e in range(nvis))
        assert ntiles == group * per_head


def test_recording_is_off_by_default_and_after(ra):
    B, H, d, P, C = 1, 1, 128, 4, 256
    inp = workloads.make(workloads.FWD_CAUSAL_32K, B=B, H=H, S=P * C, d=d, P=P, seed=10)
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    buf = torch.full((4096,), SENTINEL, dtype=torch.int32, device="cuda")
    ra.trace_visits(buf)
    ra.trace_visits(None)
    o1, l1 = ra.ring_attn_fwd(q, k, v, P, True)
    assert ra.check_status() == 0
    assert (buf == SENTINEL).all().item()
    # a buffer too small for any slot is not written either
    small = torch.full((8,), SENTINEL, dtype=torch.int32, device="cuda")
    ra.trace_visits(small)
    try:
        o2, l2 = ra.ring_attn_fwd(q, k, v, P, True)
        assert ra.check_status() == 0
    finally:
        ra.trace_visits(None)
    assert (small == SENTINEL).all().item()
    # recording changes no result
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
