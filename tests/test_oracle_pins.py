"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test ties one oracle routine to something the pages or plain mathematics
fix: a hand-computed value, a closed form, an invariant, an independent
high-precision evaluation, a printed number, or a finite-difference
derivative.  All run on CPU.
"""
import math
import os

import mpmath
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(20240601)


# Both whole-tensor forward routines answer to the same pins: the C loops and
# the row-block PyTorch pass (blocks of 3 rows here, so every case spans
# several blocks).
FWD_IMPLS = {
    "c_loops": oracle.naive_fwd,
    "row_blocks": lambda q, k, v, causal, scale: oracle.naive_fwd_blocked(q, k, v, causal, scale, block=3),
}


def _rand(B, H, S, d, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((B, H, S, d)), g.standard_normal((B, H, S, d)),
            g.standard_normal((B, H, S, d)))


# --------------------------------------------------------------------------
# naive_fwd: textbook special cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("impl", FWD_IMPLS)
@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_that_value(causal, impl):
    # S = 1: the only key gets weight 1, so O = v_0 and LSE = s_00.
    q = np.array([[[[0.5, -1.0, 2.0]]]])
    k = np.array([[[[1.5, 0.25, -0.5]]]])
    v = np.array([[[[3.0, -7.0, 0.125]]]])
    o, lse = FWD_IMPLS[impl](q, k, v, causal, 0.7)
    s00 = 0.7 * (0.5 * 1.5 - 1.0 * 0.25 + 2.0 * -0.5)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    assert lse[0, 0, 0] == pytest.approx(s00, abs=1e-15)


@pytest.mark.parametrize("impl", FWD_IMPLS)
def test_hand_computed_d1(impl):
    # d = 1, scale = 1, q = 1, keys 0 and ln 3 -> scores 0, ln 3,
    # weights 1/4 and 3/4; values 2 and 6 -> O = 0.5 + 4.5 = 5; LSE = ln 4.
    q = np.array([[[[1.0], [1.0]]]])
    k = np.array([[[[0.0], [math.log(3.0)]]]])
    v = np.array([[[[2.0], [6.0]]]])
    o, lse = FWD_IMPLS[impl](q, k, v, False, 1.0)
    assert o[0, 0, 1, 0] == pytest.approx(5.0, abs=1e-14)
    assert lse[0, 0, 1] == pytest.approx(math.log(4.0), abs=1e-15)
    # causal: row 0 sees only key 0 -> O = 2, LSE = 0; row 1 as above.
    o, lse = FWD_IMPLS[impl](q, k, v, True, 1.0)
    assert o[0, 0, 0, 0] == 2.0 and lse[0, 0, 0] == 0.0
    assert o[0, 0, 1, 0] == pytest.approx(5.0, abs=1e-14)


@pytest.mark.parametrize("impl", FWD_IMPLS)
def test_two_keys_sigmoid_weights(impl):
    # Two keys: weight of key 0 is the logistic function of s_0 - s_1.
    q, k, v = _rand(1, 1, 2, 5, 1)
    scale = 0.37
    o, lse = FWD_IMPLS[impl](q, k, v, False, scale)
    for r in range(2):
        s0 = scale * float(q[0, 0, r] @ k[0, 0, 0])
        s1 = scale * float(q[0, 0, r] @ k[0, 0, 1])
        w0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        expect = w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1]
        np.testing.assert_allclose(o[0, 0, r], expect, rtol=0, atol=1e-14)
        assert lse[0, 0, r] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))),
                                             abs=1e-14)


@pytest.mark.parametrize("impl", FWD_IMPLS)
@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_match_high_precision(causal, impl):
    # With S == d and V = I, O_r is the attention row P_r itself.
    S = d = 8
    q, k, _ = _rand(1, 1, S, d, 2)
    v = np.eye(S)[None, None]
    scale = 1.0 / math.sqrt(d)
    o, lse = FWD_IMPLS[impl](q, k, v, causal, scale)
    np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-12)
    mpmath.mp.dps = 40
    for r in range(S):
        allowed = range(r + 1) if causal else range(S)
        s = {c: mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[0, 0, r, x]) * mpmath.mpf(k[0, 0, c, x])
                                                   for x in range(d)) for c in allowed}
        z = mpmath.fsum(mpmath.e ** s[c] for c in allowed)
        assert float(mpmath.log(z)) == pytest.approx(lse[0, 0, r], abs=1e-13)
        for c in range(S):
            p = float(mpmath.e ** s[c] / z) if c in s else 0.0
            assert o[0, 0, r, c] == pytest.approx(p, abs=1e-14)


@pytest.mark.parametrize("impl", FWD_IMPLS)
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal, impl):
    q, k, _ = _rand(2, 3, 17, 6, 3)
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25, 3.0, -0.75, 9.0]), q.shape).copy()
    o, _ = FWD_IMPLS[impl](q, k, v, causal, 0.9)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


@pytest.mark.parametrize("impl", FWD_IMPLS)
@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_is_uniform_average(causal, impl):
    B, H, S, d = 1, 2, 9, 4
    _, k, v = _rand(B, H, S, d, 4)
    q = np.zeros((B, H, S, d))
    o, lse = FWD_IMPLS[impl](q, k, v, causal, 0.5)
    for r in range(S):
        n = r + 1 if causal else S
        np.testing.assert_allclose(o[:, :, r], v[:, :, :n].mean(axis=2), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, r], math.log(n), rtol=0, atol=1e-14)


@pytest.mark.parametrize("impl", FWD_IMPLS)
def test_brute_force_high_precision_random(impl):
    # Independent 40-digit evaluation of the definition on tiny random inputs.
    B, H, S, d = 1, 2, 6, 3
    q, k, v = _rand(B, H, S, d, 5)
    q *= 3.0  # spread the scores so the max subtraction matters
    scale = 0.8
    mpmath.mp.dps = 40
    for causal in (False, True):
        o, lse = FWD_IMPLS[impl](q, k, v, causal, scale)
        for h in range(H):
            for r in range(S):
                allowed = range(r + 1) if causal else range(S)
                s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[0, h, r, x]) * mpmath.mpf(k[0, h, c, x])
                                                     for x in range(d)) for c in allowed]
                z = mpmath.fsum(mpmath.e ** si for si in s)
                for x in range(d):
                    ref = mpmath.fsum(mpmath.e ** si / z * mpmath.mpf(v[0, h, c, x])
                                      for si, c in zip(s, allowed))
                    assert o[0, h, r, x] == pytest.approx(float(ref), abs=1e-13)
                assert lse[0, h, r] == pytest.approx(float(mpmath.log(z)), abs=1e-13)


def test_rows_api_matches_whole_rows():
    q, k, v = _rand(2, 2, 40, 8, 6)
    o, lse = oracle.naive_fwd(q, k, v, True, 0.3)
    rows = np.array([0, 39, 40, 41, 79, 100, 159])
    o_r, lse_r = oracle.naive_fwd_rows(q, k, v, True, 0.3, rows)
    np.testing.assert_array_equal(o_r, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(lse_r, lse.reshape(-1)[rows])


@pytest.mark.parametrize("impl", FWD_IMPLS)
def test_large_scores_do_not_overflow(impl):
    # Max subtraction: scores near 1000 must not overflow exp.
    q = np.full((1, 1, 3, 1), 40.0)
    k = np.array([[[[25.0], [24.0], [-5.0]]]])
    v = np.array([[[[1.0], [2.0], [3.0]]]])
    o, lse = FWD_IMPLS[impl](q, k, v, False, 1.0)
    w = np.exp(np.array([1000.0, 960.0, -200.0]) - 1000.0)
    w /= w.sum()
    np.testing.assert_allclose(o[0, 0, 0, 0], w @ np.array([1.0, 2.0, 3.0]), atol=1e-15)
    assert lse[0, 0, 0] == pytest.approx(1000.0 + math.log1p(math.exp(-40.0)), abs=1e-12)


# --------------------------------------------------------------------------
# ring_fwd and the merge: exactness and merge algebra
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 3, 4, 6, 12])
def test_ring_equals_naive(P, causal):
    # "exact" (first page, "Ring Attention Demystified"): ring == unchunked.
    q, k, v = _rand(2, 2, 36, 7, 7)
    o_n, lse_n = oracle.naive_fwd(q, k, v, causal, 0.45)
    o_r, lse_r, _ = oracle.ring_fwd(q, k, v, P, causal, 0.45)
    np.testing.assert_allclose(o_r, o_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_r, lse_n, rtol=0, atol=1e-12)


def test_ring_rejects_unequal_split():
    q, k, v = _rand(1, 1, 10, 2, 8)
    with pytest.raises(ValueError):
        oracle.ring_fwd(q, k, v, 3, False, 1.0)


def test_merge_identity_and_self():
    o = rng.standard_normal((5, 4))
    lse = rng.standard_normal(5)
    zero = np.zeros_like(o)
    ninf = np.full(5, -np.inf)
    for a, b in (((o, lse), (zero, ninf)), ((zero, ninf), (o, lse))):
        om, lm = oracle.merge(a[0], a[1], b[0], b[1])
        np.testing.assert_array_equal(om, o)
        np.testing.assert_array_equal(lm, lse)
    om, lm = oracle.merge(o, lse, o, lse)
    np.testing.assert_allclose(om, o, atol=1e-15)
    np.testing.assert_allclose(lm, lse + math.log(2.0), atol=1e-15)
    om, lm = oracle.merge(zero, ninf, zero, ninf)
    assert np.all(om == 0) and np.all(lm == -np.inf)


def test_merge_commutative_associative():
    o = [rng.standard_normal((6, 3)) for _ in range(3)]
    l = [rng.standard_normal(6) * 4 for _ in range(3)]
    ab = oracle.merge(o[0], l[0], o[1], l[1])
    ba = oracle.merge(o[1], l[1], o[0], l[0])
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-14)
    np.testing.assert_allclose(ab[1], ba[1], atol=1e-14)
    left = oracle.merge(ab[0], ab[1], o[2], l[2])
    bc = oracle.merge(o[1], l[1], o[2], l[2])
    right = oracle.merge(o[0], l[0], bc[0], bc[1])
    np.testing.assert_allclose(left[0], right[0], atol=1e-13)
    np.testing.assert_allclose(left[1], right[1], atol=1e-13)


def test_merge_of_split_keys_equals_whole():
    # Attention over keys A u B equals the merge of attention over A and B.
    # The 12 query rows are laid out as 2 "heads" of 6 rows so that each
    # call sees 6 queries against the same 6-key half.
    q, k, v = _rand(1, 1, 12, 5, 9)
    o_w, l_w = oracle.naive_fwd(q, k, v, False, 0.6)
    qh = q.reshape(1, 2, 6, 5)
    parts = []
    for s in (slice(0, 6), slice(6, 12)):
        kh = np.concatenate([k[:, :, s]] * 2, axis=1)
        vh = np.concatenate([v[:, :, s]] * 2, axis=1)
        parts.append(oracle.naive_fwd(qh, kh, vh, False, 0.6))
    o_m, l_m = oracle.merge(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    np.testing.assert_allclose(o_m.reshape(o_w.shape), o_w, atol=1e-13)
    np.testing.assert_allclose(l_m.reshape(l_w.shape), l_w, atol=1e-13)


# --------------------------------------------------------------------------
# Ring schedule
# --------------------------------------------------------------------------

def _golden_schedule():
    rows = []
    with open(os.path.join(GOLDEN, "ring_schedule_p4.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            i, t, j, kn, kc = line.split()
            rows.append((int(i), int(t), int(j), kn, kc))
    return rows


def test_schedule_matches_printed_rotation():
    names = {oracle.KIND_LOCAL: "local", oracle.KIND_FULL: "full", oracle.KIND_SKIP: "skip"}
    for i, t, j, kn, kc in _golden_schedule():
        assert oracle.ring_visits(4, False, i)[t] == (t, j, oracle.KIND_LOCAL if kn == "local"
                                                       else oracle.KIND_FULL)
        tt, jj, kk = oracle.ring_visits(4, True, i)[t]
        assert (tt, jj, names[kk]) == (t, j, kc)


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16])
def test_schedule_coverage(P):
    # After P - 1 rotations every query chunk has met every KV chunk once.
    seen = {}
    for i in range(P):
        for t, j, kind in oracle.ring_visits(P, False, i):
            seen[(i, j)] = seen.get((i, j), 0) + 1
            assert j == (i - t) % P
    assert len(seen) == P * P and set(seen.values()) == {1}
    kept = [(i, j) for i in range(P) for _, j, kind in oracle.ring_visits(P, True, i)
            if kind != oracle.KIND_SKIP]
    assert len(kept) == P * (P + 1) // 2 and all(j <= i for i, j in kept)


def test_ring_log_is_the_schedule():
    q, k, v = _rand(1, 1, 8, 2, 10)
    _, _, log = oracle.ring_fwd(q, k, v, 4, True, 1.0)
    for i in range(4):
        for t in range(4):
            assert tuple(log[i, t]) == oracle.ring_visits(4, True, i)[t]


# --------------------------------------------------------------------------
# Backward: finite differences and identities
# --------------------------------------------------------------------------

def _loss(q, k, v, dO, causal, scale):
    o, _ = oracle.naive_fwd(q, k, v, causal, scale)
    return float((o * dO).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,d", [(5, 3), (8, 4)])
def test_backward_finite_differences(S, d, causal):
    q, k, v = _rand(1, 1, S, d, 11 + S)
    dO = np.random.default_rng(99).standard_normal(q.shape)
    scale = 0.7
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, dO, causal, scale)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
            num[idx] = (_loss(args_p["q"], args_p["k"], args_p["v"], dO, causal, scale)
                        - _loss(args_m["q"], args_m["k"], args_m["v"], dO, causal, scale)) / (2 * eps)
        err = np.abs(num - g).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (name, err)


def test_backward_D_two_ways_and_constant_v():
    q, k, v = _rand(1, 2, 10, 4, 21)
    dO = np.random.default_rng(3).standard_normal(q.shape)
    for causal in (False, True):
        _, _, _, lse, D = oracle.bwd(q, k, v, dO, causal, 0.5)
        o, lse2 = oracle.naive_fwd(q, k, v, causal, 0.5)
        np.testing.assert_allclose(D, (dO * o).sum(-1), atol=1e-13)
        np.testing.assert_allclose(lse, lse2, atol=0)
    vc = np.broadcast_to(np.array([1.0, -2.0, 0.5, 3.0]), q.shape).copy()
    dq, dk, dv, _, _ = oracle.bwd(q, k, vc, dO, True, 0.5)
    np.testing.assert_allclose(dq, 0, atol=1e-13)
    np.testing.assert_allclose(dk, 0, atol=1e-13)


def test_backward_column_sums():
    # Rows of P sum to 1: sum_c dV_c = sum_r dO_r; and sum_c dS_rc = 0,
    # so sum_c dK_c = 0.  These hold at any size.
    q, k, v = _rand(1, 2, 24, 6, 31)
    dO = np.random.default_rng(4).standard_normal(q.shape)
    for causal in (False, True):
        dq, dk, dv, _, _ = oracle.bwd(q, k, v, dO, causal, 0.4)
        np.testing.assert_allclose(dv.sum(2), dO.sum(2), atol=1e-12)
        np.testing.assert_allclose(dk.sum(2), 0, atol=1e-12)


def test_backward_dq_rows_matches_full():
    q, k, v = _rand(1, 2, 20, 5, 41)
    dO = np.random.default_rng(5).standard_normal(q.shape)
    dq, _, _, _, D = oracle.bwd(q, k, v, dO, True, 0.6)
    rows = np.array([0, 7, 19, 20, 33, 39])
    dq_r, D_r = oracle.bwd_dq_rows(q, k, v, dO, True, 0.6, rows)
    np.testing.assert_allclose(dq_r, dq.reshape(-1, 5)[rows], atol=1e-13)
    np.testing.assert_allclose(D_r, D.reshape(-1)[rows], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_key_rows_finite_differences(causal):
    # dK_c and dV_c of chosen key rows, with LSE and D taken over every query
    # row inside the routine, against central differences of L = sum(dO * O)
    # in the key row's own entries.
    S, d = 7, 3
    q, k, v = _rand(1, 1, S, d, 61)
    dO = np.random.default_rng(62).standard_normal(q.shape)
    scale = 0.8
    keys = np.array([0, 3, 6])
    dk, dv, lse, D = oracle.bwd_dkdv_rows(q, k, v, dO, causal, scale, keys, block=2)
    eps = 1e-6
    for n, c in enumerate(keys):
        for x in range(d):
            for name, grad in (("k", dk), ("v", dv)):
                a = {"q": q, "k": k.copy(), "v": v.copy()}
                b = {"q": q, "k": k.copy(), "v": v.copy()}
                a[name][0, 0, c, x] += eps
                b[name][0, 0, c, x] -= eps
                num = (_loss(a["q"], a["k"], a["v"], dO, causal, scale)
                       - _loss(b["q"], b["k"], b["v"], dO, causal, scale)) / (2 * eps)
                assert abs(num - grad[n, x]) <= 1e-6 * max(1.0, abs(num)), (name, c, x)
    # D_r = sum_k dO_rk O_rk (the identity sum_c P_rc dP_rc = <dO_r, O_r>)
    o, lse_ref = oracle.naive_fwd(q, k, v, causal, scale)
    np.testing.assert_allclose(D, (dO * o).sum(-1)[0, 0], atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref[0, 0], atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_key_rows_match_full(causal):
    # Many row blocks, keys on and off the block edges, against the C loops.
    S, d = 200, 8
    q, k, v = _rand(1, 1, S, d, 71)
    dO = np.random.default_rng(72).standard_normal(q.shape)
    dq, dk, dv, lse, D = oracle.bwd(q, k, v, dO, causal, 0.45)
    keys = np.array([0, 1, 31, 32, 33, 100, 150, 198, 199])
    dk_r, dv_r, lse_r, D_r = oracle.bwd_dkdv_rows(q, k, v, dO, causal, 0.45, keys, block=32)
    np.testing.assert_allclose(dk_r, dk[0, 0][keys], atol=1e-13)
    np.testing.assert_allclose(dv_r, dv[0, 0][keys], atol=1e-13)
    np.testing.assert_allclose(lse_r, lse[0, 0], atol=1e-13)
    np.testing.assert_allclose(D_r, D[0, 0], atol=1e-13)
    # every key: the column sums sum_c dV_c = sum_r dO_r and sum_c dK_c = 0
    dk_a, dv_a, _, _ = oracle.bwd_dkdv_rows(q, k, v, dO, causal, 0.45, np.arange(S), block=32)
    np.testing.assert_allclose(dv_a.sum(0), dO[0, 0].sum(0), atol=1e-12)
    np.testing.assert_allclose(dk_a.sum(0), 0, atol=1e-12)


def test_backward_key_rows_rejects_bad_input():
    q, k, v = _rand(1, 2, 8, 4, 73)
    with pytest.raises(ValueError):
        oracle.bwd_dkdv_rows(q, k, v, q, True, 0.5, [0])          # two heads
    with pytest.raises(ValueError):
        oracle.bwd_dkdv_rows(q[:, :1], k[:, :1], v[:, :1], q[:, :1], True, 0.5, [8])


def test_bf16_rounding_matches_the_library_conversion():
    # the rounding model's bf16 step against torch's own fp32 -> bf16
    # conversion (round to nearest even), including exact ties
    import torch
    from oracle.oracle import _bf16_rne
    g = torch.Generator().manual_seed(81)
    x = torch.randn(200000, generator=g, dtype=torch.float64) * torch.exp(
        torch.randn(200000, generator=g, dtype=torch.float64) * 8)
    ties = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 0.0, -0.0,
                         float("inf"), -float("inf")], dtype=torch.float64)
    for t in (x, ties):
        want = t.to(torch.float32).to(torch.bfloat16).to(torch.float64)
        assert torch.equal(_bf16_rne(t), want)


@pytest.mark.parametrize("causal", [False, True])
def test_rounding_model_without_rounding_is_the_derivative(causal):
    # every rounding replaced by the identity leaves the plain derivative,
    # which the finite-difference pins above fix
    q, k, v = _rand(2, 2, 24, 8, 91)
    dO = np.random.default_rng(92).standard_normal(q.shape)
    dq, dk, dv, _, _ = oracle.bwd(q, k, v, dO, causal, 0.35)
    mq, mk, mv = oracle.bwd_bf16_rounding_model(q, k, v, dO, causal, 0.35, round_bf16=False)
    np.testing.assert_allclose(mq, dq, atol=1e-12)
    np.testing.assert_allclose(mk, dk, atol=1e-12)
    np.testing.assert_allclose(mv, dv, atol=1e-12)
    # with rounding, every output is a bf16 value and lies within a few bf16
    # units of the exact derivative on N(0, 1) inputs
    import torch
    rq, rk, rv = oracle.bwd_bf16_rounding_model(q, k, v, dO, causal, 0.35)
    for got, ref in ((rq, dq), (rk, dk), (rv, dv)):
        t = torch.as_tensor(got)
        assert torch.equal(t, t.to(torch.float32).to(torch.bfloat16).to(torch.float64))
        assert np.abs(got - ref).max() <= 4 * 2.0 ** -8 * max(1.0, np.abs(ref).max())


# --------------------------------------------------------------------------
# Analytic helpers against the guide's printed numbers
# --------------------------------------------------------------------------

def _golden_bytes():
    out = {}
    unit = {"MiB": 2 ** 20, "KiB": 2 ** 10, "GiB": 2 ** 30, "Gi": 2 ** 30}
    with open(os.path.join(GOLDEN, "analytic_bytes.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, val, u = line.split()[:3]
            out[name] = int(val) * unit[u]
    return out


def test_printed_worked_example_numbers():
    g = _golden_bytes()
    S, P, dk, heads = 128 * 1024, 4, 128, 32
    assert oracle.ring_step_bytes(S, P, dk) == g["ring_step_bytes_per_head"]
    assert oracle.ring_total_bytes(S, P, dk) == g["ring_three_steps_per_head"]
    # 512 KB/token: the reading is 32 layers (a 7B MHA model), K and V, BF16.
    per_tok = oracle.kv_cache_bytes_per_token(32, heads, dk)
    assert per_tok == g["kv_cache_bytes_per_token"]
    assert S * per_tok == g["kv_cache_bytes_128k"]
    assert (S // P) * per_tok == g["kv_cache_bytes_per_gpu_cp4"]
    assert oracle.score_matrix_elements(S) == g["score_elements_128k"]
    assert oracle.score_matrix_elements(S) * 2 == g["score_bytes_per_head_128k"]


def test_flop_count_reading():
    # 4 d FLOPs per allowed pair; causal counts c <= r.
    assert oracle.attention_flops(1, 2, 1024, 64, False) == 536_870_912
    f = oracle.attention_flops(1, 32, 131072, 128, True)
    assert f == 4 * 128 * 32 * (131072 * 131073 // 2)
    assert abs(f - 1.4074e14) / 1.4074e14 < 1e-3


# --------------------------------------------------------------------------
# Grouped-query attention
# --------------------------------------------------------------------------

def test_gqa_with_one_group_member_is_mha():
    q, k, v = _rand(1, 3, 9, 4, 51)
    o1, l1 = oracle.naive_fwd_gqa(q, k, v, True, 0.5)
    o2, l2 = oracle.naive_fwd(q, k, v, True, 0.5)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_gqa_heads_of_a_group_see_the_same_keys():
    # MQA (one K/V head): a query head's output depends only on its own
    # queries and the shared K/V -- recomputing head h alone gives the same.
    B, H, S, d = 1, 4, 7, 3
    g = np.random.default_rng(52)
    q = g.standard_normal((B, H, S, d))
    k = g.standard_normal((B, 1, S, d))
    v = g.standard_normal((B, 1, S, d))
    o, lse = oracle.naive_fwd_gqa(q, k, v, False, 0.7)
    for h in range(H):
        o_h, l_h = oracle.naive_fwd(q[:, h:h + 1], k, v, False, 0.7)
        np.testing.assert_allclose(o[:, h:h + 1], o_h, atol=1e-15)
        np.testing.assert_allclose(lse[:, h:h + 1], l_h, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_backward_finite_differences(causal):
    # dK, dV of a shared head collect the whole group: checked against
    # central differences of the GQA forward.
    B, H, Hkv, S, d = 1, 4, 2, 5, 3
    g = np.random.default_rng(53)
    q = g.standard_normal((B, H, S, d))
    k = g.standard_normal((B, Hkv, S, d))
    v = g.standard_normal((B, Hkv, S, d))
    dO = g.standard_normal((B, H, S, d))
    scale = 0.6
    dq, dk, dv = oracle.bwd_gqa(q, k, v, dO, causal, scale)

    def loss(q_, k_, v_):
        o, _ = oracle.naive_fwd_gqa(q_, k_, v_, causal, scale)
        return float((o * dO).sum())
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            a = {"q": q, "k": k, "v": v}; a[name] = xp
            b = {"q": q, "k": k, "v": v}; b[name] = xm
            num[idx] = (loss(a["q"], a["k"], a["v"]) - loss(b["q"], b["k"], b["v"])) / (2 * eps)
        assert np.abs(num - grad).max() / np.abs(num).max() < 1e-6, name
