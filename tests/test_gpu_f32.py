"""fp32 inputs on the GPU (the small fp32 workload, B=1 H=2 S=1024 d=64 P=4,
taken natively): ring_attn_fwd_f32 rounds q, k, v to bf16 on the device and
returns O in fp32.

The kernel computes the same fp32 values as the bf16 entry point on the
rounded inputs and only skips the last rounding of O, so rounding its O to
bf16 must give the bf16 call's O bit for bit, and LSE must be identical.
Both are also checked against the oracle on the bf16-rounded inputs."""
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
    # workload, overrides
    (workloads.TINY_F32, {}),
    (workloads.TINY_F32, dict(causal=True, seed=7)),
    (workloads.FWDBWD_GQA_128K, dict(B=1, H=8, H_kv=2, S=2048, P=4, seed=8)),
    (workloads.FWD_CAUSAL_32K, dict(H=2, S=1200, P=3, seed=9)),        # ragged chunk tails
]


@pytest.mark.parametrize("w,over", CASES)
def test_f32_forward_matches_bf16_call_and_oracle(ra, w, over):
    inp = workloads.make(w, keep_fp32=True, **over)
    q32, k32, v32 = (inp[x].cuda() for x in ("q32", "k32", "v32"))
    q, k, v = (inp[x].cuda() for x in ("q", "k", "v"))
    P, causal, sc = inp["P"], inp["causal"], inp["scale"]
    o32, lse32 = ra.ring_attn_fwd_f32(q32, k32, v32, P, causal, sc)
    o, lse = ra.ring_attn_fwd(q, k, v, P, causal, sc)
    assert ra.check_status() == ra.RA_OK
    assert o32.dtype == torch.float32
    assert torch.equal(o32.to(torch.bfloat16), o), "rounded fp32 O differs from the bf16 call"
    assert torch.equal(lse32, lse), "LSE differs from the bf16 call"
    if inp["H_kv"] == inp["H"]:
        o_ref, lse_ref = oracle.naive_fwd(f64(q), f64(k), f64(v), causal, sc)
    else:
        o_ref, lse_ref = oracle.naive_fwd_gqa(f64(q), f64(k), f64(v), causal, sc)
    mx, _ = assert_o_close(f64(o32), o_ref)
    # no output rounding: the error is the fp32 accumulation and the bf16 P
    assert mx < 8e-3, f"fp32 O max error {mx:.3e}"
    assert_lse_close(f64(lse32), lse_ref)


def test_f32_output_may_alias_q(ra):
    inp = workloads.make(workloads.TINY_F32, keep_fp32=True)
    q32, k32, v32 = (inp[x].cuda() for x in ("q32", "k32", "v32"))
    P, causal, sc = inp["P"], inp["causal"], inp["scale"]
    want, _ = ra.ring_attn_fwd_f32(q32, k32, v32, P, causal, sc)
    buf = q32.clone()
    got, _ = ra.ring_attn_fwd_f32(buf, k32, v32, P, causal, sc, o=buf)
    assert ra.check_status() == ra.RA_OK
    assert got.data_ptr() == buf.data_ptr()
    assert torch.equal(got, want)


@pytest.mark.slow
def test_f32_forward_full_size_matches_bf16_call(ra):
    # the 128K causal shape (32 heads, P = 4) from fp32 inputs
    w = workloads.FWD_CAUSAL_128K
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    shape = (w.B, w.H, w.S, w.d)
    q32, k32, v32 = (torch.randn(shape, generator=g, device="cuda") for _ in range(3))
    sc = 1.0 / w.d ** 0.5
    o32, lse32 = ra.ring_attn_fwd_f32(q32, k32, v32, w.P, w.causal, sc)
    q, k, v = (x.to(torch.bfloat16) for x in (q32, k32, v32))
    del q32, k32, v32
    o, lse = ra.ring_attn_fwd(q, k, v, w.P, w.causal, sc)
    assert ra.check_status() == ra.RA_OK
    assert torch.equal(o32.to(torch.bfloat16), o)
    assert torch.equal(lse32, lse)
