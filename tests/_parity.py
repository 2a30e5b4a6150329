"""Helpers shared by the GPU parity tests: moving seeded inputs to the device,
widening them for the oracle, and the tolerances.

Tolerances (bf16 inputs/outputs, fp32 accumulation):
  O:        max |err| <= 2e-2 and mean |err| <= 2e-3
  LSE:      max |err| <= 1e-3
  dQ/dK/dV: max |err| <= 5e-2 on the N(0, 1) forward + backward recipe
            (assert_grad_max); elsewhere |err| <= 5e-2 + 2^-8 |ref| element
            by element (assert_grad_close) -- the 5e-2 bound plus the
            rounding of the exact value to the bf16 output format, which
            matters where a gradient sums a group of heads (grouped-query
            K/V) or grows large.
  Stress inputs whose gradients reach ~20 (the peaked-key input, keys
  c % 64 == 0 scaled x8): max |err| <= 5e-2 + the error of
  oracle.bwd_bf16_rounding_model on the same input -- an exact-arithmetic
  backward whose O, P, dS and outputs are stored in bf16 already misses
  the exact derivative by that much (0.088 for dQ on heads 0 of the
  2048-token case, mostly through D = <dO, O> formed from the bf16 O).
Integer / index results (the ring schedule) must match exactly.
"""
import numpy as np
import torch

O_MAX, O_MEAN, LSE_MAX, GRAD_MAX = 2e-2, 2e-3, 1e-3, 5e-2


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_o_close(got, ref, what="O"):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), f"{what}: non-finite values"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= O_MAX and mean <= O_MEAN, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def assert_lse_close(got, ref, what="LSE"):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), f"{what}: non-finite values"
    mx = float(err.max())
    assert mx <= LSE_MAX, f"{what}: max {mx:.3e}"
    return mx


BF16_U = 2.0 ** -8


def assert_grad_close(got, ref, what):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), f"{what}: non-finite values"
    excess = float((err - BF16_U * np.abs(ref)).max())
    assert excess <= GRAD_MAX, f"{what}: max err {float(err.max()):.3e}, beyond bf16 rounding {excess:.3e}"
    return float(err.max())


def assert_grad_max(got, ref, what):
    """The gradient bound as stated: max |err| <= 5e-2."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), f"{what}: non-finite values"
    mx = float(err.max())
    assert mx <= GRAD_MAX, f"{what}: max err {mx:.3e}"
    return mx


def assert_grad_close_model(got, ref, model, what):
    """Stress inputs: max |err| <= 5e-2 + max |model - ref|, where `model` is
    the bf16-storage rounding model's result (see the module docstring)."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    assert np.isfinite(err).all(), f"{what}: non-finite values"
    bound = GRAD_MAX + float(np.abs(np.asarray(model) - ref).max())
    mx = float(err.max())
    assert mx <= bound, f"{what}: max err {mx:.3e} > {bound:.3e}"
    return mx
