"""Shared helpers of the GPU parity tests: tolerances and error metrics.

Tolerances (float): 2e-2 max relative error for bf16 inputs, 1e-4 for fp32.
* attention-mass scores are sums of positive terms, so the relative error is
  taken element by element, with a floor of 1e-6 x the largest score of the
  head (tiny scores carry no ranking information and their absolute error is
  already ~1e-8 of the head's mass);
* linear scores and attention outputs can cancel, so their error is taken
  relative to the largest magnitude of the row (per (unit, kv head) for
  scores, per (unit, q head) for outputs);
* lse values are compared with |delta| <= tol * max(1, |lse|).
Integer and byte results (indices, counts, offsets, compacted rows) must be
bit-exact.
"""
import numpy as np
import torch

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def mass_rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = 1e-6 * np.abs(ref).max(axis=-1, keepdims=True)
    den = np.maximum(np.abs(ref), floor)
    return float((np.abs(got - ref) / den).max())


def row_rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max(axis=-1, keepdims=True)
    den = np.where(den > 0, den, 1.0)
    return float((np.abs(got - ref) / den).max())


def lse_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(got - ref) / np.maximum(1.0, np.abs(ref)))
    return float(np.nan_to_num(d, nan=np.inf).max())
