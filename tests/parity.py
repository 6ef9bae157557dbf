"""Helpers for GPU-vs-oracle parity: error measures, tolerances, conversions.

Two measures of the same difference d = gpu - oracle:

* per tensor (the bar the tests assert): max |d| / max(max |ref|, 1e-6);
  2e-3 for fp16 state (two fp16 half-ulps at the tensor's largest magnitude
  plus fp32 accumulation slack), 1e-5 for fp32 state;
* element-wise (reported beside it): max over elements of |d| / (|ref| + 1e-3),
  which shows how large the error is on the small elements of a tensor. With
  fp16 operands on the tensor cores the absolute error of an element follows the
  magnitudes it was summed from, not its own, so this measure has no bar; the
  worst value per check is printed in the pytest summary.
"""

import numpy as np
import torch

TOL = {"f16": 2e-3, "f32": 1e-5}

# (check name, per-tensor error, element-wise error, tolerance) of every assert_close
REPORT = []


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-6))


def elem_rel_err(got, ref, floor=1e-3):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    return float((np.abs(got - ref) / (np.abs(ref) + floor)).max())


def np64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def assert_close(name, got, ref, tol):
    g = np64(got) if isinstance(got, torch.Tensor) else got
    e = rel_err(g, ref)
    ee = elem_rel_err(g, ref)
    REPORT.append((name, e, ee, tol))
    assert e <= tol, "%s: max relative error %.3g > %.1g (element-wise |d|/(|ref|+1e-3): %.3g)" % (
        name, e, tol, ee)
    return e


def dtype_name(t):
    return {torch.float16: "f16", torch.float32: "f32"}[t.dtype]
