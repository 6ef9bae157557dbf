"""Helpers for GPU-vs-oracle parity: error measure, tolerances, conversions."""

import numpy as np
import torch

# Maximum relative error, normalised per tensor by the oracle's largest magnitude:
#   max |gpu - oracle| / max(max |oracle|, 1e-6)
# 2e-3 for fp16 state (two fp16 half-ulps plus fp32 accumulation), 1e-5 for fp32 state.
TOL = {"f16": 2e-3, "f32": 1e-5}


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-6))


def np64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def assert_close(name, got, ref, tol):
    e = rel_err(np64(got) if isinstance(got, torch.Tensor) else got, ref)
    assert e <= tol, "%s: max relative error %.3g > %.1g" % (name, e, tol)
    return e


def dtype_name(t):
    return {torch.float16: "f16", torch.float32: "f32"}[t.dtype]
