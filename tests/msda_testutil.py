"""Helpers shared by the GPU tests: numpy <-> torch marshalling and the
tolerances the parity tests use.

Tolerances: fp32 forward max|err| <= 1e-5 * max|out|; fp32 gradients
<= 1e-4 relative L2 (grad_value is summed by atomics in any order);
fp16 / bf16 forward and gradients <= 2e-2 relative L2, all against the fp64
oracle on identical inputs.
"""
from __future__ import annotations

import numpy as np

from workloads import to_torch  # noqa: F401  (re-exported for the tests)


def f64(t):
    return t.detach().double().cpu().numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def max_rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    m = np.max(np.abs(b)) if b.size else 0.0
    return float(np.max(np.abs(a - b)) / m) if m > 0 else float(np.max(np.abs(a)) if a.size else 0.0)


def assert_forward(dtype: str, got, ref, what=""):
    if dtype == "f32":
        e = max_rel(got, ref)
        assert e <= 1e-5, f"{what} fp32 forward max|err|/max|out| = {e:.3e} > 1e-5"
    else:
        e = rel_l2(got, ref)
        assert e <= 2e-2, f"{what} {dtype} forward rel-L2 = {e:.3e} > 2e-2"
    return e


def assert_grad(dtype: str, got, ref, what=""):
    lim = 1e-4 if dtype == "f32" else 2e-2
    e = rel_l2(got, ref)
    assert e <= lim, f"{what} {dtype} rel-L2 = {e:.3e} > {lim:g}"
    return e
