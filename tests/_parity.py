"""Shared helpers for the GPU parity tests (comparison metrics, tolerances).

Tolerances (relative L2 over the whole tensor, separately for o and the final
state; max-abs over all elements):
  * fp32 q/k/v:                 rel-L2 <= 1e-4
  * bf16 q/k/v, fp32 gates/state: rel-L2 <= 5e-3 and max-abs <= 2e-2
"""
import numpy as np
import torch

TOL_FP32 = dict(rel=1e-4, abs=None)
TOL_BF16 = dict(rel=5e-3, abs=2e-2)


def tol_for(dtype):
    return TOL_FP32 if dtype == torch.float32 else TOL_BF16


def to64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


def rel_l2(x, ref) -> float:
    x, ref = to64(x), to64(ref)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def max_abs(x, ref) -> float:
    x, ref = to64(x), to64(ref)
    return float(np.abs(x - ref).max()) if x.size else 0.0


def assert_close(name, x, ref, tol):
    x64, r64 = to64(x), to64(ref)
    assert x64.shape == r64.shape, f"{name}: shape {x64.shape} vs {r64.shape}"
    assert np.all(np.isfinite(x64)), f"{name}: non-finite values"
    rl = rel_l2(x64, r64)
    assert rl <= tol["rel"], f"{name}: rel-L2 {rl:.3e} > {tol['rel']:.1e}"
    if tol.get("abs") is not None:
        ma = max_abs(x64, r64)
        assert ma <= tol["abs"], f"{name}: max-abs {ma:.3e} > {tol['abs']:.1e}"
    return rl
