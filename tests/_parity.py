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


class ErrAccum:
    """Whole-tensor rel-L2 and max-abs built up piece by piece (pieces of one
    tensor, e.g. groups of heads or sequences that the oracle runs one at a
    time): sum of squared differences, sum of squared references, largest
    absolute difference."""

    def __init__(self, name):
        self.name, self.d2, self.r2, self.mx, self.n = name, 0.0, 0.0, 0.0, 0

    def add(self, x, ref):
        x64, r64 = to64(x), to64(ref)
        assert x64.shape == r64.shape, f"{self.name}: shape {x64.shape} vs {r64.shape}"
        assert np.all(np.isfinite(x64)), f"{self.name}: non-finite values"
        d = x64 - r64
        self.d2 += float(np.sum(d * d))
        self.r2 += float(np.sum(r64 * r64))
        if d.size:
            self.mx = max(self.mx, float(np.abs(d).max()))
        self.n += d.size

    def rel(self) -> float:
        return (self.d2 ** 0.5) / (self.r2 ** 0.5 if self.r2 > 0 else 1.0)

    def check(self, tol):
        rl = self.rel()
        assert rl <= tol["rel"], f"{self.name}: rel-L2 {rl:.3e} > {tol['rel']:.1e} over {self.n} elements"
        if tol.get("abs") is not None:
            assert self.mx <= tol["abs"], f"{self.name}: max-abs {self.mx:.3e} > {tol['abs']:.1e}"
        print(f"{self.name}: rel-L2 {rl:.3e}, max-abs {self.mx:.3e} over {self.n} elements")
        return rl
