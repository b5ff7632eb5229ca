"""KDA float64 reference oracle (CPU).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The CUDA library never
imports, links or runs anything in this folder, and this folder imports
nothing from the CUDA package.

Two independent evaluations of the method live here:

* :func:`run` - the C oracle (``kda_oracle.c``): the KDA update of the web
  page "研究KimiK3，我发现大模型正在学会“管理自己的计算”" (pwwt.cn), §四,
  evaluated token by token in float64 in its rank-1 expanded form.
* :mod:`oracle.brute` - explicit d_k x d_k transition matrices multiplied out
  (same page, §五), for tiny inputs only; it pins the C oracle.
* :func:`backward` - the C gradient oracle (``kda_oracle_bwd.c``): the chain
  rule applied to that token-by-token update in reverse time, in float64,
  with the states replayed from checkpoints. The pages give no gradients;
  central finite differences of :func:`run` pin it.

Every input is upcast exactly to float64 before the call, so the oracle sees
precisely the values (fp32 or bf16) that a device kernel receives.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_BWD_SRC = os.path.join(_HERE, "kda_oracle_bwd.c")
_BWD_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle_bwd.so")
_lock = threading.Lock()
_lib = None
_bwd_lib = None

# -ffp-contract=off keeps every multiply and add separately rounded, so the
# x86 build and the aarch64 build return the same bits.
GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc into ``out`` (skipped when up to date)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


def build_all(force: bool = False):
    """Compile both oracle libraries (forward and gradients)."""
    build(force)
    build(force, src=_BWD_SRC, out=_BWD_LIB_PATH)


def load_backward(path: str | None = None):
    """Load (building first if needed) the gradient oracle library."""
    global _bwd_lib
    with _lock:
        if path is not None:
            return _bind_backward(ctypes.CDLL(path))
        if _bwd_lib is None:
            _bwd_lib = _bind_backward(ctypes.CDLL(build(src=_BWD_SRC, out=_BWD_LIB_PATH)))
        return _bwd_lib


def _bind_backward(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kda_oracle_backward.restype = ctypes.c_int
    lib.kda_oracle_backward.argtypes = [dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int32),
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        dp, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kda_oracle_run.restype = ctypes.c_int
    lib.kda_oracle_run.argtypes = [dp, dp, dp, dp, dp,
                                   ctypes.POINTER(ctypes.c_int32),
                                   ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int64,
                                   dp, dp, dp, ctypes.c_int]
    lib.kda_oracle_max_threads.restype = ctypes.c_int
    lib.kda_oracle_max_threads.argtypes = [ctypes.c_int]
    return lib


def _f64(x) -> np.ndarray:
    """Exact upcast of a numpy array or a CPU torch tensor (fp32/bf16/f64)."""
    if hasattr(x, "detach"):  # torch tensor: bf16 has no numpy twin
        x = x.detach().to("cpu")
        import torch  # local: only needed when a tensor is passed
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def run(q, k, v, alpha, beta, cu_seqlens=None, initial_state=None,
        nthreads: int = 0, lib=None):
    """Evaluate KDA over packed or batched sequences in float64.

    Shapes: q, k, alpha ``[B, T, H, dk]`` (or packed ``[T_total, H, dk]`` with
    ``cu_seqlens``), v ``[..., H, dv]``, beta ``[..., H]``, initial_state
    ``[N, H, dk, dv]`` or None (zeros).
    Returns ``(o, final_state)`` as float64 arrays; o has v's leading shape.
    """
    q, k, v, alpha, beta = (_f64(x) for x in (q, k, v, alpha, beta))
    lead = v.shape[:-2]
    H, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    if cu_seqlens is None:
        if len(lead) != 2:
            raise ValueError("batched inputs must be [B, T, H, d]")
        B, T = lead
        cu = np.arange(B + 1, dtype=np.int32) * T
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    s0 = None if initial_state is None else _f64(initial_state)
    if s0 is not None and s0.shape != (N, H, dk, dv):
        raise ValueError(f"initial_state must be {(N, H, dk, dv)}, got {s0.shape}")
    o = np.zeros(v.shape, dtype=np.float64)
    sT = np.zeros((N, H, dk, dv), dtype=np.float64)
    lib = lib or load()
    rc = lib.kda_oracle_run(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                            cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                            N, H, dk, dv, _ptr(s0), _ptr(o), _ptr(sT), int(nthreads))
    if rc != 0:
        raise ValueError(f"kda_oracle_run failed with code {rc}")
    return o, sT


def backward(q, k, v, alpha, beta, d_o, d_final_state=None, cu_seqlens=None, initial_state=None,
             nthreads: int = 0, lib=None):
    """Gradients of L = sum <d_o, o> + <d_final_state, S_T> in float64.

    Inputs as for :func:`run`; ``d_o`` has o's shape, ``d_final_state`` the
    final state's (None: zero). Returns a dict with ``dq``, ``dk``, ``dv``,
    ``dalpha``, ``dbeta`` (shaped like their inputs) and ``d_initial_state``
    ``[N, H, dk, dv]``.
    """
    q, k, v, alpha, beta, d_o = (_f64(x) for x in (q, k, v, alpha, beta, d_o))
    lead = v.shape[:-2]
    H, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    if d_o.shape != v.shape:
        raise ValueError(f"d_o must be {v.shape}, got {d_o.shape}")
    if cu_seqlens is None:
        if len(lead) != 2:
            raise ValueError("batched inputs must be [B, T, H, d]")
        B, T = lead
        cu = np.arange(B + 1, dtype=np.int32) * T
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    s0 = None if initial_state is None else _f64(initial_state)
    dsT = None if d_final_state is None else _f64(d_final_state)
    for name, x in (("initial_state", s0), ("d_final_state", dsT)):
        if x is not None and x.shape != (N, H, dk, dv):
            raise ValueError(f"{name} must be {(N, H, dk, dv)}, got {x.shape}")
    out = {"dq": np.zeros(q.shape), "dk": np.zeros(k.shape), "dv": np.zeros(v.shape),
           "dalpha": np.zeros(alpha.shape), "dbeta": np.zeros(beta.shape),
           "d_initial_state": np.zeros((N, H, dk, dv))}
    lib = lib or load_backward()
    rc = lib.kda_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                 cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), N, H, dk, dv,
                                 _ptr(s0), _ptr(d_o), _ptr(dsT), _ptr(out["dq"]), _ptr(out["dk"]),
                                 _ptr(out["dv"]), _ptr(out["dalpha"]), _ptr(out["dbeta"]),
                                 _ptr(out["d_initial_state"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"kda_oracle_backward failed with code {rc}")
    return out


def expand_gate(alpha, gate: str, lead: tuple, dk: int) -> np.ndarray:
    """The per-channel gate that a scalar gate or no gate stands for.

    The K3 essay's §四 sets KDA's per-channel gate Diag(alpha_t) beside the
    scalar gate alpha_t of Gated DeltaNet; without a gate the update is the
    delta rule of §三 (alpha_t = 1). A scalar gate multiplies every channel by
    the same alpha_t, so it is the per-channel gate with alpha_t repeated
    over the d_k channels. Returns float64 ``[*lead, dk]``. (Input preparation
    only: the recurrence itself is :func:`run`.)
    """
    lead = tuple(lead)
    if gate == "channel":
        a = _f64(alpha)
        if a.shape != lead + (dk,):
            raise ValueError(f"channel gate must be {lead + (dk,)}, got {a.shape}")
        return a
    if gate == "scalar":
        a = _f64(alpha)
        if a.shape != lead:
            raise ValueError(f"scalar gate must be {lead}, got {a.shape}")
        return np.repeat(a[..., None], dk, axis=-1)
    if gate == "none":
        return np.ones(lead + (dk,), dtype=np.float64)
    raise ValueError(f"unknown gate {gate!r}")


def dequant_mxfp8(codes, scales, block: int = 32) -> np.ndarray:
    """FP8 E4M3 codes with E8M0 block scales (one per ``block`` consecutive
    elements of the last axis) -> float64 values, decoded from the bit fields:
    sign s, exponent e (4 bits, bias 7), mantissa m (3 bits); e = 0 is
    subnormal, m * 2^-9; otherwise (1 + m/8) * 2^(e-7); 0x7F / 0xFF are NaN.
    The scale byte t stands for 2^(t - 127). (Input preparation for the FP8
    path: the recurrence itself is :func:`run`.)"""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    t = np.asarray(scales, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    val = sign * mag
    d = val.shape[-1]
    if d % block or t.shape[-1] != d // block:
        raise ValueError("scales must hold one byte per block of the last axis")
    return val * np.repeat(np.exp2(t - 127.0), block, axis=-1)


def max_threads(nthreads: int = 0) -> int:
    """Threads the oracle's OpenMP loop will use."""
    return int(load().kda_oracle_max_threads(int(nthreads)))
