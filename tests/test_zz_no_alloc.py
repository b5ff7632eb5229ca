"""kda_varlen_prefill_noalloc: the packed prefill for callers that may not
allocate device memory (engines that plan all device memory up front,
plug-ins handed only the call's tensors). It keeps its scratch in a fixed
array inside the library, shared by every call.

This file is collected last so that a run that stops at the first failure
has already run every other test. It must pass on its own in a fresh process
and after the other tests: two calls in a row on different batches must each
match kda_varlen_prefill (which takes a caller workspace), so nothing of the
first call's scratch may leak into the second.
"""
import ctypes

import pytest
import torch

from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

pytestmark = pytest.mark.gpu

MAX_SEQS = 16384  # KDA_NOALLOC_MAX_SEQS in include/kda.h


def _noalloc_fn(kda):
    lib = kda.load()
    fn = lib.kda_varlen_prefill_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp, vp]
    return lib, fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run_noalloc(kda, x, status=None):
    lib, fn = _noalloc_fn(kda)
    d = torch.device("cuda")
    q, k, v, a, b = (t.to(d) for t in x.tensors())
    cu = x.cu_seqlens.to(d)
    s0 = None if x.initial_state is None else x.initial_state.to(d)
    N = cu.numel() - 1
    Tt, H, dk = q.shape
    dv = v.shape[-1]
    o = torch.empty_like(v)
    sT = torch.empty((N, H, dk, dv), dtype=torch.float32, device=d)
    st = fn(_p(q), _p(k), _p(v), 1 if q.dtype == torch.bfloat16 else 0, _p(a), _p(b), _p(s0), _p(o), _p(sT),
            _p(cu), N, Tt, H, dk, dv, _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.kda_last_error()
    torch.cuda.synchronize()
    return o, sT


def _run_workspace(kda, x):
    d = torch.device("cuda")
    q, k, v, a, b = (t.to(d) for t in x.tensors())
    s0 = None if x.initial_state is None else x.initial_state.to(d)
    o, s = kda.varlen_prefill(q, k, v, a, b, x.cu_seqlens.to(d), s0)
    torch.cuda.synchronize()
    return o, s


def test_noalloc_matches_workspace_entry_point_twice(kda):
    # Two different batches back to back: the second call reuses the shared
    # scratch the first one filled (a different number of sequences, other
    # lengths, so a stale order or counter would show).
    batches = [W.packed([300, 64, 1, 0, 129, 700], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=31),
               W.packed([65, 513, 2, 200], 4, 128, 128, dtype="bf16", s0_std=0.05, seed=32)]
    for x in batches:
        o_na, s_na = _run_noalloc(kda, x)
        o_ws, s_ws = _run_workspace(kda, x)
        tol = tol_for(x.q.dtype)
        assert_close("o", o_na, o_ws, tol)
        assert_close("final_state", s_na, s_ws, tol)
        # same kernels and the same work split: the results are bitwise equal
        assert torch.equal(o_na, o_ws) and torch.equal(s_na, s_ws)


def test_noalloc_reports_bad_cu_seqlens_and_recovers(kda):
    d = torch.device("cuda")
    x = W.packed([40, 50, 60], 2, 64, 64, dtype="fp32", s0_std=0.05, seed=33)
    bad = W.Inputs(x.name, *x.tensors(), x.initial_state, x.cu_seqlens.clone())
    bad.cu_seqlens[1] = 100  # decreasing
    status = torch.full((1,), -1, dtype=torch.int32, device=d)
    _run_noalloc(kda, bad, status)
    assert int(status.item()) == kda.KDA_DEV_BAD_CU_SEQLENS
    status.fill_(-1)
    o_na, s_na = _run_noalloc(kda, x, status)
    assert int(status.item()) == kda.KDA_DEV_OK
    o_ws, s_ws = _run_workspace(kda, x)
    assert torch.equal(o_na, o_ws) and torch.equal(s_na, s_ws)


def test_noalloc_rejects_too_many_sequences(kda):
    lib, fn = _noalloc_fn(kda)
    p = ctypes.c_void_p(0x1000)
    st = fn(p, p, p, 1, p, p, None, p, None, p, MAX_SEQS + 1, 100000, 4, 128, 128, None, None)
    assert st == 2
    assert str(MAX_SEQS).encode() in lib.kda_last_error()
