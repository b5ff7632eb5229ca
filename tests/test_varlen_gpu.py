"""GPU tests of kda_varlen_prefill: cu_seqlens indexing is bit-exact (each
packed sequence gives exactly the bits of kda_prefill run on it alone),
device-side checks of bad cu_seqlens, and oracle parity on the lognormal
64-sequence workload (306,055 tokens, and its lengths rescaled to 2^20
tokens), every sequence and head checked."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import ErrAccum, assert_close, tol_for

pytestmark = pytest.mark.gpu


def _dev(x):
    d = torch.device("cuda")
    return [t.to(d) for t in x.tensors()], x.cu_seqlens.to(d), (
        None if x.initial_state is None else x.initial_state.to(d))


def _bitexact_vs_single(kda, x):
    (q, k, v, a, b), cu, s0 = _dev(x)
    o, s = kda.varlen_prefill(q, k, v, a, b, cu, s0)
    cuh = x.cu_seqlens.tolist()
    for n in range(len(cuh) - 1):
        lo, hi = cuh[n], cuh[n + 1]
        on, sn = kda.prefill(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], a[None, lo:hi],
                             b[None, lo:hi], None if s0 is None else s0[n:n + 1])
        assert torch.equal(o[lo:hi], on[0]), f"sequence {n}: o differs from the single-sequence run"
        assert torch.equal(s[n], sn[0]), f"sequence {n}: state differs"
    return o, s


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_varlen_bitexact_small(kda, dtype):
    x = W.packed([130, 1, 64, 0, 257, 63, 65], 3, 128, 128, dtype=dtype, s0_std=0.05, seed=2)
    o, s = _bitexact_vs_single(kda, x)
    ro, rs = oracle.run(*x.tensors(), cu_seqlens=x.cu_seqlens, initial_state=x.initial_state)
    tol = tol_for(x.q.dtype)
    assert_close("o", o, ro, tol)
    assert_close("S", s, rs, tol)
    # the zero-length sequence keeps its initial state
    assert torch.equal(s[3].cpu(), x.initial_state[3])


def test_varlen_without_initial_state(kda):
    x = W.packed([100, 37, 200], 2, 64, 64, dtype="fp32", s0_std=None, seed=4)
    x.initial_state = None
    _bitexact_vs_single(kda, x)


@pytest.mark.parametrize("bad", ["decreasing", "short_total", "nonzero_start"])
def test_bad_cu_seqlens_sets_device_status(kda, bad):
    x = W.packed([40, 50, 60], 2, 64, 64, dtype="fp32", s0_std=0.05, seed=1)
    (q, k, v, a, b), cu, s0 = _dev(x)
    cu_bad = cu.clone()
    if bad == "decreasing":
        cu_bad[1] = 100
    elif bad == "short_total":
        cu_bad[-1] = 140
    else:
        cu_bad[0] = 1
    status = torch.full((1,), -1, dtype=torch.int32, device=q.device)
    o = torch.full_like(v, 7.0)
    s = torch.full_like(s0, 7.0)
    kda.varlen_prefill(q, k, v, a, b, cu_bad, s0, out=o, final_state=s, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_BAD_CU_SEQLENS
    assert torch.all(o == 7.0) and torch.all(s == 7.0), "outputs written despite bad cu_seqlens"
    # a good call clears the status
    kda.varlen_prefill(q, k, v, a, b, cu, s0, out=o, final_state=s, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_OK


def _oracle_whole(x, o, s):
    """Every (sequence, head) pair against the oracle, one sequence (all its
    heads) per oracle call; rel-L2 and max-abs over the whole packed o and
    the whole final state."""
    oc, sc = o.cpu(), s.cpu()
    eo, es = ErrAccum("o"), ErrAccum("final_state")
    cuh = x.cu_seqlens.tolist()
    for n in range(len(cuh) - 1):
        lo, hi = cuh[n], cuh[n + 1]
        ro, rs = oracle.run(*(t[lo:hi][None] for t in x.tensors()), initial_state=x.initial_state[n:n + 1])
        eo.add(oc[lo:hi][None], ro)
        es.add(sc[n:n + 1], rs)
    tol = tol_for(x.q.dtype)
    eo.check(tol)
    es.check(tol)


def test_varlen_64seq_full(kda):
    """64 lognormal-length sequences (306,055 tokens), H=16, d=128, bf16,
    per-sequence S0: every sequence bit-exact against its own single-sequence
    prefill, and every (sequence, head) pair against the oracle."""
    x = W.varlen_64seq()
    o, s = _bitexact_vs_single(kda, x)
    torch.cuda.synchronize()
    _oracle_whole(x, o, s)


@pytest.mark.slow
def test_varlen_64seq_1m_full(kda):
    """The same 64 lengths scaled to 2^20 = 1,048,576 tokens in all (re-clipped
    to [512, 32768]; each sequence drawn on its own): every sequence
    bit-exact against its own single-sequence prefill, and every (sequence,
    head) pair against the oracle."""
    x = W.varlen_64seq_1m()
    assert x.meta["T_total"] == 1 << 20
    o, s = _bitexact_vs_single(kda, x)
    torch.cuda.synchronize()
    _oracle_whole(x, o, s)
