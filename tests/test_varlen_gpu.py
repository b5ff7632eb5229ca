"""GPU tests of kda_varlen_prefill: cu_seqlens indexing is bit-exact (each
packed sequence gives exactly the bits of kda_prefill run on it alone),
device-side checks of bad cu_seqlens, and oracle parity on the lognormal
64-sequence workload."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

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


def test_varlen_64seq_sampled(kda):
    """64 lognormal-length sequences (306,055 tokens), H=16, d=128, bf16,
    per-sequence S0: bit-exact against single-sequence runs on a sample of
    sequences, and oracle parity on sampled (sequence, head) pairs including
    the longest sequence."""
    x = W.varlen_64seq()
    (q, k, v, a, b), cu, s0 = _dev(x)
    o, s = kda.varlen_prefill(q, k, v, a, b, cu, s0)
    torch.cuda.synchronize()
    cuh = x.cu_seqlens.tolist()
    lengths = np.diff(cuh)
    longest = int(np.argmax(lengths))
    for n in (0, longest, 63):
        lo, hi = cuh[n], cuh[n + 1]
        on, sn = kda.prefill(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], a[None, lo:hi],
                             b[None, lo:hi], s0[n:n + 1])
        assert torch.equal(o[lo:hi], on[0]) and torch.equal(s[n], sn[0])
    oc, sc = o.cpu(), s.cpu()
    tol = tol_for(x.q.dtype)
    for (n, h) in [(longest, 3), (5, 0), (40, 15)]:
        lo, hi = cuh[n], cuh[n + 1]
        sl = (slice(lo, hi), slice(h, h + 1))
        ro, rs = oracle.run(*(t[sl][None] for t in x.tensors()),
                            initial_state=x.initial_state[n:n + 1, h:h + 1])
        assert_close(f"o[seq {n}, head {h}]", oc[sl][None], ro, tol)
        assert_close(f"S[seq {n}, head {h}]", sc[n:n + 1, h:h + 1], rs, tol)
