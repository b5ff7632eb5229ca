"""GPU parity of kda_decode_step against the float64 oracle (one token per
sequence: the oracle runs T = 1 from the same state)."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

pytestmark = pytest.mark.gpu


def _oracle_decode(x: W.Inputs):
    q, k, v, a, b = (t[:, None] for t in x.tensors())  # [N, 1, H, d]: one-token sequences
    o, s = oracle.run(q, k, v, a, b, initial_state=x.initial_state)
    return o[:, 0], s


def _run(kda, x: W.Inputs):
    dev = torch.device("cuda")
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    state = x.initial_state.to(dev).clone()
    o = kda.decode_step(q, k, v, a, b, state)
    torch.cuda.synchronize()
    return o, state


def test_decode_256x32_full(kda):
    """256 sequences x 32 heads, d = 128, bf16 q/k/v, fp32 state (every head)."""
    x = W.decode_256x32()
    o, s = _run(kda, x)
    ro, rs = _oracle_decode(x)
    tol = tol_for(x.q.dtype)
    assert_close("o", o, ro, tol)
    assert_close("state", s, rs, tol)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_shapes_and_dtypes(kda, dk, dv, dtype):
    q, k, v, a, b, s0 = W.draw((5,), 3, dk, dv, dtype=dtype, alpha_scale=0.1, s0_std=0.1, seed=dk + dv)
    x = W.Inputs("d", q, k, v, a, b, s0)
    o, s = _run(kda, x)
    ro, rs = _oracle_decode(x)
    tol = tol_for(q.dtype)
    assert_close("o", o, ro, tol)
    assert_close("state", s, rs, tol)


def test_decode_gate_edge_cases(kda):
    """beta = 0 is pure decay; alpha = 0 erases a channel before the write."""
    q, k, v, a, b, s0 = W.draw((4,), 2, 128, 128, dtype="fp32", s0_std=0.1, seed=3)
    b[0] = 0.0
    a[1, :, :64] = 0.0
    x = W.Inputs("edge", q, k, v, a, b, s0)
    o, s = _run(kda, x)
    ro, rs = _oracle_decode(x)
    assert_close("o", o, ro, tol_for(torch.float32))
    assert_close("state", s, rs, tol_for(torch.float32))
    np.testing.assert_allclose(s[0].cpu().numpy(), (a[0][..., None] * s0[0]).numpy(), rtol=1e-6, atol=1e-7)


def test_decode_equals_one_token_prefill(kda):
    """A decode step is the prefill of a one-token sequence from that state."""
    dev = torch.device("cuda")
    q, k, v, a, b, s0 = W.draw((6,), 4, 128, 128, dtype="bf16", s0_std=0.1, seed=9)
    st = s0.to(dev).clone()
    o_dec = kda.decode_step(q.to(dev), k.to(dev), v.to(dev), a.to(dev), b.to(dev), st)
    o_pre, s_pre = kda.prefill(q[:, None].to(dev), k[:, None].to(dev), v[:, None].to(dev),
                               a[:, None].to(dev), b[:, None].to(dev), s0.to(dev), algo="simt")
    torch.cuda.synchronize()
    assert_close("o", o_dec, o_pre[:, 0], dict(rel=1e-5, abs=None))
    assert_close("state", st, s_pre, dict(rel=1e-5, abs=None))


def test_decode_host_buffers_round_trip(kda):
    """The binding accepts host tensors: copies in, runs, copies out."""
    q, k, v, a, b, s0 = W.draw((3,), 2, 64, 64, dtype="fp32", s0_std=0.1, seed=4)
    x = W.Inputs("h", q, k, v, a, b, s0.clone())
    state = s0.clone()
    o = kda.decode_step(q, k, v, a, b, state)
    ro, rs = _oracle_decode(x)
    assert o.device.type == "cpu"
    assert_close("o", o, ro, tol_for(torch.float32))
    assert_close("state", state, rs, tol_for(torch.float32))
