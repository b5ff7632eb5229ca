"""GPU tests of the FP8 input path (MX block format: E4M3 codes, one E8M0
power-of-two scale per 32 channels). The dequantised values are exactly
representable in bf16, so the FP8 prefill must give, bit for bit, what the
bf16 prefill gives on those values; both follow the float64 oracle run on
the values decoded by the oracle's own E4M3 decoder."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _fp8_inputs(B, T, H, seed, alpha_scale=0.1, s0_std=0.05):
    q, k, v, a, b, s0 = W.draw((B, T), H, 128, 128, dtype="fp32", alpha_scale=alpha_scale, s0_std=s0_std,
                               seed=seed)
    (qc, qs, qv), (kc, ks, kv), (vc, vs, vv) = (W.to_mxfp8(t) for t in (q, k, v))
    return dict(codes=(qc, kc, vc), scales=(qs, ks, vs), values=(qv, kv, vv), alpha=a, beta=b, s0=s0)


def _run_both(kda, x, gate="channel", alpha=None):
    a = x["alpha"] if alpha is None else alpha
    ag = None if gate == "none" else a.to(DEV)
    b, s0 = x["beta"].to(DEV), x["s0"].to(DEV)
    qc, kc, vc = (t.to(DEV) for t in x["codes"])
    qs, ks, vs = (t.to(DEV) for t in x["scales"])
    o8, s8 = kda.prefill_fp8(qc, kc, vc, qs, ks, vs, ag, b, s0, gate=gate)
    qv, kv, vv = (t.to(DEV).to(torch.bfloat16) for t in x["values"])
    ob, sb = kda.prefill(qv, kv, vv, ag, b, s0, algo="tc", gate=gate)
    torch.cuda.synchronize()
    return o8, s8, ob, sb


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
@pytest.mark.parametrize("T", [64, 130, 300])
def test_fp8_equals_bf16_on_the_dequantised_values(kda, gate, T):
    x = _fp8_inputs(2, T, 3, seed=40 + T)
    alpha = x["alpha"][..., 0].contiguous() if gate == "scalar" else None
    o8, s8, ob, sb = _run_both(kda, x, gate, alpha)
    assert o8.dtype == torch.bfloat16
    assert torch.equal(o8, ob), "o differs from the bf16 path"
    assert torch.equal(s8, sb), "final state differs from the bf16 path"


def test_fp8_follows_the_oracle(kda):
    x = _fp8_inputs(1, 257, 2, seed=50)
    o8, s8, _, _ = _run_both(kda, x)
    dq = [oracle.dequant_mxfp8(c.numpy(), s.numpy()) for c, s in zip(x["codes"], x["scales"])]
    np.testing.assert_array_equal(dq[0], x["values"][0].double().numpy())  # the decoder agrees with the inputs
    ro, rs = oracle.run(dq[0], dq[1], dq[2], x["alpha"], x["beta"], initial_state=x["s0"])
    tol = tol_for(torch.bfloat16)
    assert_close("o", o8, ro, tol)
    assert_close("state", s8, rs, tol)


def test_fp8_token_loop_chunks(kda):
    """A zero gate in one token and a stretch of tiny gates: those chunks run
    token by token, reading the FP8 codes and scales directly."""
    x = _fp8_inputs(1, 200, 2, seed=51)
    x["alpha"][0, 10, 0, :] = 0.0
    x["alpha"][0, 70:100, 1, 5] = 1e-3
    o8, s8, ob, sb = _run_both(kda, x)
    assert torch.equal(o8, ob) and torch.equal(s8, sb)


def test_fp8_benchmark_size(kda):
    """The 4 x 16 x 4096 workload in FP8: bit for bit the bf16 path on the
    dequantised values."""
    x = _fp8_inputs(4, 4096, 16, seed=52, alpha_scale=0.05, s0_std=None)
    x["s0"] = torch.zeros(4, 16, 128, 128)
    o8, s8, ob, sb = _run_both(kda, x)
    assert torch.equal(o8, ob) and torch.equal(s8, sb)
