"""GPU parity of kda_prefill_backward against the float64 gradient oracle.

The loss is L = sum_t <d_o_t, o_t> + <dS_T, S_T> with random d_o and dS_T;
every gradient (q, k, v, alpha, beta, S_0) is compared element by element
with ``oracle.backward`` on the same seeded inputs. The kernels compute in
fp32 whatever the input dtype, so fp32 inputs are held to rel-L2 <= 1e-4 and
bf16 inputs (whose rounded values both sides consume) to the bf16 criterion
rel-L2 <= 5e-3, here on gradients rather than unit-scale outputs, so with a
max-abs bound relative to the tensor's largest reference entry.
"""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, rel_l2, to64

pytestmark = pytest.mark.gpu
KEYS = ("dq", "dk", "dv", "dalpha", "dbeta", "d_initial_state")


def _upstream(x: W.Inputs, seed: int):
    r = np.random.default_rng(seed)
    d_o = torch.from_numpy(r.standard_normal(x.v.shape, dtype=np.float32)).to(x.v.dtype)
    B, _, H, dk = x.q.shape
    dsT = torch.from_numpy(r.standard_normal((B, H, dk, x.v.shape[-1]), dtype=np.float32))
    return d_o, dsT


def _run(kda, x, d_o, dsT):
    d = torch.device("cuda")
    s0 = None if x.initial_state is None else x.initial_state.to(d)
    g = kda.prefill_backward(*(t.to(d) for t in x.tensors()), d_o.to(d), initial_state=s0,
                             d_final_state=None if dsT is None else dsT.to(d))
    torch.cuda.synchronize()
    return {k_: v_.cpu() for k_, v_ in g.items()}


def _check(kda, x, seed=0, with_final=True, rel=None):
    d_o, dsT = _upstream(x, seed)
    if not with_final:
        dsT = None
    g = _run(kda, x, d_o, dsT)
    ref = oracle.backward(*x.tensors(), d_o, dsT, initial_state=x.initial_state)
    rel = rel if rel is not None else (1e-4 if x.q.dtype == torch.float32 else 5e-3)
    for key in KEYS:
        r = ref[key]
        tol = dict(rel=rel, abs=max(1e-6, rel * 4 * float(np.abs(r).max())))
        assert_close(key, g[key], r, tol)
    return g, ref


def test_backward_fp32_small(kda):
    """B=1, H=1, T=256, d=64, fp32 (the small forward workload) with S0."""
    x = W.fwd_fp32_small()
    x.initial_state = torch.from_numpy(np.random.default_rng(3).standard_normal((1, 1, 64, 64), dtype=np.float32) * 0.1)
    _check(kda, x)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
def test_backward_ragged_and_head_sizes(kda, T, dk, dv):
    x = W.batched(2, T, 2, dk, dv, dtype="fp32", alpha_scale=0.2, s0_std=0.05, seed=T + dk)
    _check(kda, x, seed=T)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_backward_bf16_head_sizes(kda, dk, dv):
    """bf16 inputs with d_k or d_v = 64 (the other template instances of every
    pass), two full chunks and a ragged tail, with a token-level chunk."""
    x = W.batched(2, 150, 2, dk, dv, dtype="bf16", alpha_scale=0.2, s0_std=0.05, seed=60 + dk + dv)
    x.alpha[1, 70:90, 0, 3] = 1e-3  # one channel decays past e^-80 in the second chunk of head 0
    _check(kda, x, seed=61)


def test_varlen_backward_small_heads(kda):
    """Packed sequences with d_k = d_v = 64 on bf16 inputs against the oracle."""
    x = W.packed([70, 0, 129, 5], 2, 64, 64, dtype="bf16", s0_std=0.05, seed=62)
    d_o, dsT = _packed_upstream(x, 63)
    d = torch.device("cuda")
    q, k, v, a, b = (t.to(d) for t in x.tensors())
    g = kda.varlen_prefill_backward(q, k, v, a, b, d_o.to(d), x.cu_seqlens.to(d), x.initial_state.to(d), dsT.to(d))
    torch.cuda.synchronize()
    ref = oracle.backward(*x.tensors(), d_o, dsT, cu_seqlens=x.cu_seqlens, initial_state=x.initial_state)
    for key in KEYS:
        r = ref[key]
        assert_close(key, g[key].cpu(), r, dict(rel=5e-3, abs=max(1e-6, 5e-3 * 4 * float(np.abs(r).max()))))


def test_backward_without_final_state_gradient_or_initial_state(kda):
    x = W.batched(1, 200, 3, 128, 128, dtype="fp32", alpha_scale=0.1, seed=7)
    assert x.initial_state is None
    _check(kda, x, seed=1, with_final=False)


def test_backward_bf16_ragged(kda):
    x = W.batched(2, 333, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=9)
    _check(kda, x, seed=2)


def test_backward_strong_decay_chunks(kda):
    """Chunks whose gates decay past the factorised range (alpha = 0 tokens,
    one channel at 1e-3 for 20 tokens, e^-103 over a chunk) take the
    token-level reverse steps."""
    x = W.batched(1, 300, 2, 128, 128, dtype="fp32", alpha_scale=0.1, s0_std=0.05, seed=5)
    x.alpha[0, 10, 0, :] = 0.0
    x.alpha[0, 70:90, 1, 5] = 1e-3
    x.alpha[0, 200:264, 0, :64] = 0.2
    _check(kda, x, seed=3)


def test_backward_prefill_4x16x4096(kda):
    """The benchmark workload (B=4, H=16, T=4096, d=128, bf16 q/k/v): every
    gradient of every (sequence, head) against the oracle."""
    x = W.prefill_4x16x4096()
    g, ref = _check(kda, x, seed=4)
    for key in KEYS:
        print(f"{key}: rel-L2 {rel_l2(g[key], ref[key]):.2e}")


def test_backward_is_deterministic(kda):
    x = W.batched(2, 500, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=12)
    d_o, dsT = _upstream(x, 5)
    g1 = _run(kda, x, d_o, dsT)
    g2 = _run(kda, x, d_o, dsT)
    for key in KEYS:
        assert torch.equal(g1[key], g2[key]), key


def test_backward_zero_length(kda):
    d = torch.device("cuda")
    e = torch.empty(2, 0, 3, 64, device=d)
    dsT = torch.randn(2, 3, 64, 64, device=d)
    g = kda.prefill_backward(e, e, e, e, torch.empty(2, 0, 3, device=d), e, d_final_state=dsT)
    torch.cuda.synchronize()
    torch.testing.assert_close(g["d_initial_state"], dsT, rtol=0, atol=0)


@pytest.mark.parametrize("gate", ["scalar", "none"])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_backward_gate_kinds(kda, gate, dtype):
    """Scalar gate (Gated DeltaNet) and no gate (the delta rule): the oracle
    runs the per-channel gate expanded from them (alpha repeated over the
    channels, or all ones); the scalar gate's gradient is the sum over the
    channels of the per-channel one. Includes a chunk decaying past e^-80 (a
    token-level chunk) for the scalar gate."""
    x = W.batched(2, 200, 2, 128, 128, dtype=dtype, alpha_scale=0.1, s0_std=0.05, seed=40)
    B, T, H, dk = x.q.shape
    a_s = x.alpha[..., 0].contiguous()
    if gate == "scalar":
        a_s[0, 70:134, 1] = 0.2  # e^-103 over one chunk of head 1
    d_o, dsT = _upstream(x, 41)
    d = torch.device("cuda")
    g = kda.prefill_backward(x.q.to(d), x.k.to(d), x.v.to(d), None if gate == "none" else a_s.to(d), x.beta.to(d),
                             d_o.to(d), initial_state=x.initial_state.to(d), d_final_state=dsT.to(d), gate=gate)
    torch.cuda.synchronize()
    full = oracle.expand_gate(a_s.numpy(), gate, (B, T, H), dk)
    ref = oracle.backward(x.q, x.k, x.v, full, x.beta, d_o, dsT, initial_state=x.initial_state)
    rel = 1e-4 if dtype == "fp32" else 5e-3
    for key in ("dq", "dk", "dv", "dbeta", "d_initial_state"):
        r = ref[key]
        assert_close(key, g[key].cpu(), r, dict(rel=rel, abs=max(1e-6, rel * 4 * float(np.abs(r).max()))))
    if gate == "none":
        assert g["dalpha"] is None
    else:
        r = ref["dalpha"].sum(axis=-1)
        assert_close("dalpha", g["dalpha"].cpu(), r, dict(rel=rel, abs=max(1e-6, rel * 4 * float(np.abs(r).max()))))


def _packed_upstream(x, seed):
    r = np.random.default_rng(seed)
    d_o = torch.from_numpy(r.standard_normal(x.v.shape, dtype=np.float32)).to(x.v.dtype)
    N, H, dk, dv = x.num_seqs, x.q.shape[1], x.q.shape[2], x.v.shape[-1]
    dsT = torch.from_numpy(r.standard_normal((N, H, dk, dv), dtype=np.float32))
    return d_o, dsT


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_varlen_backward_bitexact_and_oracle(kda, dtype):
    """Packed sequences (lengths 130, 1, 64, 0, 257, 63, 65): every sequence's
    gradients are bitwise those of the equal-length backward on it alone, and
    the whole packed result matches the oracle."""
    x = W.packed([130, 1, 64, 0, 257, 63, 65], 3, 128, 128, dtype=dtype, s0_std=0.05, seed=50)
    d_o, dsT = _packed_upstream(x, 51)
    d = torch.device("cuda")
    q, k, v, a, b = (t.to(d) for t in x.tensors())
    cu, s0, do_d, dsT_d = x.cu_seqlens.to(d), x.initial_state.to(d), d_o.to(d), dsT.to(d)
    status = torch.full((1,), -1, dtype=torch.int32, device=d)
    g = kda.varlen_prefill_backward(q, k, v, a, b, do_d, cu, s0, dsT_d, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_OK
    cuh = x.cu_seqlens.tolist()
    for n in range(len(cuh) - 1):
        lo, hi = cuh[n], cuh[n + 1]
        gn = kda.prefill_backward(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], a[None, lo:hi], b[None, lo:hi],
                                  do_d[None, lo:hi], s0[n:n + 1], dsT_d[n:n + 1])
        for key in ("dq", "dk", "dv", "dalpha", "dbeta"):
            assert torch.equal(g[key][lo:hi], gn[key][0]), f"sequence {n}: {key} differs from its own backward"
        assert torch.equal(g["d_initial_state"][n], gn["d_initial_state"][0]), f"sequence {n}: dS0 differs"
    ref = oracle.backward(*x.tensors(), d_o, dsT, cu_seqlens=x.cu_seqlens, initial_state=x.initial_state)
    rel = 1e-4 if dtype == "fp32" else 5e-3
    for key in KEYS:
        r = ref[key]
        assert_close(key, g[key].cpu(), r, dict(rel=rel, abs=max(1e-6, rel * 4 * float(np.abs(r).max()))))


def test_varlen_backward_bad_cu_seqlens_sets_status(kda):
    x = W.packed([40, 50, 60], 2, 64, 64, dtype="fp32", s0_std=0.05, seed=52)
    d_o, dsT = _packed_upstream(x, 53)
    d = torch.device("cuda")
    q, k, v, a, b = (t.to(d) for t in x.tensors())
    cu = x.cu_seqlens.to(d).clone()
    cu[1] = 100  # decreasing
    status = torch.full((1,), -1, dtype=torch.int32, device=d)
    kda.varlen_prefill_backward(q, k, v, a, b, d_o.to(d), cu, x.initial_state.to(d), dsT.to(d),
                                device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_BAD_CU_SEQLENS


def test_varlen_backward_64seq_full(kda):
    """The packed workload of 64 lognormal-length sequences (306,055 tokens,
    16 heads, d = 128, bf16): every gradient element of the packed backward
    against the oracle, which runs sequence by sequence (host memory stays
    bounded), with rel-L2 over each whole gradient tensor."""
    from _parity import ErrAccum
    x = W.varlen_64seq()
    d_o, dsT = _packed_upstream(x, 70)
    d = torch.device("cuda")
    q, k, v, a, b = (t.to(d) for t in x.tensors())
    g = kda.varlen_prefill_backward(q, k, v, a, b, d_o.to(d), x.cu_seqlens.to(d), x.initial_state.to(d), dsT.to(d))
    torch.cuda.synchronize()
    g = {key: val.cpu() for key, val in g.items()}
    acc = {key: ErrAccum(key) for key in KEYS}
    top = dict.fromkeys(KEYS, 0.0)
    cu = x.cu_seqlens.tolist()
    for n in range(len(cu) - 1):
        lo, hi = cu[n], cu[n + 1]
        ref = oracle.backward(x.q[lo:hi], x.k[lo:hi], x.v[lo:hi], x.alpha[lo:hi], x.beta[lo:hi], d_o[lo:hi],
                              dsT[n:n + 1], cu_seqlens=np.array([0, hi - lo], dtype=np.int32),
                              initial_state=x.initial_state[n:n + 1])
        for key in KEYS:
            mine = g[key][n:n + 1] if key == "d_initial_state" else g[key][lo:hi]
            acc[key].add(mine, ref[key])
            top[key] = max(top[key], float(np.abs(ref[key]).max()) if ref[key].size else 0.0)
    for key in KEYS:
        acc[key].check(dict(rel=5e-3, abs=5e-3 * 4 * top[key]))


@pytest.mark.slow
def test_backward_long_131k_full(kda):
    """The long-context workload (1 sequence x 32 heads x 131,072 tokens, split
    decay scales): every gradient element against the oracle, which runs 4
    heads at a time (host memory stays bounded)."""
    from _parity import ErrAccum
    x = W.prefill_long_131k()
    d_o, dsT = _upstream(x, 71)
    d = torch.device("cuda")
    g = kda.prefill_backward(*(t.to(d) for t in x.tensors()), d_o.to(d), initial_state=x.initial_state.to(d),
                             d_final_state=dsT.to(d))
    torch.cuda.synchronize()
    g = {key: val.cpu() for key, val in g.items()}
    acc = {key: ErrAccum(key) for key in KEYS}
    top = dict.fromkeys(KEYS, 0.0)
    qc, kc, vc, ac, bc = x.tensors()
    for h0 in range(0, x.q.shape[2], 4):
        hs = slice(h0, h0 + 4)
        ref = oracle.backward(qc[:, :, hs], kc[:, :, hs], vc[:, :, hs], ac[:, :, hs], bc[:, :, hs], d_o[:, :, hs],
                              dsT[:, hs], initial_state=x.initial_state[:, hs])
        for key in KEYS:
            mine = g[key][:, hs] if key == "d_initial_state" else g[key][:, :, hs]
            acc[key].add(mine, ref[key])
            top[key] = max(top[key], float(np.abs(ref[key]).max()))
        del ref
    for key in KEYS:
        acc[key].check(dict(rel=5e-3, abs=5e-3 * 4 * top[key]))
