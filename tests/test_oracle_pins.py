"""Pins for the float64 oracle: nothing here trusts the oracle's own formula.

Each test checks the oracle against something the KDA pages or plain
mathematics fix independently of the oracle's rank-1 recurrence:

* hand-derived worked examples in exact fractions (tests/golden/);
* the explicit transition-matrix product (K3 essay §五) on tiny inputs;
* closed forms: exact retrieval (§三), decay only (§四 with beta = 0),
  orthonormal keys (gated linear attention, §二.1 + §四), the scalar-gate
  Gated DeltaNet form (§四);
* invariants: state passing / split invariance (§六's S_t = A_t S_{t-1} + B_t),
  linearity in (v, S0), per-sequence independence of packed batches, and the
  contraction bound that follows from ||(I - beta k k^T) Diag(alpha)||_2 <= 1.

The K3 essay is the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
(pwwt.cn/news/3763336).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, B, T, H, dk, dv, unit_k=False, s0=True):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    alpha = rng.uniform(0.05, 1.0, (B, T, H, dk))
    beta = rng.uniform(0.0, 1.0, (B, T, H))
    S0 = rng.standard_normal((B, H, dk, dv)) if s0 else None
    return q, k, v, alpha, beta, S0


def _frac_array(x):
    return np.vectorize(lambda s: float(Fraction(s)))(np.array(x, dtype=object)).astype(np.float64)


@pytest.mark.parametrize("fname", ["hand_kda_d2x2_t2.json", "hand_kda_d2x3_t1.json"])
def test_hand_worked_examples(fname):
    with open(os.path.join(GOLDEN, fname)) as f:
        g = json.load(f)
    args = [_frac_array(g[n]) for n in ("q", "k", "v", "alpha", "beta")]
    o, sT = oracle.run(*args, initial_state=_frac_array(g["initial_state"]))
    # every value is a dyadic rational: float64 holds it exactly
    np.testing.assert_array_equal(o, _frac_array(g["expected_o"]))
    np.testing.assert_array_equal(sT, _frac_array(g["expected_final_state"]))


@pytest.mark.parametrize("dk,dv,T", [(5, 3, 12), (3, 7, 16), (8, 8, 9), (1, 1, 5)])
def test_brute_force_transition_products(dk, dv, T):
    rng = np.random.default_rng(100 + dk * 10 + dv)
    q, k, v, a, b, S0 = _rand_inputs(rng, 2, T, 2, dk, dv)
    o, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    ob, sb = brute.run(q, k, v, a, b, S0)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sT, sb, rtol=0, atol=1e-12)


def test_brute_force_zero_initial_state():
    rng = np.random.default_rng(7)
    q, k, v, a, b, _ = _rand_inputs(rng, 1, 10, 3, 4, 6, s0=False)
    o, sT = oracle.run(q, k, v, a, b)
    ob, sb = brute.run(q, k, v, a, b, None)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(sT, sb, rtol=0, atol=1e-12)


def test_exact_retrieval():
    """§三: with beta = 1, ||k|| = 1 and alpha = 1 the memory returns v_t for
    k_t right after writing it, whatever it held before."""
    rng = np.random.default_rng(1)
    q, k, v, a, b, S0 = _rand_inputs(rng, 2, 20, 2, 8, 5, unit_k=True)
    a[:] = 1.0
    b[:] = 1.0
    o, _ = oracle.run(k, k, v, a, b, initial_state=S0)  # read with q_t = k_t
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def test_decay_only():
    """§四 with beta = 0: S_t = Diag(alpha_t) S_{t-1}, so S_t = Diag(prod alpha) S0."""
    rng = np.random.default_rng(2)
    B, T, H, dk, dv = 2, 9, 3, 6, 4
    q, k, v, a, b, S0 = _rand_inputs(rng, B, T, H, dk, dv)
    b[:] = 0.0
    o, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    cum = np.cumprod(a, axis=1)  # [B, T, H, dk]
    exp_o = np.einsum("bthi,bthi,bhij->bthj", q, cum, S0)
    exp_s = cum[:, -1, :, :, None] * S0
    np.testing.assert_allclose(o, exp_o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sT, exp_s, rtol=1e-13, atol=1e-13)


def test_orthonormal_keys_gated_linear_attention():
    """k_t = e_t (T <= d_k) and S0 = 0: nothing is ever predicted (v_hat = 0),
    so row j of S is beta_j v_j decayed by the later gates of channel j:
    S_T[j] = beta_j (prod_{s>j} alpha_s[j]) v_j, and
    o_t = sum_{j<=t} beta_j (prod_{j<s<=t} alpha_s[j]) q_t[j] v_j."""
    rng = np.random.default_rng(3)
    T, dk, dv = 6, 7, 3
    q, _, v, a, b, _ = _rand_inputs(rng, 1, T, 1, dk, dv, s0=False)
    k = np.zeros((1, T, 1, dk))
    for t in range(T):
        k[0, t, 0, t] = 1.0
    o, sT = oracle.run(q, k, v, a, b)
    exp_o = np.zeros((T, dv))
    for t in range(T):
        for j in range(t + 1):
            decay = np.prod(a[0, j + 1:t + 1, 0, j])
            exp_o[t] += b[0, j, 0] * decay * q[0, t, 0, j] * v[0, j, 0]
    exp_s = np.zeros((dk, dv))
    for j in range(T):
        exp_s[j] = b[0, j, 0] * np.prod(a[0, j + 1:, 0, j]) * v[0, j, 0]
    np.testing.assert_allclose(o[0, :, 0], exp_o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sT[0, 0], exp_s, rtol=1e-13, atol=1e-13)


def test_scalar_gate_is_gated_deltanet():
    """§四: when alpha_t is the same in every channel the KDA update equals the
    scalar-gate Gated DeltaNet form alpha_t (I - beta k k^T) S + beta k v^T."""
    rng = np.random.default_rng(4)
    T, dk, dv = 11, 5, 4
    q, k, v, _, b, S0 = _rand_inputs(rng, 1, T, 1, dk, dv)
    s = rng.uniform(0.1, 1.0, T)
    a = np.broadcast_to(s[None, :, None, None], (1, T, 1, dk)).copy()
    o, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    S = S0[0, 0].copy()
    for t in range(T):
        kt = k[0, t, 0]
        S = s[t] * (np.eye(dk) - b[0, t, 0] * np.outer(kt, kt)) @ S + b[0, t, 0] * np.outer(kt, v[0, t, 0])
        np.testing.assert_allclose(o[0, t, 0], S.T @ q[0, t, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sT[0, 0], S, rtol=1e-12, atol=1e-12)


def test_gate_acts_before_erase():
    """§四 orders the per-channel decay before the erase/write. With
    alpha != const the other order, Diag(alpha)(I - beta k k^T), differs; the
    oracle must agree with the essay's order and not with the other one."""
    rng = np.random.default_rng(5)
    dk, dv = 4, 3
    q, k, v, a, b, S0 = _rand_inputs(rng, 1, 1, 1, dk, dv)
    _, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    kt, at, bt, vt, S = k[0, 0, 0], a[0, 0, 0], b[0, 0, 0], v[0, 0, 0], S0[0, 0]
    essay = (np.eye(dk) - bt * np.outer(kt, kt)) @ np.diag(at) @ S + bt * np.outer(kt, vt)
    other = np.diag(at) @ (np.eye(dk) - bt * np.outer(kt, kt)) @ S + bt * np.outer(kt, vt)
    np.testing.assert_allclose(sT[0, 0], essay, rtol=1e-13, atol=1e-13)
    assert np.abs(sT[0, 0] - other).max() > 1e-3


def test_state_passing_split_invariance():
    """§六: S_t = A_t S_{t-1} + B_t, so running T1 tokens and then T2 tokens
    from the final state equals one run over T1 + T2 tokens."""
    rng = np.random.default_rng(6)
    q, k, v, a, b, S0 = _rand_inputs(rng, 2, 37, 3, 6, 5)
    o, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    T1 = 15
    o1, s1 = oracle.run(q[:, :T1], k[:, :T1], v[:, :T1], a[:, :T1], b[:, :T1], initial_state=S0)
    o2, s2 = oracle.run(q[:, T1:], k[:, T1:], v[:, T1:], a[:, T1:], b[:, T1:], initial_state=s1)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s2, sT, rtol=0, atol=1e-12)


def test_linear_in_values_and_initial_state():
    """For fixed q, k, alpha, beta the update is affine in v with S0 entering
    linearly: (o, S_T) is linear in the pair (v, S0)."""
    rng = np.random.default_rng(8)
    q, k, v1, a, b, S1 = _rand_inputs(rng, 1, 13, 2, 5, 4)
    v2 = rng.standard_normal(v1.shape)
    S2 = rng.standard_normal(S1.shape)
    c1, c2 = 0.75, -1.5
    oa, sa = oracle.run(q, k, v1, a, b, initial_state=S1)
    ob, sb = oracle.run(q, k, v2, a, b, initial_state=S2)
    oc, sc = oracle.run(q, k, c1 * v1 + c2 * v2, a, b, initial_state=c1 * S1 + c2 * S2)
    np.testing.assert_allclose(oc, c1 * oa + c2 * ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sc, c1 * sa + c2 * sb, rtol=1e-12, atol=1e-12)


def test_packed_sequences_are_independent():
    """Packed sequences are separate recurrences, each from its own S0."""
    rng = np.random.default_rng(9)
    lengths = [5, 1, 0, 9, 3]
    Tt = sum(lengths)
    H, dk, dv = 2, 4, 3
    q = rng.standard_normal((Tt, H, dk))
    k = rng.standard_normal((Tt, H, dk))
    v = rng.standard_normal((Tt, H, dv))
    a = rng.uniform(0.1, 1, (Tt, H, dk))
    b = rng.uniform(0, 1, (Tt, H))
    S0 = rng.standard_normal((len(lengths), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o, sT = oracle.run(q, k, v, a, b, cu_seqlens=cu, initial_state=S0)
    for n, (lo, hi) in enumerate(zip(cu[:-1], cu[1:])):
        on, sn = oracle.run(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], a[None, lo:hi],
                            b[None, lo:hi], initial_state=S0[n:n + 1])
        np.testing.assert_array_equal(o[lo:hi], on[0])
        np.testing.assert_array_equal(sT[n], sn[0])
    # a zero-length sequence keeps its initial state
    np.testing.assert_array_equal(sT[2], S0[2])


def test_contraction_bound():
    """||k|| = 1, beta, alpha in [0,1]: ||S_t||_F <= ||S_{t-1}||_F + beta_t ||v_t||."""
    rng = np.random.default_rng(10)
    q, k, v, a, b, S0 = _rand_inputs(rng, 1, 40, 1, 6, 6, unit_k=True)
    norms = [np.linalg.norm(S0[0, 0])]
    for t in range(40):
        _, s = oracle.run(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], a[:, :t + 1], b[:, :t + 1],
                          initial_state=S0)
        norms.append(np.linalg.norm(s[0, 0]))
    for t in range(40):
        assert norms[t + 1] <= norms[t] + b[0, t, 0] * np.linalg.norm(v[0, t, 0]) + 1e-12


def test_zero_length_and_bad_cu_seqlens():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((4, 1, 2))
    v = rng.standard_normal((4, 1, 3))
    a = np.ones((4, 1, 2))
    b = np.ones((4, 1))
    with pytest.raises(ValueError):
        oracle.run(q, q, v, a, b, cu_seqlens=np.array([0, 3, 2, 4], dtype=np.int32))
    o, sT = oracle.run(q, q, v, a, b, cu_seqlens=np.array([0, 0], dtype=np.int32))
    assert np.all(sT == 0)


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(12)
    q, k, v, a, b, S0 = _rand_inputs(rng, 3, 30, 4, 8, 8)
    o1, s1 = oracle.run(q, k, v, a, b, initial_state=S0, nthreads=1)
    o4, s4 = oracle.run(q, k, v, a, b, initial_state=S0, nthreads=4)
    np.testing.assert_array_equal(o1, o4)
    np.testing.assert_array_equal(s1, s4)


def test_scalar_gate_expansion_is_gated_deltanet():
    """The scalar gate of Gated DeltaNet (§四), given per token and head and
    expanded by oracle.expand_gate, is the per-channel gate repeated over the
    channels: the oracle then follows alpha_t (I - beta k k^T) S + beta k v^T
    with a different alpha in every token and head."""
    rng = np.random.default_rng(41)
    B, T, H, dk, dv = 2, 9, 3, 5, 4
    q, k, v, _, b, S0 = _rand_inputs(rng, B, T, H, dk, dv)
    s = rng.uniform(0.1, 1.0, (B, T, H))
    a = oracle.expand_gate(s, "scalar", (B, T, H), dk)
    assert a.shape == (B, T, H, dk)
    o, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    for bi in range(B):
        for hi in range(H):
            S = S0[bi, hi].copy()
            for t in range(T):
                kt = k[bi, t, hi]
                S = s[bi, t, hi] * (np.eye(dk) - b[bi, t, hi] * np.outer(kt, kt)) @ S \
                    + b[bi, t, hi] * np.outer(kt, v[bi, t, hi])
                np.testing.assert_allclose(o[bi, t, hi], S.T @ q[bi, t, hi], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(sT[bi, hi], S, rtol=1e-12, atol=1e-12)


def test_no_gate_is_the_delta_rule():
    """Without a gate (§三) the update is S = (I - beta k k^T) S + beta k v^T;
    writing two values under the same unit key with beta = 1 leaves only the
    second one (the erase removes the first)."""
    rng = np.random.default_rng(42)
    B, T, H, dk, dv = 1, 12, 2, 6, 3
    q, k, v, _, b, S0 = _rand_inputs(rng, B, T, H, dk, dv)
    a = oracle.expand_gate(None, "none", (B, T, H), dk)
    assert np.all(a == 1.0)
    o, sT = oracle.run(q, k, v, a, b, initial_state=S0)
    for hi in range(H):
        S = S0[0, hi].copy()
        for t in range(T):
            kt = k[0, t, hi]
            S = S - b[0, t, hi] * np.outer(kt, kt @ S) + b[0, t, hi] * np.outer(kt, v[0, t, hi])
            np.testing.assert_allclose(o[0, t, hi], S.T @ q[0, t, hi], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sT[0, hi], S, rtol=1e-12, atol=1e-12)
    # overwrite: same unit key twice, beta = 1, read back with q = k
    u = rng.standard_normal(dk)
    u /= np.linalg.norm(u)
    kk = np.broadcast_to(u, (1, 2, 1, dk)).copy()
    vv = rng.standard_normal((1, 2, 1, dv))
    bb = np.ones((1, 2, 1))
    o2, _ = oracle.run(kk, kk, vv, oracle.expand_gate(None, "none", (1, 2, 1), dk), bb)
    np.testing.assert_allclose(o2[0, 1, 0], vv[0, 1, 0], rtol=0, atol=1e-12)


def test_expand_gate_rejects_wrong_shapes():
    with pytest.raises(ValueError):
        oracle.expand_gate(np.ones((2, 3)), "scalar", (2, 3, 1), 4)
    with pytest.raises(ValueError):
        oracle.expand_gate(np.ones((2, 3, 4)), "channel", (2, 3), 5)
    with pytest.raises(ValueError):
        oracle.expand_gate(None, "sigmoid", (1,), 2)


def test_mxfp8_decoding_fixed_codes():
    """E4M3 code points fixed by the format: 0x38 = 1, 0x40 = 2, 0x7E = 448
    (largest), 0x01 = 2^-9 (smallest subnormal), 0x08 = 2^-6 (smallest
    normal), 0xB8 = -1; 0x7F is NaN; a scale byte t multiplies by 2^(t-127)."""
    codes = np.array([[0x38, 0x40, 0x7E, 0x01, 0x08, 0xB8, 0x00, 0x3C] * 4], dtype=np.uint8)
    v = oracle.dequant_mxfp8(codes, np.array([[127]], dtype=np.uint8))
    np.testing.assert_array_equal(v[0, :8], [1.0, 2.0, 448.0, 2.0 ** -9, 2.0 ** -6, -1.0, 0.0, 1.5])
    v2 = oracle.dequant_mxfp8(codes, np.array([[130]], dtype=np.uint8))
    np.testing.assert_array_equal(v2, v * 8.0)
    assert np.isnan(oracle.dequant_mxfp8(np.full((1, 32), 0x7F, np.uint8), np.array([[127]], np.uint8))).all()


def test_mxfp8_round_trip_of_the_input_generator():
    """The inputs' quantiser and the oracle's decoder agree on every element:
    the dequantised values the generator hands to the kernels are exactly
    the oracle's decoding of its codes and scales, and within half an E4M3
    step of the original numbers."""
    from kda_gated_delta_chunkwise_gb300 import workloads as W
    import torch
    x = torch.randn(7, 3, 128, generator=torch.Generator().manual_seed(5)) * 3.0
    codes, scales, values = W.to_mxfp8(x)
    dec = oracle.dequant_mxfp8(codes.numpy(), scales.numpy())
    np.testing.assert_array_equal(dec, values.double().numpy())
    blk = np.repeat(np.exp2(scales.numpy().astype(np.float64) - 127.0), 32, axis=-1)
    assert np.all(np.abs(dec - x.double().numpy()) <= 2.0 ** -4 * np.maximum(np.abs(x.double().numpy()), 2.0 ** -6 * blk) + 1e-300)
