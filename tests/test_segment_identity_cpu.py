"""The identity the segmented prefill rests on, checked in float64 on the
oracle alone (no GPU, no CUDA library).

The K3 essay (pwwt.cn/news/3763336) writes the update as an affine map of the
state, S_t = A_t S_{t-1} + B_t (§六), with the transition from token j to t
the product A_t ... A_{j+1} (§五). Over a stretch of tokens, then,
S_end = Phi S_start + b, and inside it o_t = S_loc,t^T q_t + S_start^T z_t
with z_t = Phi_t^T q_t. A run of the recurrence with v = 0 from the identity
gives z_t as its outputs and Phi as its final state; a run from zero gives
S_loc (outputs o_loc, final state b). Put together segment by segment, these
must reproduce the whole-sequence result to rounding.
"""
import numpy as np
import pytest

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W


def _split(x, cuts):
    """Per segment (q, k, v, alpha, beta) slices of a B = 1 batch."""
    edges = [0, *cuts, x.q.shape[1]]
    t = [np.asarray(a, dtype=np.float64) for a in x.tensors()]
    return [[a[:, lo:hi] for a in t] for lo, hi in zip(edges[:-1], edges[1:])]


def _segmented(x, cuts):
    """The segmented evaluation, all in float64 through the oracle."""
    H, dk = x.q.shape[2], x.q.shape[3]
    segs = _split(x, cuts)
    s0 = np.asarray(x.initial_state, dtype=np.float64)
    o0, s = oracle.run(*segs[0], initial_state=s0)
    outs = [o0]
    eye = np.broadcast_to(np.eye(dk), (1, H, dk, dk)).copy()
    for q, k, v, a, b in segs[1:]:
        o_loc, b_end = oracle.run(q, k, v, a, b)                          # from zero
        z, phi = oracle.run(q, k, np.zeros(q.shape[:-1] + (dk,)), a, b,  # v = 0, from I
                            initial_state=eye)
        outs.append(o_loc + np.einsum("bthi,bhij->bthj", z, s))
        s = np.einsum("bhim,bhmj->bhij", phi, s) + b_end
    return np.concatenate(outs, axis=1), s


@pytest.mark.parametrize("dk,dv,cuts", [(8, 8, (64, 150)), (8, 5, (1, 2, 250)), (6, 10, (100,))])
def test_segments_reproduce_the_whole_sequence(dk, dv, cuts):
    x = W.batched(1, 300, 2, dk, dv, dtype="fp32", alpha_scale=0.05, s0_std=0.5, seed=dk * 7 + dv)
    x.beta.mul_(0.3)  # slow erasure: the start states matter across whole segments
    o_ref, s_ref = oracle.run(*x.tensors(), initial_state=x.initial_state)
    o, s = _segmented(x, cuts)
    scale_o, scale_s = np.abs(o_ref).max(), np.abs(s_ref).max()
    assert np.abs(o - o_ref).max() <= 1e-12 * max(1.0, scale_o)
    assert np.abs(s - s_ref).max() <= 1e-12 * max(1.0, scale_s)


def test_the_correction_is_needed():
    """Without the S_start terms the later segments are wrong: the pin above
    would catch a combine that dropped them."""
    x = W.batched(1, 300, 2, 8, 8, dtype="fp32", alpha_scale=0.05, s0_std=0.5, seed=3)
    x.beta.mul_(0.3)
    o_ref, _ = oracle.run(*x.tensors(), initial_state=x.initial_state)
    segs = _split(x, (150,))
    o_loc, _ = oracle.run(*segs[1])
    err = np.linalg.norm(o_loc - o_ref[:, 150:]) / np.linalg.norm(o_ref[:, 150:])
    assert err > 1e-2
