"""Pins of the gradient oracle (``oracle.backward``), none of which uses it
to check itself.

The pages give no gradients; the map being differentiated is the KDA update
of the K3 essay §四 with the read-out of §二.1, and the loss is
L = sum_t <do_t, o_t> + <dS_T, S_T>. The oracle's gradients are checked
against
  * central finite differences of the forward oracle (``oracle.run``, a
    separate C file) on every input coordinate of small cases, including
    one that crosses the gradient oracle's 64-token replay stretches;
  * reverse-mode differentiation (torch autograd, float64) of the §四
    update written in its projector form (I - b k k^T) Diag(a) S + b k v^T,
    a different arrangement of the arithmetic from both C files;
  * closed forms: one token from a zero state, and the frozen state
    (alpha = 1, beta = 0) where S_t = S_0 for every t;
  * linearity in (do, dS_T) and independence of packed sequences.
Nothing here touches a GPU.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _inputs(B, T, H, dk, dv, seed, s0=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, dk))
    k = r.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, H, dv))
    alpha = np.exp(-np.logaddexp(0, r.standard_normal((B, T, H, dk))) * 0.3)
    beta = 1 / (1 + np.exp(-r.standard_normal((B, T, H))))
    S0 = 0.3 * r.standard_normal((B, H, dk, dv)) if s0 else None
    do = r.standard_normal((B, T, H, dv))
    dsT = r.standard_normal((B, H, dk, dv))
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0, do=do, dsT=dsT)


def _loss(x, **over):
    y = dict(x, **over)
    o, sT = oracle.run(y["q"], y["k"], y["v"], y["alpha"], y["beta"], initial_state=y["S0"])
    return float(np.sum(o * y["do"]) + np.sum(sT * y["dsT"]))


def _grads(x):
    return oracle.backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["do"], x["dsT"],
                           initial_state=x["S0"])


NAMES = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("alpha", "dalpha"), ("beta", "dbeta"),
         ("S0", "d_initial_state")]


def _fd_check(x, g, coords=None, h=1e-6, tol=2e-7):
    """Central differences on every coordinate (or `coords` random ones per
    tensor); returns the worst scaled error."""
    worst = 0.0
    for name, gname in NAMES:
        base = x[name]
        flat = base.reshape(-1)
        idx = range(flat.size) if coords is None else RNG.choice(flat.size, size=min(coords, flat.size),
                                                                 replace=False)
        for i in idx:
            xp, xm = flat.copy(), flat.copy()
            xp[i] += h
            xm[i] -= h
            fd = (_loss(x, **{name: xp.reshape(base.shape)}) - _loss(x, **{name: xm.reshape(base.shape)})) / (2 * h)
            an = g[gname].reshape(-1)[i]
            err = abs(fd - an) / max(1.0, abs(fd))
            worst = max(worst, err)
            assert err <= tol, f"d{name}[{i}]: finite difference {fd:.9g} vs oracle {an:.9g}"
    return worst


def test_finite_differences_every_coordinate():
    x = _inputs(2, 9, 2, 4, 3, seed=1)
    _fd_check(x, _grads(x))


def test_finite_differences_across_replay_stretches():
    """70 tokens: the reverse pass replays two stretches (64 + 6 tokens) from
    their checkpoints."""
    x = _inputs(1, 70, 1, 4, 3, seed=2)
    _fd_check(x, _grads(x), coords=60)


def test_finite_differences_zero_gates_and_no_initial_state():
    """alpha = 0 on some channels (erasure) and beta above 1: the gradient
    has no 1/alpha anywhere, so it stays exact there."""
    x = _inputs(1, 12, 2, 4, 3, seed=3, s0=False)
    x["alpha"][0, 4, 0, :2] = 0.0
    x["alpha"][0, 7, 1, 3] = 0.0
    x["beta"][0, 5, 1] = 1.7
    g = _grads(x)
    x_fd = dict(x, S0=np.zeros((1, 2, 4, 3)))
    g["S0"] = g["d_initial_state"]
    _fd_check(x_fd, g)


def _autograd(x):
    """Reverse mode through the projector form of the §四 update."""
    t = {n: torch.tensor(x[n], dtype=torch.float64, requires_grad=True) for n in ("q", "k", "v", "alpha", "beta")}
    B, T, H, dk = x["q"].shape
    dv = x["v"].shape[-1]
    S0 = torch.tensor(x["S0"], dtype=torch.float64, requires_grad=True)
    do = torch.tensor(x["do"])
    dsT = torch.tensor(x["dsT"])
    loss = 0.0
    eye = torch.eye(dk, dtype=torch.float64)
    for b in range(B):
        for h in range(H):
            S = S0[b, h]
            for s in range(T):
                kk, bb = t["k"][b, s, h], t["beta"][b, s, h]
                A = (eye - bb * torch.outer(kk, kk)) @ torch.diag(t["alpha"][b, s, h])
                S = A @ S + bb * torch.outer(kk, t["v"][b, s, h])
                loss = loss + torch.dot(S.T @ t["q"][b, s, h], do[b, s, h])
            loss = loss + torch.sum(S * dsT[b, h])
    loss.backward()
    out = {"d" + n: t[n].grad.numpy() for n in ("q", "k", "v")}
    out["dalpha"] = t["alpha"].grad.numpy()
    out["dbeta"] = t["beta"].grad.numpy()
    out["d_initial_state"] = S0.grad.numpy()
    return out


def test_reverse_mode_of_the_projector_form():
    x = _inputs(2, 11, 2, 5, 3, seed=4)
    g, ref = _grads(x), _autograd(x)
    for key in ref:
        np.testing.assert_allclose(g[key], ref[key], rtol=1e-10, atol=1e-12, err_msg=key)


def test_one_token_from_zero_state_closed_form():
    """S_1 = b k v^T, o = b (k.q) v: dq = b (v.do) k, dv = b (k.q) do + b dS^T k,
    dbeta = (k.q)(v.do) + k^T dS v, dk = b (v.do) q + b dS v, dalpha = 0,
    dS_0 = Diag(a) (G - b k (G^T k)^T) with G = dS + q do^T."""
    x = _inputs(1, 1, 1, 4, 3, seed=5, s0=False)
    g = _grads(x)
    q, k, v, a, b = (x[n][0, 0, 0] for n in ("q", "k", "v", "alpha", "beta"))
    do, dS = x["do"][0, 0, 0], x["dsT"][0, 0]
    kq, vdo = k @ q, v @ do
    np.testing.assert_allclose(g["dq"][0, 0, 0], b * vdo * k, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(g["dv"][0, 0, 0], b * kq * do + b * dS.T @ k, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(g["dbeta"][0, 0, 0], kq * vdo + k @ dS @ v, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(g["dk"][0, 0, 0], b * vdo * q + b * dS @ v, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(g["dalpha"][0, 0, 0], np.zeros(4))
    G = dS + np.outer(q, do)
    np.testing.assert_allclose(g["d_initial_state"][0, 0], a[:, None] * (G - b * np.outer(k, G.T @ k)),
                               rtol=1e-13, atol=1e-14)


def test_frozen_state_closed_form():
    """alpha = 1, beta = 0: S_t = S_0, o_t = S_0^T q_t. Then dq_t = S_0 do_t,
    dv = dk = 0, dS_0 = dS_T + sum_t q_t do_t^T, and with G_t = dS_T +
    sum_{s>=t} q_s do_s^T: dalpha_t = rowsum(G_t (.) S_0),
    dbeta_t = (G_t^T k_t) . (v_t - S_0^T k_t)."""
    x = _inputs(1, 6, 1, 4, 3, seed=6)
    x["alpha"][:] = 1.0
    x["beta"][:] = 0.0
    g = _grads(x)
    S0, dS = x["S0"][0, 0], x["dsT"][0, 0]
    q, k, v, do = (x[n][0, :, 0] for n in ("q", "k", "v", "do"))
    np.testing.assert_allclose(g["dq"][0, :, 0], do @ S0.T, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(g["dv"], 0.0)
    np.testing.assert_array_equal(g["dk"], 0.0)
    np.testing.assert_allclose(g["d_initial_state"][0, 0], dS + q.T @ do, rtol=1e-13, atol=1e-14)
    for t in range(6):
        Gt = dS + q[t:].T @ do[t:]
        np.testing.assert_allclose(g["dalpha"][0, t, 0], np.sum(Gt * S0, axis=1), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dbeta"][0, t, 0], (Gt.T @ k[t]) @ (v[t] - S0.T @ k[t]), rtol=1e-12,
                                   atol=1e-13)


def test_linear_in_the_upstream_gradients():
    x = _inputs(1, 20, 2, 4, 3, seed=7)
    g1 = _grads(x)
    x2 = dict(x, do=RNG.standard_normal(x["do"].shape), dsT=RNG.standard_normal(x["dsT"].shape))
    g2 = _grads(x2)
    g12 = _grads(dict(x, do=x["do"] + 2 * x2["do"], dsT=x["dsT"] + 2 * x2["dsT"]))
    for key in g1:
        np.testing.assert_allclose(g12[key], g1[key] + 2 * g2[key], rtol=1e-11, atol=1e-12, err_msg=key)


def test_packed_sequences_are_independent():
    x = _inputs(3, 50, 2, 4, 3, seed=8)
    lens = [50, 17, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    pk = {n: np.concatenate([x[n][i, :lens[i]] for i in range(3)]) for n in ("q", "k", "v", "alpha", "beta", "do")}
    gp = oracle.backward(pk["q"], pk["k"], pk["v"], pk["alpha"], pk["beta"], pk["do"], x["dsT"], cu_seqlens=cu,
                         initial_state=x["S0"])
    for i in range(3):
        sl = {n: x[n][i:i + 1, :lens[i]] for n in ("q", "k", "v", "alpha", "beta", "do")}
        gi = oracle.backward(sl["q"], sl["k"], sl["v"], sl["alpha"], sl["beta"], sl["do"], x["dsT"][i:i + 1],
                             initial_state=x["S0"][i:i + 1])
        for key in ("dq", "dk", "dv", "dalpha", "dbeta"):
            np.testing.assert_array_equal(gp[key][cu[i]:cu[i + 1]], gi[key][0], err_msg=key)
        np.testing.assert_array_equal(gp["d_initial_state"][i], gi["d_initial_state"][0])


def test_zero_length_sequence_passes_the_state_gradient_through():
    x = _inputs(1, 0, 1, 4, 3, seed=9)
    g = _grads(x)
    np.testing.assert_array_equal(g["d_initial_state"], x["dsT"])


@pytest.mark.parametrize("threads", [1, 3])
def test_thread_count_does_not_change_a_bit(threads):
    x = _inputs(2, 30, 3, 4, 3, seed=10)
    g = _grads(x)
    gt = oracle.backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["do"], x["dsT"], initial_state=x["S0"],
                         nthreads=threads)
    for key in g:
        np.testing.assert_array_equal(g[key], gt[key])
