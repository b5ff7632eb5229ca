"""Brute-force KDA with explicit transition matrices (tiny inputs only).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the web page "研究KimiK3，我发现大模型正在学会“管理自己的计算”"
(pwwt.cn), §五: information written at token j reaches token t through the
product A_t A_{t-1} ... A_{j+1}, with A_i = (I - beta_i k_i k_i^T) Diag(alpha_i)
(§四 gives the same A_i as the KDA update's linear part), and §六's
S_t = A_t S_{t-1} + B_t with B_t = beta_t k_t v_t^T. Unrolling that
recursion gives the closed form used here,

    S_t = (A_t ... A_1) S_0 + sum_{j<=t} (A_t ... A_{j+1}) beta_j k_j v_j^T,
    o_t = S_t^T q_t                                  (§二.1 read-out)

evaluated with every A_i formed as a dense d_k x d_k matrix and every product
multiplied out from scratch for every t: O(T^2 d_k^3), so T <= 16, d <= 8.
This shares no arithmetic with the C oracle's rank-1 recurrence.
"""
from __future__ import annotations

import numpy as np


def transition(k_i: np.ndarray, alpha_i: np.ndarray, beta_i: float) -> np.ndarray:
    """A_i = (I - beta_i k_i k_i^T) Diag(alpha_i)  (§五)."""
    dk = k_i.shape[0]
    return (np.eye(dk) - beta_i * np.outer(k_i, k_i)) @ np.diag(alpha_i)


def chain(A: list[np.ndarray], lo: int, hi: int, dk: int) -> np.ndarray:
    """A_hi A_{hi-1} ... A_{lo}  (identity when hi < lo); 1-based token ids."""
    M = np.eye(dk)
    for i in range(lo, hi + 1):
        M = A[i - 1] @ M
    return M


def run_head(q, k, v, alpha, beta, s0=None):
    """One head. q, k, alpha: [T, dk]; v: [T, dv]; beta: [T]; s0: [dk, dv]."""
    q, k, v, alpha, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha, beta))
    T, dk = k.shape
    dv = v.shape[1]
    if T > 64 or dk > 16:
        raise ValueError("brute force is for tiny inputs only")
    S0 = np.zeros((dk, dv)) if s0 is None else np.asarray(s0, dtype=np.float64)
    A = [transition(k[i], alpha[i], beta[i]) for i in range(T)]
    o = np.zeros((T, dv))
    S_t = S0
    for t in range(1, T + 1):
        S_t = chain(A, 1, t, dk) @ S0
        for j in range(1, t + 1):
            S_t = S_t + chain(A, j + 1, t, dk) @ (beta[j - 1] * np.outer(k[j - 1], v[j - 1]))
        o[t - 1] = S_t.T @ q[t - 1]
    return o, S_t


def run(q, k, v, alpha, beta, s0=None):
    """Batched brute force. q, k, alpha: [B, T, H, dk]; v: [B, T, H, dv];
    beta: [B, T, H]; s0: [B, H, dk, dv] or None. Returns (o, S_T)."""
    q, k, v, alpha, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    sT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            o[b, :, h], sT[b, h] = run_head(q[b, :, h], k[b, :, h], v[b, :, h],
                                            alpha[b, :, h], beta[b, :, h],
                                            None if s0 is None else s0[b, h])
    return o, sT
