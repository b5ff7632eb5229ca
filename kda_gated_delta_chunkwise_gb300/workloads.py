"""Seeded synthetic inputs for the KDA workloads.

This module holds no arithmetic of the method itself: it only draws the
inputs (q, k, v, the gates alpha and beta, an initial state and, for packed
batches, cu_seqlens) that both the CUDA library and the float64 oracle
consume. Everything is drawn on the host with ``numpy.random.default_rng``
(PCG64, identical on x86 and aarch64) in a fixed order:

    sequence lengths (packed batches only), q, k, v, beta logits,
    alpha logits, initial state

q and k are drawn as fp32 N(0,1), L2-normalised per (token, head) over d_k in
fp32, and only then rounded to the kernel dtype, so the oracle sees exactly
the rounded values the GPU sees. beta = sigmoid(N(0,1)). alpha =
exp(-softplus(N(0,1)) * scale) per channel, scale either one number or one
per key channel. The gates stay fp32.

Workloads (sizes as used by the tests and the benchmark):

* ``fwd_fp32_small``:   B=1, H=1, T=256, d=64, fp32, alpha scale 0.1, S0=0
* ``prefill_4x16x4096``: B=4, H=16, T=4096, d=128, bf16, scale 0.05, S0=0
* ``prefill_long_131k``: B=1, H=32, T=131072, d=128, bf16, channels
  c < d/2 with scale 1e-4 and c >= d/2 with scale 0.2, S0 ~ N(0, 0.01^2)
* ``decode_256x32``:     256 sequences x H=32, one token, d=128, bf16,
  scale 0.1, S ~ N(0, 0.1^2)
* ``varlen_64seq``:      64 packed sequences, lengths
  round(lognormal(8, 1)) clipped to [512, 32768] (306,055 tokens at seed 0),
  H=16, d=128, bf16, scale 0.1, per-sequence S0 ~ N(0, 0.01^2)
* ``varlen_64seq_1m``:   the same lengths scaled to about 2^20 tokens in all
  and re-clipped, each sequence drawn from its own generator

``to_mxfp8`` quantises a tensor to FP8 E4M3 with one power-of-two scale per
32 consecutive elements of the last axis (the MX block format) for the FP8
input path; the kernels and the oracle then see the same dequantised values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class Inputs:
    """One batch of inputs, all CPU tensors in the kernel's layouts."""
    name: str
    q: torch.Tensor             # [B, T, H, dk] or packed [T_total, H, dk]
    k: torch.Tensor
    v: torch.Tensor             # [..., H, dv]
    alpha: torch.Tensor         # fp32 [..., H, dk]
    beta: torch.Tensor          # fp32 [..., H]
    initial_state: torch.Tensor | None  # fp32 [N, H, dk, dv] or None (zeros)
    cu_seqlens: torch.Tensor | None = None  # int32 [N + 1] for packed batches
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        if self.cu_seqlens is not None:
            return int(self.cu_seqlens.numel() - 1)
        return int(self.q.shape[0])

    def tensors(self):
        return (self.q, self.k, self.v, self.alpha, self.beta)


def _normal(rng, shape, dtype=np.float32):
    return rng.standard_normal(size=shape, dtype=np.float32).astype(dtype, copy=False)


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-6))).astype(np.float32)


def _to(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(DTYPES[dtype])


def draw(lead: tuple, H: int, dk: int, dv: int, *, dtype: str = "bf16",
         alpha_scale=0.1, s0_std: float | None = None, n_states: int | None = None,
         normalise_qk: bool = True, rng=None, seed: int = 0):
    """Draw q, k, v, alpha, beta (and S0) with leading shape ``lead``.

    alpha_scale: a number, or an array of d_k per-channel scales.
    s0_std: standard deviation of the initial state (None -> no state).
    n_states: number of sequences for the initial state (defaults to lead[0]).
    """
    rng = rng if rng is not None else np.random.default_rng(seed)
    q = _normal(rng, (*lead, H, dk))
    k = _normal(rng, (*lead, H, dk))
    v = _normal(rng, (*lead, H, dv))
    if normalise_qk:
        q = _l2_normalise(q)
        k = _l2_normalise(k)
    b_logit = _normal(rng, (*lead, H)).astype(np.float64)
    beta = (1.0 / (1.0 + np.exp(-b_logit))).astype(np.float32)
    a_logit = _normal(rng, (*lead, H, dk)).astype(np.float64)
    scale = np.asarray(alpha_scale, dtype=np.float64)
    alpha = np.exp(-np.logaddexp(0.0, a_logit) * scale).astype(np.float32)
    s0 = None
    if s0_std is not None:
        n = lead[0] if n_states is None else n_states
        s0 = torch.from_numpy(_normal(rng, (n, H, dk, dv)) * np.float32(s0_std))
    return (_to(q, dtype), _to(k, dtype), _to(v, dtype), torch.from_numpy(alpha),
            torch.from_numpy(beta), s0)


def batched(B: int, T: int, H: int, dk: int = 128, dv: int = 128, *, dtype="bf16",
            alpha_scale=0.1, s0_std=None, seed=0, name="batched") -> Inputs:
    """A [B, T, H, d] batch of equal-length sequences."""
    q, k, v, a, b, s0 = draw((B, T), H, dk, dv, dtype=dtype, alpha_scale=alpha_scale,
                             s0_std=s0_std, seed=seed)
    return Inputs(name, q, k, v, a, b, s0, None,
                  dict(B=B, T=T, H=H, dk=dk, dv=dv, dtype=dtype))


def varlen_lengths(n_seqs: int, rng, mu=8.0, sigma=1.0, lo=512, hi=32768) -> np.ndarray:
    """Sequence lengths round(lognormal(mu, sigma)) clipped to [lo, hi]."""
    return np.clip(np.rint(rng.lognormal(mu, sigma, n_seqs)), lo, hi).astype(np.int64)


def packed(lengths, H: int, dk: int = 128, dv: int = 128, *, dtype="bf16",
           alpha_scale=0.1, s0_std=0.01, seed=0, rng=None, name="packed") -> Inputs:
    """Sequences of the given lengths packed along the token axis."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(lengths.size + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    q, k, v, a, b, s0 = draw((int(cu[-1]),), H, dk, dv, dtype=dtype,
                             alpha_scale=alpha_scale, s0_std=s0_std,
                             n_states=lengths.size, rng=rng)
    return Inputs(name, q, k, v, a, b, s0, torch.from_numpy(cu),
                  dict(N=int(lengths.size), T_total=int(cu[-1]), H=H, dk=dk, dv=dv,
                       dtype=dtype))


def split_scales(dk: int, slow=1e-4, fast=0.2) -> np.ndarray:
    """Per-channel alpha scales: c < dk/2 slow, c >= dk/2 fast."""
    s = np.full(dk, fast, dtype=np.float64)
    s[: dk // 2] = slow
    return s


# ---- the five named workloads ------------------------------------------------

def fwd_fp32_small(seed=0) -> Inputs:
    x = batched(1, 256, 1, 64, 64, dtype="fp32", alpha_scale=0.1, seed=seed,
                name="fwd_fp32_small")
    return x


def prefill_4x16x4096(seed=0, B=4, H=16, T=4096) -> Inputs:
    return batched(B, T, H, 128, 128, dtype="bf16", alpha_scale=0.05, seed=seed,
                   name=f"prefill_{B}x{H}x{T}")


def prefill_long_131k(seed=0, T=131072, H=32) -> Inputs:
    return batched(1, T, H, 128, 128, dtype="bf16", alpha_scale=split_scales(128),
                   s0_std=0.01, seed=seed, name=f"prefill_long_{T}x{H}")


def decode_256x32(seed=0, N=256, H=32) -> Inputs:
    """One decode token per sequence: tensors are [N, H, d]; state [N, H, d, d]."""
    q, k, v, a, b, s0 = draw((N,), H, 128, 128, dtype="bf16", alpha_scale=0.1,
                             s0_std=0.1, seed=seed)
    return Inputs(f"decode_{N}x{H}", q, k, v, a, b, s0, None,
                  dict(N=N, H=H, dk=128, dv=128, dtype="bf16"))


def varlen_64seq(seed=0, n_seqs=64, H=16, rescale_to=None) -> Inputs:
    """Packed lognormal-length batch; rescale_to scales the lengths so that
    they total about that many tokens (then re-clips)."""
    rng = np.random.default_rng(seed)
    L = varlen_lengths(n_seqs, rng)
    if rescale_to is not None:
        L = np.clip(np.rint(L * (rescale_to / L.sum())), 512, 32768).astype(np.int64)
    return packed(L, H, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.01, rng=rng,
                  name=f"varlen_{n_seqs}seq")


def packed_per_sequence(lengths, H: int, dk: int = 128, dv: int = 128, *, dtype="bf16",
                        alpha_scale=0.1, s0_std=0.01, seed=0, name="packed", threads=16) -> Inputs:
    """Sequences of the given lengths packed along the token axis, each drawn
    from its own generator ``default_rng([seed, n])`` (q, k, v, beta logits,
    alpha logits, S0 of that sequence, in that order) and rounded to the
    kernel dtype sequence by sequence. No full-size fp32 temporary of q, k or
    v ever exists, and the sequences are drawn on ``threads`` host threads, so
    batches of millions of tokens stay cheap to make. (A different random
    stream from :func:`packed`, which draws every tensor for the whole batch
    at once.)"""
    import concurrent.futures as cf

    lengths = np.asarray(lengths, dtype=np.int64)
    N = int(lengths.size)
    cu = np.zeros(N + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    Tt = int(cu[-1])
    tdt = DTYPES[dtype]
    q = torch.empty((Tt, H, dk), dtype=tdt)
    k = torch.empty((Tt, H, dk), dtype=tdt)
    v = torch.empty((Tt, H, dv), dtype=tdt)
    alpha = torch.empty((Tt, H, dk), dtype=torch.float32)
    beta = torch.empty((Tt, H), dtype=torch.float32)
    s0 = torch.empty((N, H, dk, dv), dtype=torch.float32) if s0_std is not None else None

    def one(n):
        lo, hi = int(cu[n]), int(cu[n + 1])
        qn, kn, vn, an, bn, sn = draw((hi - lo,), H, dk, dv, dtype=dtype, alpha_scale=alpha_scale,
                                      s0_std=s0_std, n_states=1, rng=np.random.default_rng([seed, n]))
        q[lo:hi], k[lo:hi], v[lo:hi], alpha[lo:hi], beta[lo:hi] = qn, kn, vn, an, bn
        if s0 is not None:
            s0[n] = sn[0]

    with cf.ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        list(ex.map(one, range(N)))
    return Inputs(name, q, k, v, alpha, beta, s0, torch.from_numpy(cu.astype(np.int32)),
                  dict(N=N, T_total=Tt, H=H, dk=dk, dv=dv, dtype=dtype))


def varlen_lengths_rescaled(n_seqs=64, total=1 << 20, seed=0, lo=512, hi=32768) -> np.ndarray:
    """The lengths of ``varlen_64seq`` scaled by one common factor so that,
    rounded and re-clipped to [lo, hi], they total as close to ``total`` as
    that factor can bring them (bisection on the factor: the clip at ``hi``
    takes tokens away, so the plain ratio total / sum falls short). The second
    reading of the packed workload's "about a million tokens"."""
    L = varlen_lengths(n_seqs, np.random.default_rng(seed))

    def lengths(f):
        return np.clip(np.rint(L * f), lo, hi).astype(np.int64)

    a, b = 0.0, 2.0 * hi / max(1, int(L.min()))
    for _ in range(100):
        m = 0.5 * (a + b)
        if lengths(m).sum() < total:
            a = m
        else:
            b = m
    la, lb = lengths(a), lengths(b)
    return la if abs(int(la.sum()) - total) <= abs(int(lb.sum()) - total) else lb


def varlen_64seq_1m(seed=0, n_seqs=64, H=16, total=1 << 20) -> Inputs:
    """The packed lognormal workload at about a million tokens: the lengths of
    ``varlen_64seq`` rescaled (:func:`varlen_lengths_rescaled`), every
    sequence drawn on its own (:func:`packed_per_sequence`)."""
    L = varlen_lengths_rescaled(n_seqs, total, seed)
    return packed_per_sequence(L, H, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.01, seed=seed,
                               name=f"varlen_{n_seqs}seq_{int(L.sum())}tok")


MX_BLOCK = 32


def to_mxfp8(x: torch.Tensor):
    """FP8 E4M3 codes and E8M0 block scales of ``x`` (last axis in blocks of
    32): scale 2^e with e = ceil(log2(amax / 448)) per block, so no code
    saturates; codes round to nearest even. Returns ``(codes uint8, scales
    uint8 [..., d/32], values float32)`` where ``values`` are the exact
    dequantised numbers (code value x 2^e) both sides consume."""
    xf = x.float()
    d = xf.shape[-1]
    if d % MX_BLOCK:
        raise ValueError("the last axis must be a multiple of 32")
    blocks = xf.reshape(*xf.shape[:-1], d // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.ceil(torch.log2(amax / 448.0)), torch.zeros_like(amax))
    e = e.clamp(-126, 127)
    scaled = blocks / torch.exp2(e)[..., None]
    codes = scaled.to(torch.float8_e4m3fn)
    values = (codes.float() * torch.exp2(e)[..., None]).reshape(xf.shape)
    scales = (e + 127).to(torch.uint8)
    return codes.view(torch.uint8).reshape(xf.shape).contiguous(), scales.contiguous(), values.contiguous()
