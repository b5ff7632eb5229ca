"""Fixed workloads for profiling the kernels under ncu.

    python -m kda_gated_delta_chunkwise_gb300.profile_cases CASE [--reps N]

CASE is one of:
  prefill_4x16x4096   the benchmark workload (B=4, H=16, T=4096, d=128, bf16)
  prefill_1x16x4096   a quarter of it (B=1): small enough for full ncu captures
  variants_4x16x4096  the benchmark workload with a scalar gate, with no gate,
                      and with FP8 q, k, v (one launch of each per rep)
  decode_256x32       the decode workload (256 sequences x 32 heads, d=128)
  decode_64x32        a quarter of it, for full ncu captures

Each case draws its seeded inputs, runs the kernel --reps times (default 3)
and synchronises; it prints one line and exits 0 on success.
"""
from __future__ import annotations

import argparse

import torch

from . import _binding as kda
from . import workloads as W


def _prefill(B: int, reps: int):
    dev = torch.device("cuda")
    x = W.prefill_4x16x4096(B=B)
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    o = torch.empty_like(v)
    s = torch.empty((B, 16, 128, 128), dtype=torch.float32, device=dev)
    for _ in range(reps):
        kda.prefill(q, k, v, a, b, None, out=o, final_state=s)
    torch.cuda.synchronize()


def _variants(reps: int):
    dev = torch.device("cuda")
    x = W.prefill_4x16x4096()
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    a_s = a[..., 0].contiguous()
    cq, sq, _ = W.to_mxfp8(q)
    ck, sk, _ = W.to_mxfp8(k)
    cv, sv, _ = W.to_mxfp8(v)
    o = torch.empty_like(v)
    s = torch.empty((4, 16, 128, 128), dtype=torch.float32, device=dev)
    for _ in range(reps):
        kda.prefill(q, k, v, a_s, b, None, gate="scalar", out=o, final_state=s)
        kda.prefill(q, k, v, None, b, None, gate="none", out=o, final_state=s)
        kda.prefill_fp8(cq, ck, cv, sq, sk, sv, a, b, None, out=o, final_state=s)
    torch.cuda.synchronize()


def _decode(N: int, reps: int):
    dev = torch.device("cuda")
    x = W.decode_256x32(N=N)
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    state = x.initial_state.to(dev)
    o = torch.empty_like(v)
    for _ in range(reps):
        kda.decode_step(q, k, v, a, b, state, out=o)
    torch.cuda.synchronize()


CASES = {
    "prefill_4x16x4096": lambda r: _prefill(4, r),
    "prefill_1x16x4096": lambda r: _prefill(1, r),
    "variants_4x16x4096": _variants,
    "decode_256x32": lambda r: _decode(256, r),
    "decode_64x32": lambda r: _decode(64, r),
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    kda.load()
    CASES[args.case](args.reps)
    errs = kda.device_errors()
    if errs:
        raise SystemExit(f"device error word {errs}")
    print(f"{args.case}: {args.reps} runs ok")


if __name__ == "__main__":
    main()
