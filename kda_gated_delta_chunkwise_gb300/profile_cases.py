"""Fixed workloads for profiling the kernels under ncu.

    python -m kda_gated_delta_chunkwise_gb300.profile_cases CASE [--reps N]

CASE is one of:
  prefill_4x16x4096   the benchmark workload (B=4, H=16, T=4096, d=128, bf16)
  prefill_1x16x4096   a quarter of it (B=1): small enough for full ncu captures
  variants_4x16x4096  the benchmark workload with a scalar gate, with no gate,
                      and with FP8 q, k, v (one launch of each per rep)
  decode_256x32       the decode workload (256 sequences x 32 heads, d=128)
  decode_64x32        a quarter of it, for full ncu captures
  long_131k           one 131,072-token sequence with 32 heads (d=128, bf16)
  long_131k_segmented the same through kda_prefill_segmented (the library's plan)
  long_65k_segmented  half of it (65,536 tokens): small enough for full ncu captures
  varlen_64seq        the packed batch of 64 lognormal-length sequences
  varlen_64seq_1m     the same lengths scaled to 2^20 tokens
  backward_4x16x4096  the gradients of the benchmark workload (kda_prefill_backward)
  backward_1x16x1024  a small case of it, for full ncu captures
  hostlink            no kernel: the host link's copy rates (page-locked host
                      memory to the device, back, and both at once), printed

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


def _long(reps: int):
    dev = torch.device("cuda")
    x = W.prefill_long_131k()
    q, k, v, a, b, s0 = (t.to(dev) for t in (*x.tensors(), x.initial_state))
    o = torch.empty_like(v)
    s = torch.empty_like(s0)
    for _ in range(reps):
        kda.prefill(q, k, v, a, b, s0, out=o, final_state=s)
    torch.cuda.synchronize()


def _long_segmented(reps: int, T: int = 131072):
    dev = torch.device("cuda")
    x = W.prefill_long_131k(T=T)
    q, k, v, a, b, s0 = (t.to(dev) for t in (*x.tensors(), x.initial_state))
    o = torch.empty_like(v)
    s = torch.empty_like(s0)
    T, H = q.shape[1], q.shape[2]
    ws = torch.empty(kda.prefill_segmented_workspace_bytes(T, H), dtype=torch.uint8, device=dev)
    for _ in range(reps):
        kda.prefill_segmented(q, k, v, a, b, s0, out=o, final_state=s, workspace=ws)
    torch.cuda.synchronize()


def _varlen(x, reps: int):
    dev = torch.device("cuda")
    (q, k, v, a, b), cu, s0 = [t.to(dev) for t in x.tensors()], x.cu_seqlens.to(dev), x.initial_state.to(dev)
    o = torch.empty_like(v)
    s = torch.empty_like(s0)
    for _ in range(reps):
        kda.varlen_prefill(q, k, v, a, b, cu, s0, out=o, final_state=s)
    torch.cuda.synchronize()


def _backward(B: int, T: int, reps: int):
    dev = torch.device("cuda")
    x = W.prefill_4x16x4096(B=B, T=T)
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    d_o = torch.randn(v.shape, generator=torch.Generator(device=dev).manual_seed(7), device=dev).to(v.dtype)
    for _ in range(reps):
        kda.prefill_backward(q, k, v, a, b, d_o)
    torch.cuda.synchronize()


def _hostlink(reps: int):
    """Copy rates between page-locked host memory and the device: 256 MiB
    buffers, each direction alone on its own stream, then both directions
    at once on two streams; CUDA events, best of ``reps`` (at least 5)."""
    dev = torch.device("cuda")
    n = 256 << 20
    h_in = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(n, dtype=torch.uint8, device=dev)
    d_out = torch.ones(n, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        best = None
        for _ in range(max(reps, 5)):
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            s1.wait_event(t0)
            s2.wait_event(t0)
            fn()
            e1, e2 = torch.cuda.Event(), torch.cuda.Event()
            e1.record(s1)
            e2.record(s2)
            torch.cuda.current_stream().wait_event(e1)
            torch.cuda.current_stream().wait_event(e2)
            t1.record()
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1)
            best = ms if best is None else min(best, ms)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    for name, fn, nbytes in (("host-to-device", h2d, n), ("device-to-host", d2h, n), ("both at once", both, 2 * n)):
        ms = timed(fn)
        print(f"hostlink {name}: {nbytes / (ms / 1e3) / 1e9:.1f} GB/s ({nbytes >> 20} MiB in {ms:.3f} ms, best of "
              f"{max(reps, 5)})")


CASES = {
    "prefill_4x16x4096": lambda r: _prefill(4, r),
    "prefill_1x16x4096": lambda r: _prefill(1, r),
    "variants_4x16x4096": _variants,
    "decode_256x32": lambda r: _decode(256, r),
    "decode_64x32": lambda r: _decode(64, r),
    "long_131k": _long,
    "long_131k_segmented": _long_segmented,
    "long_65k_segmented": lambda r: _long_segmented(r, T=65536),
    "varlen_64seq": lambda r: _varlen(W.varlen_64seq(), r),
    "varlen_64seq_1m": lambda r: _varlen(W.varlen_64seq_1m(), r),
    "hostlink": _hostlink,
    "backward_4x16x4096": lambda r: _backward(4, 4096, r),
    "backward_1x16x1024": lambda r: _backward(1, 1024, r),
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
