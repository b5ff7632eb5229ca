#!/usr/bin/env python
"""Benchmark of the KDA hot path on GB300.

One step = one chunkwise prefill over the batch B=4, H=16, T=4096,
d_k=d_v=128 (bf16 q/k/v, fp32 gates and state, S0 = 0): every token of every
head goes through the full path. Inputs are resident in HBM when the timed
region starts and are larger than L2 (0.34 GB of inputs, 0.4 GB moved per
step vs a 129 MB L2), so back-to-back steps read from HBM.

Prints ONE JSON line (rank 0). Keys beyond the basic contract:
  roofline      the prefill kernel against the measured HBM copy bandwidth
                (algorithmic bytes per launch / mean launch time)
  cpu_baseline  the float64 CPU oracle timed on a bounded sample
  e2e           the same metric through the public API with host buffers,
                host<->device copies inside the timed region
  decode        the decode step on 256 sequences x 32 heads (state GB/s)
  long_context  prefill of one 131,072-token sequence with 32 heads, cut
                into segments that run at once (kda_prefill_segmented), with
                the plain one-cluster-per-head launch beside it
  varlen        packed prefill of 64 lognormal-length sequences (306,055
                tokens, 16 heads), and varlen_1m: the same lengths scaled to
                2^20 tokens
  backward      gradients of the benchmark workload (kda_prefill_backward);
                more_workloads: the long-context sequence and the packed
                64-sequence batch
  gate_variants the benchmark workload with a scalar gate, no gate, FP8 inputs
  clocks        SM clocks and throttle reasons sampled during the timed region
                (and during about a second of the same steps just before it)

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torchrun (one process per GPU, independent batches:
weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (% bf16 TC peak); decode step state GB/s (% HBM peak)"
B, H, T, DK, DV, CHUNK = 4, 16, 4096, 128, 128, 64
DEC_N, DEC_H = 256, 32
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def prefill_bytes(B, T, H, dk, dv, qkv_bytes=2, with_s0=False, gate="channel"):
    """Algorithmic HBM bytes of one prefill call: q, k, v, alpha, beta read
    once, o written once, final state written once (and S0 read if given).
    alpha is d_k floats per token-head for the per-channel gate, one for the
    scalar gate, none without a gate."""
    alpha_bytes = {"channel": dk * 4, "scalar": 4, "none": 0}[gate]
    per_tok_head = 2 * dk * qkv_bytes + dv * qkv_bytes + alpha_bytes + 4 + dv * qkv_bytes
    state = B * H * dk * dv * 4
    return B * T * H * per_tok_head + state * (2 if with_s0 else 1)


def prefill_flops(B, T, H, dk, dv, C=CHUNK):
    """Algorithmic flops per token-head of the chunked form: the three
    d_k x d_v products (state read-outs X, Y and the state update), the
    triangular halves of the intra-chunk products, the substitution."""
    f = 6 * dk * dv + (C - 1) * (2 * dk + dv) + (C + 1) * (dk + dv) + C * C / 3
    return B * T * H * f


def decode_bytes(N, H, dk, dv, qkv_bytes=2):
    return N * H * (2 * dk * dv * 4 + 2 * dk * qkv_bytes + dv * qkv_bytes + dk * 4 + 4 + dv * qkv_bytes)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 200 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def rank_env():
    """(world, rank, local_rank) from the launcher's environment; (1, 0, 0)
    when run alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_seed(rank: int) -> int:
    """Seed of a rank's batch. Every rank draws its own independent batch of
    (sequence, head) work: weak scaling, nothing is exchanged."""
    return rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (the job's time). The only collective of the
    benchmark besides its barriers; `device` is the tensor's device for the
    process group's backend (cuda for nccl, cpu for gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, seconds: float) -> float:
    """Whole-job throughput: the tokens of all ranks over the slowest rank's time."""
    return world * tokens_per_rank / seconds


def kernel_traffic(kernel_file: str, key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(key)
    if not ent:
        return None
    src = os.path.join(ROOT, "kda_gated_delta_chunkwise_gb300", "csrc", kernel_file)
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return ent.get("bytes_per_launch") if ent.get("source_sha") == sha else None


def cpu_baseline_oracle(target_s: float = 12.0):
    """Time the float64 oracle on a bounded sample of the prefill workload: all
    B*H = 64 (sequence, head) pairs over the first Ts tokens, with Ts chosen so
    the timed run takes about target_s seconds on the host cores."""
    import oracle
    from kda_gated_delta_chunkwise_gb300 import workloads as W

    x = W.prefill_4x16x4096(T=4096)
    cores = oracle.max_threads()
    lib = oracle.load()

    def run(Ts):
        args = [t[:, :Ts] for t in x.tensors()]
        t0 = time.perf_counter()
        oracle.run(*args, lib=lib)
        return time.perf_counter() - t0

    Ts = 64
    dt = run(Ts)
    Ts = int(min(T, max(64, Ts * target_s / max(dt, 1e-3))))
    reps, total = 0, 0.0
    while reps == 0 or total < 0.5 * target_s:  # the whole workload is shorter: repeat it
        total += run(Ts)
        reps += 1
    dt = total / reps
    return {"value": B * Ts / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"B={B} x H={H} (all 64 sequence-head pairs) x first {Ts} of {T} tokens, "
                      f"d={DK}, float64, {reps} run(s), {total:.1f} s in all"}


def time_events(fn, steps: int, warmup: int, stream) -> float:
    """Mean CUDA-event time (ms) of ``fn`` over ``steps`` launches after
    ``warmup`` untimed ones, events recorded on ``stream`` (the launching
    stream)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s_, e_ in ev:
        s_.record(stream)
        fn()
        e_.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(s_.elapsed_time(e_) for s_, e_ in ev)


def oracle_tokens_per_s(x, n_tokens_of, sample: str, target_s: float = 4.0, lib=None):
    """The float64 oracle on a bounded sample of a workload: ``n_tokens_of(Ts)``
    gives the oracle inputs (and token count) for the first Ts tokens of every
    sequence; Ts is chosen so the run takes about ``target_s`` seconds."""
    import oracle
    lib = lib or oracle.load()

    def run(Ts):
        args, kw, ntok = n_tokens_of(Ts)
        t0 = time.perf_counter()
        oracle.run(*args, **kw, lib=lib)
        return time.perf_counter() - t0, ntok

    Ts = 64
    dt, _ = run(Ts)
    Ts = max(64, int(Ts * target_s / max(dt, 1e-3)) // 64 * 64)
    dt, ntok = run(Ts)
    return {"value": ntok / dt, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": sample.format(Ts=Ts) + f", float64, {dt:.1f} s"}


def bench_long_context(kda, W, dev, stream, peaks, steps, warmup, with_cpu):
    """One 131,072-token sequence with 32 heads (split decay scales, S0 given):
    the case where a sequence is far longer than the batch is wide, so the
    per-chunk state chain of each head sets the time. Timed through
    kda_prefill_segmented (segments of the sequence run at once, joined by
    their transition products) with the plain launch beside it."""
    x = W.prefill_long_131k()
    q, k, v, a, b, s0 = (t.to(dev) for t in (*x.tensors(), x.initial_state))
    Bl, Tl, Hl = 1, x.q.shape[1], x.q.shape[2]
    o = torch_empty_like(v)
    sT = torch_empty_like(s0)
    nbytes = prefill_bytes(Bl, Tl, Hl, DK, DV, with_s0=True)
    # the sequence cut into segments that run at once (kda_prefill_segmented,
    # the library's plan), and the plain one-cluster-per-head launch beside it
    G, first, seg = kda.segment_plan(Tl, Hl)
    ws = torch_empty_bytes(kda.prefill_segmented_workspace_bytes(Tl, Hl), dev)
    ms = time_events(lambda: kda.prefill_segmented(q, k, v, a, b, s0, out=o, final_state=sT, workspace=ws),
                     steps, warmup, stream)
    ms_plain = time_events(lambda: kda.prefill(q, k, v, a, b, s0, out=o, final_state=sT), steps, warmup, stream)
    gbs = nbytes / (ms / 1e3) / 1e9
    gbs_plain = nbytes / (ms_plain / 1e3) / 1e9
    res = {"workload": f"kda_prefill_segmented B=1 H={Hl} T={Tl} d_k={DK} d_v={DV} chunk={CHUNK}, bf16 q/k/v, "
                       "alpha scales 1e-4 / 0.2 per half of the key channels, S0 ~ N(0, 0.01^2)",
           "value": Bl * Tl / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
           "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
           "kernels": "kda_prefill_tc (segment 0 from S0 on a high-priority stream; later segments from zero "
                      "and, with v = 0, from the identity on a second stream), seg_combine, seg_correct",
           "segments": {"n": G, "first_tokens": first, "tokens_each_later": seg},
           "workspace_bytes": ws.numel(),
           "plain": {"kernel": "kda_prefill_tc, one cluster per head", "clusters": Bl * Hl,
                     "value": Bl * Tl / (ms_plain / 1e3), "ms_per_step": ms_plain, "achieved_gbs": gbs_plain,
                     "frac": gbs_plain / peaks["hbm_gbs"]}}
    del q, k, v, a, b, o, sT, ws
    if with_cpu:
        res["cpu_baseline"] = oracle_tokens_per_s(
            x, lambda Ts: ([t[:, :Ts] for t in x.tensors()], {"initial_state": x.initial_state}, Ts),
            "all 32 heads x first {Ts} of 131072 tokens")
    return res


def bench_varlen(kda, W, x, dev, stream, peaks, steps, warmup, with_cpu, label):
    """Packed prefill (kda_varlen_prefill) of the lognormal 64-sequence batch."""
    (q, k, v, a, b), cu, s0 = [t.to(dev) for t in x.tensors()], x.cu_seqlens.to(dev), x.initial_state.to(dev)
    N, Tt, Hv = x.num_seqs, x.q.shape[0], x.q.shape[1]
    o = torch_empty_like(v)
    sT = torch_empty_like(s0)
    ws = torch_empty_bytes(kda.varlen_workspace_bytes(N, Hv), dev)
    ms = time_events(lambda: kda.varlen_prefill(q, k, v, a, b, cu, s0, out=o, final_state=sT, workspace=ws),
                     steps, warmup, stream)
    # every token-head's inputs and o, plus each sequence's S0 read and final state written
    nbytes = prefill_bytes(1, Tt, Hv, DK, DV) - Hv * DK * DV * 4 + 2 * N * Hv * DK * DV * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    L = (x.cu_seqlens[1:] - x.cu_seqlens[:-1]).tolist()
    res = {"workload": f"kda_varlen_prefill N={N} T_total={Tt} H={Hv} d_k={DK} d_v={DV}, {label}, "
                       f"lengths {min(L)}..{max(L)}, bf16 q/k/v, per-sequence S0 ~ N(0, 0.01^2)",
           "value": Tt / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
           "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
           "kernel": "kda_prefill_tc (+ kda_varlen_prep)", "clusters": N * Hv}
    del q, k, v, a, b, o, sT, cu, s0, ws
    if with_cpu:
        cuh = x.cu_seqlens.tolist()

        def first(Ts):
            # the first Ts tokens of every sequence, packed
            idx = [(cuh[n], min(cuh[n + 1], cuh[n] + Ts)) for n in range(N)]
            cut = [0]
            for lo, hi in idx:
                cut.append(cut[-1] + hi - lo)
            import torch
            args = [torch.cat([t[lo:hi] for lo, hi in idx]) for t in x.tensors()]
            return args, {"cu_seqlens": cut, "initial_state": x.initial_state}, cut[-1]
        res["cpu_baseline"] = oracle_tokens_per_s(x, first, "all 64 sequences x 16 heads, first {Ts} tokens of each")
    return res


def backward_bytes(B, T, H, dk, dv, qkv_bytes=2):
    """Algorithmic HBM bytes of one backward call: q, k, v, alpha, beta and
    d_o read once, the fp32 gradients dq, dk, dalpha, dv, dbeta written once,
    and the initial state's gradient written once."""
    per_tok_head = (2 * dk + 2 * dv) * qkv_bytes + dk * 4 + 4 + (3 * dk + dv) * 4 + 4
    return B * T * H * per_tok_head + B * H * dk * dv * 4


def bench_backward(kda, W, dev, stream, peaks, steps, warmup):
    """Gradients of the 4x16x4096 prefill (kda_prefill_backward) for a random d_o."""
    import torch
    x = W.prefill_4x16x4096()
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    d_o = torch.randn(v.shape, generator=torch.Generator(device=dev).manual_seed(7), device=dev).to(v.dtype)
    Bb, Tb, Hb = q.shape[0], q.shape[1], q.shape[2]
    ws = torch_empty_bytes(kda.load().kda_prefill_backward_workspace_bytes(Bb, Tb, Hb, DK, DV), dev)
    ms = time_events(lambda: kda.prefill_backward(q, k, v, a, b, d_o, workspace=ws), steps, warmup, stream)
    nbytes = backward_bytes(Bb, Tb, Hb, DK, DV)
    gbs = nbytes / (ms / 1e3) / 1e9
    res = {"workload": f"kda_prefill_backward B={Bb} H={Hb} T={Tb} d_k={DK} d_v={DV}, bf16 q/k/v/d_o, fp32 gradients",
           "value": Bb * Tb / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
           "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
           "kernels": "kda_bwd_tables + kda_bwd_states + kda_bwd_chain + kda_bwd_local (fp32 arithmetic; "
                      "products on the tensor cores as single tf32 products for bf16 inputs)",
           "workspace_bytes": ws.numel()}
    del q, k, v, a, b, d_o, ws
    return res


def bench_backward_more(kda, W, dev, stream, peaks, steps, warmup):
    """The backward on the long-context workload (1x32x131072, S0 given) and
    on the packed 64-sequence batch (306,055 tokens x 16 heads, S0 given), a
    random d_o each: one call per step, CUDA events."""
    import torch
    res = {}
    for key, x, packed in (("long_context", W.prefill_long_131k(), False),
                           ("varlen", W.varlen_64seq(), True)):
        q, k, v, a, b = (t.to(dev) for t in x.tensors())
        s0 = x.initial_state.to(dev)
        d_o = torch.randn(v.shape, generator=torch.Generator(device=dev).manual_seed(7), device=dev).to(v.dtype)
        if packed:
            cu = x.cu_seqlens.to(dev)
            N, Tt, H = cu.numel() - 1, q.shape[0], q.shape[1]
            ws = torch_empty_bytes(kda.load().kda_varlen_prefill_backward_workspace_bytes(N, Tt, H, DK, DV), dev)
            fn = lambda: kda.varlen_prefill_backward(q, k, v, a, b, d_o, cu, s0, workspace=ws)
            tokens, n_states = Tt, N * H
            desc = f"kda_varlen_prefill_backward N={N} sequences, T_total={Tt}, H={H}, d_k={DK} d_v={DV}"
        else:
            Bb, Tb, H = q.shape[0], q.shape[1], q.shape[2]
            ws = torch_empty_bytes(kda.load().kda_prefill_backward_workspace_bytes(Bb, Tb, H, DK, DV), dev)
            fn = lambda: kda.prefill_backward(q, k, v, a, b, d_o, s0, workspace=ws)
            tokens, n_states = Bb * Tb, Bb * H
            desc = f"kda_prefill_backward B={Bb} H={H} T={Tb} d_k={DK} d_v={DV}"
        ms = time_events(fn, max(3, steps // 4), warmup, stream)
        # backward_bytes counts one sequence-head state (dS0 written); S0 is read too
        nbytes = backward_bytes(1, tokens, H, DK, DV) + (n_states - H) * DK * DV * 4 + n_states * DK * DV * 4
        gbs = nbytes / (ms / 1e3) / 1e9
        res[key] = {"workload": desc + ", bf16 q/k/v/d_o, S0 given, fp32 gradients",
                    "value": tokens / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "steps": max(3, steps // 4),
                    "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"],
                    "workspace_bytes": ws.numel()}
        del q, k, v, a, b, s0, d_o, ws
        torch.cuda.empty_cache()
    return res


def torch_empty_like(t):
    import torch
    return torch.empty_like(t)


def torch_empty_bytes(n, dev):
    import torch
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=dev)


def bench_config(world: int) -> dict:
    """The workload description both arms report."""
    return {"workload": f"kda_prefill B={B} H={H} T={T} d_k={DK} d_v={DV} chunk={CHUNK}",
            "inputs": "bf16 q/k/v (q, k L2-normalised), fp32 alpha/beta, fp32 state, S0 = 0",
            "l2": "inputs larger than L2 (0.34 GB in, 0.41 GB moved per step; L2 129 MB)",
            "parallelism": f"{world} independent replica(s)"}


def run_reference(args):
    """The reference arm: the float64 oracle on the host cores (rank 0 only)."""
    _, rank, _ = rank_env()
    if rank != 0:
        return
    import oracle
    from kda_gated_delta_chunkwise_gb300 import workloads as W

    x = W.prefill_4x16x4096(T=4096)
    lib = oracle.load()
    cores = oracle.max_threads()
    # tokens per step: the whole sequence length when a step of it takes at
    # most about 2 s on these cores (so K + W steps end within minutes),
    # else the first Ts tokens of every sequence
    t0 = time.perf_counter()
    oracle.run(*[t[:, :256] for t in x.tensors()], lib=lib)
    per_tok = (time.perf_counter() - t0) / 256
    Ts = int(min(T, max(64, 2.0 / max(per_tok, 1e-9) // 64 * 64)))
    sl = [t[:, :Ts] for t in x.tensors()]
    for _ in range(args.warmup):
        oracle.run(*sl, lib=lib)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run(*sl, lib=lib)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    val = B * Ts / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(bench_config(args.gpus),
                           sample=f"each step: all 64 sequence-head pairs, first {Ts} of {T} tokens"),
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"B={B} x H={H} x first {Ts} tokens per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algo", choices=["auto", "simt", "tc"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the long-context and packed-batch legs")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    import kda_gated_delta_chunkwise_gb300 as kda
    from kda_gated_delta_chunkwise_gb300 import workloads as W

    world, rank, local = rank_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    kda.load()
    peaks, peak_src = load_peaks()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- inputs (seeded; each rank its own batch) ----
    x = W.prefill_4x16x4096(seed=shard_seed(rank))
    q, k, v, a, b = (t.to(dev) for t in x.tensors())
    o = torch.empty_like(v)
    sT = torch.empty((B, H, DK, DV), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        kda.prefill(q, k, v, a, b, None, out=o, final_state=sT, algo=args.algo)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    # about a second of the same steps (untimed) right before the timed
    # region, so that the clock samples (every 200 ms) cover this load
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.0:
        for _ in range(50):
            step()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    if clk:
        clk["window"] = "about 1 s of the same steps, untimed, then the timed region"
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = statistics.mean(s.elapsed_time(e) for s, e in ev)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_tokens_per_s(world, B * T, ms_per_step / 1e3)

    algo_bytes = prefill_bytes(B, T, H, DK, DV)
    algo_flops = prefill_flops(B, T, H, DK, DV)
    achieved = algo_bytes / (launch_ms / 1e3) / 1e9
    tflops = algo_flops / (launch_ms / 1e3) / 1e12
    used_tc = args.algo == "tc" or (args.algo == "auto" and kda_uses_tc(kda, dev))
    kfile = "kda_prefill_tc.cu" if used_tc else "kda_prefill_simt.cu"
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": kernel_traffic(kfile, "prefill_tc" if used_tc else "prefill_simt"),
                "peak_source": f"{peak_src} STREAM-style copy (hbm_gbs)",
                "algorithmic_bytes_per_launch": algo_bytes,
                "kernel": "kda_prefill_tc" if used_tc else "kda_prefill_simt",
                "tflops_algorithmic": tflops,
                "tensor_frac": tflops / peaks["bf16_tflops"]}

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, ha, hb = (t.pin_memory() for t in x.tensors())
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ha, hb))
        d2h = o.numel() * o.element_size() + sT.numel() * 4
        # warm-up in the timed loop's pattern (the previous step's host outputs
        # alive while the next step allocates), so the page-locked output
        # buffers are cached before timing
        oh = sh = None
        for _ in range(3):
            oh, sh = kda.prefill(hq, hk, hv, ha, hb, None, algo=args.algo)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 10))
        barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            oh, sh = kda.prefill(hq, hk, hv, ha, hb, None, algo=args.algo)  # returns host tensors
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / n_e2e
        dt = max_over_ranks(dt, world, dev)
        e2e = {"value": job_tokens_per_s(world, B * T, dt), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
               "path": "kda_prefill_host: page-locked host tensors, copied in pieces along T (about 32 MiB "
                       "of input each) with copy-in, kernels and copy-out overlapped on three streams"}

    # ---- the same workload with a scalar gate (Gated DeltaNet) and without a
    #      gate (the delta rule): fewer gate bytes, same kernels ----
    variants = None
    if not args.no_variants:
        variants = {}
        for name, gate in (("gated_deltanet", "scalar"), ("deltanet", "none")):
            av = a[..., 0].contiguous() if gate == "scalar" else None
            for _ in range(args.warmup):
                kda.prefill(q, k, v, av, b, None, out=o, final_state=sT, algo=args.algo, gate=gate)
            torch.cuda.synchronize()
            evv = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for i in range(args.steps):
                evv[i][0].record(stream)
                kda.prefill(q, k, v, av, b, None, out=o, final_state=sT, algo=args.algo, gate=gate)
                evv[i][1].record(stream)
            torch.cuda.synchronize()
            vms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in evv)
            vbytes = prefill_bytes(B, T, H, DK, DV, gate=gate)
            variants[name] = {"gate": gate, "value": B * T / (vms / 1e3), "unit": "tokens/s",
                              "ms_per_step": vms, "algorithmic_bytes_per_launch": vbytes,
                              "achieved_gbs": vbytes / (vms / 1e3) / 1e9,
                              "frac": vbytes / (vms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        # FP8 inputs (MX block format: E4M3 codes, one scale byte per 32 channels)
        cq, sq, _ = W.to_mxfp8(q)
        ck, sk, _ = W.to_mxfp8(k)
        cv, sv, _ = W.to_mxfp8(v)
        for _ in range(args.warmup):
            kda.prefill_fp8(cq, ck, cv, sq, sk, sv, a, b, None, out=o, final_state=sT)
        torch.cuda.synchronize()
        evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            evf[i][0].record(stream)
            kda.prefill_fp8(cq, ck, cv, sq, sk, sv, a, b, None, out=o, final_state=sT)
            evf[i][1].record(stream)
        torch.cuda.synchronize()
        fms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in evf)
        # q, k, v: one byte per element instead of two, plus a scale byte per 32
        fbytes = prefill_bytes(B, T, H, DK, DV) - B * T * H * (2 * DK + DV) + B * T * H * (2 * DK + DV) // 32
        variants["fp8_inputs"] = {"inputs": "E4M3 q, k, v with E8M0 scales per 32 channels; bf16 o",
                                  "value": B * T / (fms / 1e3), "unit": "tokens/s", "ms_per_step": fms,
                                  "algorithmic_bytes_per_launch": fbytes,
                                  "achieved_gbs": fbytes / (fms / 1e3) / 1e9,
                                  "frac": fbytes / (fms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        if not args.no_e2e:
            # end to end from page-locked host memory (kda_prefill_fp8_host):
            # the host link carries one byte per q, k, v element
            fh = [t.cpu().pin_memory() for t in (cq, ck, cv, sq, sk, sv)]
            ah, bh = a.cpu().pin_memory(), b.cpu().pin_memory()
            oh = sh = None
            for _ in range(3):
                oh, sh = kda.prefill_fp8(*fh, ah, bh, None)
            torch.cuda.synchronize()
            n_e2e = max(3, min(args.steps, 10))
            t0 = time.perf_counter()
            for _ in range(n_e2e):
                oh, sh = kda.prefill_fp8(*fh, ah, bh, None)
            torch.cuda.synchronize()
            fdt = (time.perf_counter() - t0) / n_e2e
            variants["fp8_inputs"]["e2e"] = {
                "value": B * T / fdt, "unit": "tokens/s", "ms_per_step": fdt * 1e3,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in fh + [ah, bh]),
                "d2h_bytes_per_step": oh.numel() * oh.element_size() + sh.numel() * 4}
            del fh, ah, bh, oh, sh
        del cq, ck, cv, sq, sk, sv

    # ---- decode step (secondary figure of the metric) ----
    decode = None
    if not args.no_decode:
        del q, k, v, a, b, o, sT
        xd = W.decode_256x32(seed=shard_seed(rank))
        dq, dk_, dv_, da, db = (t.to(dev) for t in xd.tensors())
        # two state batches used in turn (1 GiB together, 8x the L2): a step
        # never finds its state, or the previous step's dirty lines of it, in L2
        states = [xd.initial_state.to(dev), xd.initial_state.to(dev)]
        do = torch.empty_like(dv_)
        it = [0]

        def dstep():
            kda.decode_step(dq, dk_, dv_, da, db, states[it[0] & 1], out=do)
            it[0] += 1
        for _ in range(args.warmup):
            dstep()
        torch.cuda.synchronize()
        evd = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            evd[i][0].record(stream)
            dstep()
            evd[i][1].record(stream)
        torch.cuda.synchronize()
        dms = statistics.median(s.elapsed_time(e) for s, e in evd)
        dbytes = decode_bytes(DEC_N, DEC_H, DK, DV)
        gbs = dbytes / (dms / 1e3) / 1e9
        dtraffic = kernel_traffic("kda_decode.cu", "decode")
        decode = {"metric": "decode step state GB/s", "value": gbs, "unit": "GB/s",
                  "ms_per_step": dms, "frac": gbs / peaks["hbm_gbs"], "peak": peaks["hbm_gbs"],
                  "algorithmic_bytes_per_step": dbytes,
                  "traffic": dtraffic,
                  "dram_gbs_from_traffic": None if dtraffic is None else dtraffic / (dms / 1e3) / 1e9,
                  "note": "the peak is a plain copy; this kernel streams half the bytes of that copy "
                          "per launch and can sit a hair above it",
                  "workload": f"{DEC_N} sequences x {DEC_H} heads, d={DK}, bf16 q/k/v, fp32 state in place, "
                              "two state batches in turn"}
        del states, dq, dk_, dv_, da, db, do

    backward = None
    if not args.no_backward:
        torch.cuda.empty_cache()
        backward = bench_backward(kda, W, dev, stream, peaks, args.steps, args.warmup)
        if not args.no_long:
            torch.cuda.empty_cache()
            backward["more_workloads"] = bench_backward_more(kda, W, dev, stream, peaks, args.steps, args.warmup)
    long_ctx = varlen = varlen_1m = None
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if not args.no_long:
        torch.cuda.empty_cache()
        long_ctx = bench_long_context(kda, W, dev, stream, peaks, args.steps, args.warmup, with_cpu)
        torch.cuda.empty_cache()
        varlen = bench_varlen(kda, W, W.varlen_64seq(seed=shard_seed(rank)), dev, stream, peaks, args.steps,
                              args.warmup, with_cpu, "lengths round(lognormal(8, 1)) clipped to [512, 32768]")
        torch.cuda.empty_cache()
        varlen_1m = bench_varlen(kda, W, W.varlen_64seq_1m(seed=shard_seed(rank)), dev, stream, peaks,
                                 max(3, args.steps // 2), args.warmup, with_cpu,
                                 "the same lengths scaled to 2^20 tokens and re-clipped")
        torch.cuda.empty_cache()

    cpu = None
    if with_cpu:
        cpu = cpu_baseline_oracle()

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": bench_config(world),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "decode": decode,
                "long_context": long_ctx, "varlen": varlen, "varlen_1m": varlen_1m, "backward": backward,
                "gate_variants": variants,
                "gpu_launches": args.steps, "clocks": clk}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def kda_uses_tc(kda, dev) -> bool:
    """Whether the automatic choice takes the tensor-core kernel for this
    workload: the library answers an explicit tensor-core request on an empty
    batch with KDA_OK exactly when that kernel supports the shape and dtype."""
    import ctypes
    lib = kda.load()
    p = ctypes.c_void_p(256)
    return lib.kda_prefill_ex(p, p, p, 1, p, p, None, p, None, 0, T, H, DK, DV, 2, None) == 0


if __name__ == "__main__":
    main()
