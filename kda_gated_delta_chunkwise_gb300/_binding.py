"""ctypes binding of the KDA C ABI (include/kda.h).

Argument marshalling only: shape and dtype checks, output allocation through
PyTorch, the raw pointers and the current CUDA stream. Every step of the
method runs in the library's CUDA kernels. There is no fallback: if the
shared library is missing or fails to load, every call raises.

Inputs on the host (CPU tensors) are accepted for end-to-end use: they are
copied to the current CUDA device, the call runs there, and the outputs are
copied back to the host.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_DEVICE_CHECK, KDA_ERR_WORKSPACE = range(6)
KDA_F32, KDA_BF16 = 0, 1
ALGOS = {"auto": 0, "simt": 1, "tc": 2}
# gate kinds: per-channel (KDA), one per token-head (Gated DeltaNet), none (delta rule)
GATES = {"channel": 0, "scalar": 1, "none": 2}
KDA_DEV_OK, KDA_DEV_BAD_CU_SEQLENS, KDA_DEV_BAD_SLOT = 0, 1, 2

EXPORTS = ("kda_prefill", "kda_prefill_ex", "kda_prefill_gate", "kda_prefill_fp8", "kda_prefill_host",
           "kda_prefill_host_workspace_bytes", "kda_prefill_fp8_host", "kda_prefill_fp8_host_workspace_bytes",
           "kda_varlen_prefill", "kda_varlen_prefill_slots",
           "kda_varlen_prefill_noalloc", "kda_varlen_workspace_bytes", "kda_prefill_workspace_bytes",
           "kda_prefill_segmented", "kda_prefill_segmented_workspace_bytes", "kda_prefill_segment_plan",
           "kda_decode_step", "kda_decode_step_slots", "kda_selftest_bounded_wait",
           "kda_prefill_backward", "kda_prefill_backward_gate", "kda_prefill_backward_workspace_bytes",
           "kda_varlen_prefill_backward", "kda_varlen_prefill_backward_workspace_bytes",
           "kda_device_errors", "kda_last_error", "kda_abi_version")

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"KDA error {status}: {message}")
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the shared library (it must have been built: ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or lib_path()
        if not os.path.exists(p):
            raise RuntimeError(f"KDA CUDA library not built ({p}); run the package build first")
        lib = ctypes.CDLL(p)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        lib.kda_prefill_ex.restype = ctypes.c_int
        lib.kda_prefill_ex.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.kda_prefill.restype = ctypes.c_int
        lib.kda_prefill.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
        lib.kda_varlen_prefill.restype = ctypes.c_int
        lib.kda_varlen_prefill.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                           vp, ctypes.c_size_t, vp, vp]
        lib.kda_varlen_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_varlen_workspace_bytes.argtypes = [i, i, i, i]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, i, i, i, i, vp]
        lib.kda_prefill_gate.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.kda_prefill_gate.restype = i
        lib.kda_prefill_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, vp, vp, vp, vp, i, i, i, i, i, vp]
        lib.kda_prefill_fp8.restype = i
        lib.kda_prefill_host.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, vp, i, i, i, i, i, i, i, vp,
                                         ctypes.c_size_t, vp]
        lib.kda_prefill_host.restype = i
        lib.kda_prefill_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.kda_prefill_host_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_prefill_fp8_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, vp, vp, vp, vp, i, i, i, i, i, i, vp,
                                             ctypes.c_size_t, vp]
        lib.kda_prefill_fp8_host.restype = i
        lib.kda_prefill_fp8_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.kda_prefill_fp8_host_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_varlen_prefill_slots.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, i, vp, vp, i, i, i, i, i,
                                                 vp, ctypes.c_size_t, vp, vp]
        lib.kda_varlen_prefill_slots.restype = i
        lib.kda_decode_step_slots.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, i, vp, i, i, i, i, vp, vp]
        lib.kda_decode_step_slots.restype = i
        lib.kda_prefill_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_prefill_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.kda_selftest_bounded_wait.restype = i
        lib.kda_selftest_bounded_wait.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, vp]
        lib.kda_prefill_backward.restype = i
        lib.kda_prefill_backward.argtypes = [vp, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             i, i, i, i, i, vp, ctypes.c_size_t, vp]
        lib.kda_prefill_backward_gate.restype = i
        lib.kda_prefill_backward_gate.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                  i, i, i, i, i, vp, ctypes.c_size_t, vp]
        lib.kda_varlen_prefill_backward.restype = i
        lib.kda_varlen_prefill_backward.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                    vp, i, i, i, i, i, vp, ctypes.c_size_t, vp, vp]
        lib.kda_varlen_prefill_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_varlen_prefill_backward_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.kda_prefill_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_prefill_backward_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.kda_prefill_segmented.restype = i
        lib.kda_prefill_segmented.argtypes = [vp, vp, vp, i, vp, i, vp, vp, vp, vp, i, i, i, i, i, i, vp,
                                              ctypes.c_size_t, vp]
        lib.kda_prefill_segmented_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_prefill_segmented_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.kda_prefill_segment_plan.restype = i
        lib.kda_prefill_segment_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int),
                                                 ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_abi_version.restype = ctypes.c_int
        lib.kda_abi_version.argtypes = []
        lib.kda_device_errors.restype = ctypes.c_int
        lib.kda_device_errors.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.c_int]
        del f
        if path is None:
            _lib = lib
        return lib


def device_errors(reset: bool = True) -> int:
    """The device-side error word (nonzero: a kernel's bounded wait ran out)."""
    lib = load()
    v = ctypes.c_int(0)
    _check(lib, lib.kda_device_errors(ctypes.byref(v), int(reset)))
    return v.value


def selftest_bounded_wait(q, k, v, alpha, beta, stall_chunk: int, *, stream=None):
    """Diagnostic: the tensor-core prefill of one bf16 sequence of one head
    (q, k, v [T, 128], alpha [T, 128], beta [T]) with its state chain stalled
    at chunk ``stall_chunk`` on a wait that never completes. The kernel gives
    up after about a second and returns; read the outcome with
    :func:`device_errors`. Returns the (invalid) o and final state."""
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, dev)
    _need(alpha, "alpha", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    T = q.shape[0]
    if q.shape != (T, 128) or k.shape != q.shape or v.shape != q.shape or alpha.shape != q.shape \
            or beta.shape != (T,):
        raise ValueError("q, k, v, alpha must be [T, 128] and beta [T]")
    o = torch.empty_like(v)
    s = torch.empty((128, 128), dtype=torch.float32, device=dev)
    _check(lib, lib.kda_selftest_bounded_wait(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(o), _ptr(s),
                                              T, int(stall_chunk), _stream(stream)))
    return o, s


def prefill_workspace_bytes(B: int, T: int, H: int, dk: int = 128, dv: int = 128) -> int:
    """Device scratch the equal-length prefill needs: always 0."""
    return int(load().kda_prefill_workspace_bytes(B, T, H, dk, dv))


def _check(lib, status: int):
    if status != KDA_OK:
        raise KdaError(status, lib.kda_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _need(t, name, dtype=None, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _to_host(x: torch.Tensor) -> torch.Tensor:
    """Device -> pinned host copy, queued on the current stream (pinned buffers
    come from torch's caching host allocator, so repeated calls reuse them)."""
    h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    h.copy_(x, non_blocking=True)
    return h


def _host_prefill(q, k, v, alpha, beta, initial_state, *, output_final_state, algo, gate, piece_tokens):
    """``prefill`` on host tensors through kda_prefill_host: the library moves
    the tokens to the device in pieces along T and the outputs back, overlapped
    with the kernels, on the current CUDA stream. Outputs land in page-locked
    host tensors and are complete when this returns."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    cpu = torch.device("cpu")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, cpu)
    _need(beta, "beta", torch.float32, cpu)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (B, T, H, dv) or beta.shape != (B, T, H):
        raise ValueError("shape mismatch among q, k, v, beta")
    alpha = _check_gate(gate, alpha, (B, T, H), dk, cpu)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, cpu)
        if initial_state.shape != (B, H, dk, dv):
            raise ValueError(f"initial_state must be {(B, H, dk, dv)}")
    if algo not in ALGOS:
        raise ValueError(f"algo must be one of {sorted(ALGOS)}")
    o_h = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    s_h = torch.empty((B, H, dk, dv), dtype=torch.float32, pin_memory=True) if output_final_state else None
    nbytes = lib.kda_prefill_host_workspace_bytes(B, T, H, dk, dv, _dtype_code(q), GATES[gate], piece_tokens)
    ws = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = lib.kda_prefill_host(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate], _ptr(beta),
                              _ptr(initial_state), _ptr(o_h), _ptr(s_h), B, T, H, dk, dv, ALGOS[algo],
                              int(piece_tokens), _ptr(ws), ws.numel(), _stream(stream))
    _check(lib, st)
    stream.synchronize()
    return o_h, s_h


def _host_prefill_fp8(q, k, v, q_scale, k_scale, v_scale, alpha, beta, initial_state, *, output_final_state,
                      gate, piece_tokens):
    """``prefill_fp8`` on host tensors through kda_prefill_fp8_host."""
    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device())
    cpu = torch.device("cpu")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.uint8, cpu)
    _need(beta, "beta", torch.float32, cpu)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (B, T, H, dv) or beta.shape != (B, T, H) \
            or q_scale.shape != (B, T, H, dk // 32) or k_scale.shape != (B, T, H, dk // 32) \
            or v_scale.shape != (B, T, H, dv // 32):
        raise ValueError("shape mismatch among q, k, v, the scales and beta")
    alpha = _check_gate(gate, alpha, (B, T, H), dk, cpu)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, cpu)
        if initial_state.shape != (B, H, dk, dv):
            raise ValueError(f"initial_state must be {(B, H, dk, dv)}")
    o_h = torch.empty((B, T, H, dv), dtype=torch.bfloat16, pin_memory=True)
    s_h = torch.empty((B, H, dk, dv), dtype=torch.float32, pin_memory=True) if output_final_state else None
    nbytes = lib.kda_prefill_fp8_host_workspace_bytes(B, T, H, dk, dv, GATES[gate], piece_tokens)
    ws = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = lib.kda_prefill_fp8_host(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                  _ptr(alpha), GATES[gate], _ptr(beta), _ptr(initial_state), _ptr(o_h), _ptr(s_h),
                                  B, T, H, dk, dv, int(piece_tokens), _ptr(ws), ws.numel(), _stream(stream))
    _check(lib, st)
    stream.synchronize()
    return o_h, s_h


def _host_call(fn, tensors: dict, **kw):
    """Run ``fn`` on the CUDA device for host inputs; return host outputs.
    Inputs in pinned memory are copied asynchronously; outputs land in pinned
    host memory and are complete when this returns."""
    dev = torch.device("cuda", torch.cuda.current_device())
    moved = {k: (None if v is None else v.to(dev, non_blocking=True)) for k, v in tensors.items()}
    out = fn(**moved, **kw)
    if isinstance(out, tuple):
        res = tuple(None if x is None else _to_host(x) for x in out)
    else:
        res = _to_host(out)
    torch.cuda.current_stream(dev).synchronize()
    return res


def _check_gate(gate: str, alpha, lead: tuple, dk: int, dev):
    """alpha for a gate kind: [*lead, d_k] (channel), [*lead] (scalar), unused (none)."""
    if gate not in GATES:
        raise ValueError(f"gate must be one of {sorted(GATES)}")
    if gate == "none":
        return None
    _need(alpha, "alpha", torch.float32, dev)
    want = tuple(lead) + ((dk,) if gate == "channel" else ())
    if tuple(alpha.shape) != want:
        raise ValueError(f"alpha must be {want} for gate={gate!r}, got {tuple(alpha.shape)}")
    return alpha


def prefill(q, k, v, alpha, beta, initial_state=None, *, output_final_state: bool = True,
            algo: str = "auto", gate: str = "channel", out=None, final_state=None, stream=None,
            piece_tokens: int = 0):
    """Chunkwise KDA prefill of B equal-length sequences.

    q, k: [B, T, H, d_k]; v: [B, T, H, d_v] (bf16 or fp32, same dtype);
    alpha: [B, T, H, d_k] fp32 (gate="channel"), [B, T, H] (gate="scalar",
    Gated DeltaNet) or None (gate="none", the delta rule); beta: [B, T, H] fp32;
    initial_state: [B, H, d_k, d_v] fp32 or None (zeros).
    Returns (o [B, T, H, d_v] in v's dtype, final_state [B, H, d_k, d_v] fp32 or None).

    Host (CPU) tensors go through kda_prefill_host: pieces of ``piece_tokens``
    tokens (0: the library's choice) travel to the GPU and back overlapped with
    the kernels; the outputs are page-locked host tensors. Page-locked inputs
    (``tensor.pin_memory()``) let the copies overlap.
    """
    if q.device.type == "cpu":
        if out is not None or final_state is not None or stream is not None:
            raise ValueError("out, final_state and stream apply to device tensors only")
        return _host_prefill(q, k, v, alpha, beta, initial_state, output_final_state=output_final_state,
                             algo=algo, gate=gate, piece_tokens=piece_tokens)
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(beta, "beta", torch.float32, dev)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (B, T, H, dv) or beta.shape != (B, T, H):
        raise ValueError("shape mismatch among q, k, v, beta")
    alpha = _check_gate(gate, alpha, (B, T, H), dk, dev)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev)
        if initial_state.shape != (B, H, dk, dv):
            raise ValueError(f"initial_state must be {(B, H, dk, dv)}")
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    if algo not in ALGOS:
        raise ValueError(f"algo must be one of {sorted(ALGOS)}")
    st = lib.kda_prefill_gate(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate], _ptr(beta),
                              _ptr(initial_state), _ptr(out), _ptr(final_state), B, T, H, dk, dv,
                              ALGOS[algo], _stream(stream))
    _check(lib, st)
    return out, final_state


def segment_plan(T: int, H: int, dk: int = 128, dv: int = 128, dtype=torch.bfloat16, segments: int = 0,
                 B: int = 1):
    """The split ``prefill_segmented`` makes: (segments, tokens of segment 0,
    tokens of each later segment)."""
    lib = load()
    g, f, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    _check(lib, lib.kda_prefill_segment_plan(B, T, H, dk, dv, code, segments, ctypes.byref(g), ctypes.byref(f),
                                             ctypes.byref(n)))
    return g.value, f.value, n.value


def prefill_segmented_workspace_bytes(T: int, H: int, dk: int = 128, dv: int = 128, dtype=torch.bfloat16,
                                      segments: int = 0, B: int = 1) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(load().kda_prefill_segmented_workspace_bytes(B, T, H, dk, dv, code, segments))


def prefill_segmented(q, k, v, alpha, beta, initial_state=None, *, segments: int = 0, gate: str = "channel",
                      output_final_state: bool = True, out=None, final_state=None, workspace=None, stream=None):
    """Prefill of one long sequence with its token axis cut into segments that
    run at the same time (kda_prefill_segmented). Arguments as ``prefill``
    with B = 1; ``segments`` = 0 lets the library plan the split, 1 runs the
    plain prefill, >= 2 forces that many."""
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(beta, "beta", torch.float32, dev)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (B, T, H, dv) or beta.shape != (B, T, H):
        raise ValueError("shape mismatch among q, k, v, beta")
    alpha = _check_gate(gate, alpha, (B, T, H), dk, dev)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev)
        if initial_state.shape != (B, H, dk, dv):
            raise ValueError(f"initial_state must be {(B, H, dk, dv)}")
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    nbytes = int(lib.kda_prefill_segmented_workspace_bytes(B, T, H, dk, dv, _dtype_code(q), segments))
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    wsize = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_prefill_segmented(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate], _ptr(beta),
                                   _ptr(initial_state), _ptr(out), _ptr(final_state), B, T, H, dk, dv,
                                   int(segments), _ptr(workspace), wsize, _stream(stream))
    _check(lib, st)
    return out, final_state


def varlen_workspace_bytes(N: int, H: int, dk: int = 128, dv: int = 128) -> int:
    return int(load().kda_varlen_workspace_bytes(N, H, dk, dv))


def varlen_prefill(q, k, v, alpha, beta, cu_seqlens, initial_state=None, *,
                   output_final_state: bool = True, out=None, final_state=None, workspace=None,
                   device_status=None, stream=None):
    """KDA prefill of sequences packed along the token axis.

    q, k, alpha: [T_total, H, d_k]; v: [T_total, H, d_v]; beta: [T_total, H];
    cu_seqlens: int32 [N + 1]; initial_state: [N, H, d_k, d_v] fp32 or None.
    Returns (o, final_state). ``device_status`` (int32 [1] on the device), when
    given, receives the device-side check result.
    """
    if q.device.type == "cpu":
        return _host_call(varlen_prefill, dict(q=q, k=k, v=v, alpha=alpha, beta=beta,
                                               cu_seqlens=cu_seqlens, initial_state=initial_state),
                          output_final_state=output_final_state)
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(alpha, "alpha", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    Tt, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if k.shape != q.shape or v.shape != (Tt, H, dv) or alpha.shape != q.shape or beta.shape != (Tt, H):
        raise ValueError("shape mismatch among q, k, v, alpha, beta")
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev)
        if initial_state.shape != (N, H, dk, dv):
            raise ValueError(f"initial_state must be {(N, H, dk, dv)}")
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
    nbytes = int(lib.kda_varlen_workspace_bytes(N, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = lib.kda_varlen_prefill(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), _ptr(beta),
                                _ptr(initial_state), _ptr(out), _ptr(final_state), _ptr(cu_seqlens),
                                N, Tt, H, dk, dv, _ptr(workspace), workspace.numel(),
                                _ptr(device_status), _stream(stream))
    _check(lib, st)
    return out, final_state


def decode_step(q, k, v, alpha, beta, state, *, out=None, stream=None):
    """One recurrent KDA step per (sequence, head); ``state`` is updated in place.

    q, k: [N, H, d_k]; v: [N, H, d_v]; alpha: [N, H, d_k] fp32; beta: [N, H] fp32;
    state: [N, H, d_k, d_v] fp32. Returns o [N, H, d_v].
    """
    if q.device.type == "cpu":
        dev = torch.device("cuda", torch.cuda.current_device())
        st_dev = state.to(dev)
        o = decode_step(q.to(dev), k.to(dev), v.to(dev), alpha.to(dev), beta.to(dev), st_dev)
        state.copy_(st_dev.to("cpu"))
        return o.to("cpu")
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(alpha, "alpha", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(state, "state", torch.float32, dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (N, H, dv) or alpha.shape != q.shape or beta.shape != (N, H) \
            or state.shape != (N, H, dk, dv):
        raise ValueError("shape mismatch among q, k, v, alpha, beta, state")
    if out is None:
        out = torch.empty_like(v)
    st = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), _ptr(beta),
                             _ptr(state), _ptr(out), N, H, dk, dv, _stream(stream))
    _check(lib, st)
    return out


def varlen_prefill_slots(q, k, v, alpha, beta, cu_seqlens, state_pool, slots, *, gate: str = "channel",
                         out=None, workspace=None, device_status=None, stream=None):
    """Packed prefill whose states live in a pool: sequence n starts from
    ``state_pool[slots[n]]`` (zeros when ``slots[n] = -1 - s``, a fresh request
    in slot s) and its final state is written back into that slot.

    q, k: [T_total, H, d_k]; v: [T_total, H, d_v]; alpha as for ``prefill``
    with lead [T_total, H]; beta: [T_total, H]; cu_seqlens, slots: int32 [N + 1],
    [N] on the device; state_pool: [P, H, d_k, d_v] fp32, updated in place.
    Returns o. ``device_status`` (int32 [1]) receives KDA_DEV_OK or a KDA_DEV_* code.
    """
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(slots, "slots", torch.int32, dev)
    _need(state_pool, "state_pool", torch.float32, dev)
    Tt, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if k.shape != q.shape or v.shape != (Tt, H, dv) or beta.shape != (Tt, H) or slots.shape != (N,) \
            or state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError("shape mismatch among q, k, v, beta, slots, state_pool")
    alpha = _check_gate(gate, alpha, (Tt, H), dk, dev)
    if out is None:
        out = torch.empty_like(v)
    nbytes = int(lib.kda_varlen_workspace_bytes(N, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = lib.kda_varlen_prefill_slots(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate],
                                      _ptr(beta), _ptr(state_pool), _ptr(slots), state_pool.shape[0], _ptr(out),
                                      _ptr(cu_seqlens), N, Tt, H, dk, dv, _ptr(workspace), workspace.numel(),
                                      _ptr(device_status), _stream(stream))
    _check(lib, st)
    return out


def decode_step_slots(q, k, v, alpha, beta, state_pool, slots, *, gate: str = "channel", out=None,
                      device_status=None, stream=None):
    """One recurrent step per (sequence, head) on ``state_pool[slots[n]]``
    (updated in place; ``-1 - s`` starts slot s from zeros).

    q, k: [N, H, d_k]; v: [N, H, d_v]; alpha as for ``prefill`` with lead
    [N, H]; beta: [N, H]; slots: int32 [N]; state_pool: [P, H, d_k, d_v] fp32.
    Returns o [N, H, d_v]. A sequence with a slot outside [0, P) is skipped and
    sets KDA_DEV_BAD_SLOT in ``device_status``.
    """
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(slots, "slots", torch.int32, dev)
    _need(state_pool, "state_pool", torch.float32, dev)
    N, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (N, H, dv) or beta.shape != (N, H) or slots.shape != (N,) \
            or state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (H, dk, dv):
        raise ValueError("shape mismatch among q, k, v, beta, slots, state_pool")
    alpha = _check_gate(gate, alpha, (N, H), dk, dev)
    if out is None:
        out = torch.empty_like(v)
    st = lib.kda_decode_step_slots(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate],
                                   _ptr(beta), _ptr(state_pool), _ptr(slots), state_pool.shape[0], _ptr(out),
                                   N, H, dk, dv, _ptr(device_status), _stream(stream))
    _check(lib, st)
    return out


def prefill_fp8(q, k, v, q_scale, k_scale, v_scale, alpha, beta, initial_state=None, *, gate: str = "channel",
                output_final_state: bool = True, out=None, final_state=None, stream=None, piece_tokens: int = 0):
    """``prefill`` on FP8 inputs in the MX block format: q, k, v are uint8
    E4M3 codes [B, T, H, 128], each 32 channels of a token-head sharing one
    E8M0 scale byte (q_scale, k_scale, v_scale: uint8 [B, T, H, 4]). The result
    equals ``prefill`` on bf16 inputs holding the dequantised values; o is bf16.
    Host (CPU) tensors go through kda_prefill_fp8_host (pieces of
    ``piece_tokens`` tokens, 0: the library's choice), like ``prefill``.
    """
    if q.device.type == "cpu":
        if out is not None or final_state is not None or stream is not None:
            raise ValueError("out, final_state and stream apply to device tensors only")
        return _host_prefill_fp8(q, k, v, q_scale, k_scale, v_scale, alpha, beta, initial_state,
                                 output_final_state=output_final_state, gate=gate, piece_tokens=piece_tokens)
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, n, torch.uint8, dev)
    _need(beta, "beta", torch.float32, dev)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (B, T, H, dv) or beta.shape != (B, T, H) \
            or q_scale.shape != (B, T, H, dk // 32) or k_scale.shape != (B, T, H, dk // 32) \
            or v_scale.shape != (B, T, H, dv // 32):
        raise ValueError("shape mismatch among q, k, v, the scales and beta")
    alpha = _check_gate(gate, alpha, (B, T, H), dk, dev)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, dev)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device=dev)
    if final_state is None and output_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    st = lib.kda_prefill_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr(alpha),
                             GATES[gate], _ptr(beta), _ptr(initial_state), _ptr(out), _ptr(final_state),
                             B, T, H, dk, dv, _stream(stream))
    _check(lib, st)
    return out, final_state


def prefill_backward(q, k, v, alpha, beta, d_o, initial_state=None, d_final_state=None, *,
                     gate: str = "channel", want_initial_state_grad: bool = True, workspace=None, stream=None):
    """Gradients of ``prefill`` (equal-length batches) for
    L = sum <d_o, o> + <d_final_state, S_T>.

    q, k, v, alpha, beta, initial_state, gate as for ``prefill``; d_o: o's
    shape and dtype; d_final_state: [B, H, d_k, d_v] fp32 or None (zero).
    Returns a dict of float32 tensors: ``dq``, ``dk``, ``dv``, ``dalpha``
    (alpha's shape; None without a gate), ``dbeta`` and ``d_initial_state``
    (None when not wanted)."""
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_o, "d_o")):
        _need(t, n, q.dtype, dev)
    _need(beta, "beta", torch.float32, dev)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape != (B, T, H, dv) or beta.shape != (B, T, H) or d_o.shape != v.shape:
        raise ValueError("shape mismatch among q, k, v, beta, d_o")
    alpha = _check_gate(gate, alpha, (B, T, H), dk, dev)
    for t, n in ((initial_state, "initial_state"), (d_final_state, "d_final_state")):
        if t is not None:
            _need(t, n, torch.float32, dev)
            if t.shape != (B, H, dk, dv):
                raise ValueError(f"{n} must be {(B, H, dk, dv)}")
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"dq": torch.empty(q.shape, **f32), "dk": torch.empty(k.shape, **f32), "dv": torch.empty(v.shape, **f32),
           "dalpha": None if alpha is None else torch.empty(alpha.shape, **f32),
           "dbeta": torch.empty(beta.shape, **f32),
           "d_initial_state": torch.empty((B, H, dk, dv), **f32) if want_initial_state_grad else None}
    nbytes = int(lib.kda_prefill_backward_workspace_bytes(B, T, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    st = lib.kda_prefill_backward_gate(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate],
                                       _ptr(beta), _ptr(initial_state), _ptr(d_o), _ptr(d_final_state),
                                       _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dalpha"]),
                                       _ptr(out["dbeta"]), _ptr(out["d_initial_state"]), B, T, H, dk, dv,
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    _check(lib, st)
    return out


def varlen_prefill_backward(q, k, v, alpha, beta, d_o, cu_seqlens, initial_state=None, d_final_state=None, *,
                            gate: str = "channel", workspace=None, device_status=None, stream=None):
    """Gradients of ``varlen_prefill`` (sequences packed by ``cu_seqlens``):
    q, k: [T_total, H, d_k]; v, d_o: [T_total, H, d_v]; alpha per ``gate``
    with lead [T_total, H]; beta: [T_total, H]; cu_seqlens: int32 [N + 1] on
    the device; initial_state, d_final_state: [N, H, d_k, d_v] fp32 or None.
    Returns the dict of ``prefill_backward``."""
    lib = load()
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_o, "d_o")):
        _need(t, n, q.dtype, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    Tt, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    if k.shape != q.shape or v.shape != (Tt, H, dv) or beta.shape != (Tt, H) or d_o.shape != v.shape:
        raise ValueError("shape mismatch among q, k, v, beta, d_o")
    alpha = _check_gate(gate, alpha, (Tt, H), dk, dev)
    for t, n in ((initial_state, "initial_state"), (d_final_state, "d_final_state")):
        if t is not None:
            _need(t, n, torch.float32, dev)
            if t.shape != (N, H, dk, dv):
                raise ValueError(f"{n} must be {(N, H, dk, dv)}")
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"dq": torch.empty(q.shape, **f32), "dk": torch.empty(k.shape, **f32), "dv": torch.empty(v.shape, **f32),
           "dalpha": None if alpha is None else torch.empty(alpha.shape, **f32),
           "dbeta": torch.empty(beta.shape, **f32), "d_initial_state": torch.empty((N, H, dk, dv), **f32)}
    nbytes = int(lib.kda_varlen_prefill_backward_workspace_bytes(N, Tt, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    st = lib.kda_varlen_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _dtype_code(q), _ptr(alpha), GATES[gate],
                                         _ptr(beta), _ptr(initial_state), _ptr(d_o), _ptr(d_final_state),
                                         _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dalpha"]),
                                         _ptr(out["dbeta"]), _ptr(out["d_initial_state"]), _ptr(cu_seqlens), N, Tt,
                                         H, dk, dv, _ptr(workspace), workspace.numel(), _ptr(device_status),
                                         _stream(stream))
    _check(lib, st)
    return out
