"""kda_prefill_host: prefill on host buffers, moved to the GPU in pieces along T.

Each piece is one kda_prefill_gate launch continuing from the state the
previous piece left, so the result must be bit for bit the device prefill run
piece by piece with the state passed between the pieces (and, for one piece,
the single device call); against the float64 oracle it meets the parity
tolerance like any prefill.
"""
import ctypes

import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

pytestmark = pytest.mark.gpu


def _alpha(x, gate):
    return {"channel": x.alpha, "scalar": x.alpha[..., 0].contiguous(), "none": None}[gate]


def _device_piece_loop(kda, x, gate, piece, algo="auto"):
    """Device prefill over [t0, t0 + piece) slices, state passed along."""
    d = torch.device("cuda")
    a = _alpha(x, gate)
    s = None if x.initial_state is None else x.initial_state.to(d)
    outs = []
    T = x.q.shape[1]
    for t0 in range(0, T, piece):
        sl = slice(t0, min(T, t0 + piece))
        part = [t[:, sl].contiguous().to(d) for t in (x.q, x.k, x.v)]
        ap = None if a is None else a[:, sl].contiguous().to(d)
        o, s = kda.prefill(*part, ap, x.beta[:, sl].contiguous().to(d), s, gate=gate, algo=algo)
        outs.append(o)
    torch.cuda.synchronize()
    return torch.cat(outs, 1).cpu(), s.cpu()


def _host(kda, x, gate, piece, pin=True, algo="auto", **kw):
    a = _alpha(x, gate)
    ts = [x.q, x.k, x.v, a, x.beta, x.initial_state]
    ts = [None if t is None else (t.pin_memory() if pin else t) for t in ts]
    return kda.prefill(*ts, gate=gate, algo=algo, piece_tokens=piece, **kw)


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
@pytest.mark.parametrize("algo", ["auto", "simt"])
def test_pieces_are_the_device_piece_loop_bit_for_bit(kda, gate, algo):
    """Three sequences of 700 tokens in pieces of 192 (three full pieces and a
    ragged one of 124): the bits of the device prefill run piece by piece."""
    x = W.batched(3, 700, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=41)
    o_h, s_h = _host(kda, x, gate, 192, algo=algo)
    o_d, s_d = _device_piece_loop(kda, x, gate, 192, algo=algo)
    assert o_h.is_pinned() and s_h.is_pinned()
    assert torch.equal(o_h, o_d) and torch.equal(s_h, s_d)


@pytest.mark.parametrize("piece", [64, 128, 320])
def test_pieces_match_the_oracle(kda, piece):
    """Pieces of 64, 128 and 320 tokens over T = 333 (ragged last chunk) meet
    the bf16 parity tolerance against the float64 oracle."""
    x = W.batched(2, 333, 3, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=42)
    o_h, s_h = _host(kda, x, "channel", piece)
    ro, rs = oracle.run(*x.tensors(), initial_state=x.initial_state)
    tol = tol_for(torch.bfloat16)
    assert_close("o", o_h, ro, tol)
    assert_close("final_state", s_h, rs, tol)


def test_one_piece_is_the_single_device_call(kda):
    """piece_tokens >= T, and the library's own choice on a small input, give
    one piece: the bits of one device call."""
    x = W.batched(2, 300, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=43)
    d = torch.device("cuda")
    o_d, s_d = kda.prefill(*[t.to(d) for t in x.tensors()], x.initial_state.to(d))
    for piece in (0, 320, 4096):
        o_h, s_h = _host(kda, x, "channel", piece)
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(s_h, s_d.cpu())


def test_pageable_host_memory(kda):
    """Inputs that are not page-locked take the same path (the driver copies
    them synchronously): same bits as page-locked ones."""
    x = W.batched(2, 260, 2, 64, 64, dtype="fp32", alpha_scale=0.1, s0_std=0.05, seed=44)
    o_p, s_p = _host(kda, x, "channel", 128, pin=True)
    o_u, s_u = _host(kda, x, "channel", 128, pin=False)
    assert torch.equal(o_p, o_u) and torch.equal(s_p, s_u)
    o_d, s_d = _device_piece_loop(kda, x, "channel", 128)
    assert torch.equal(o_p, o_d) and torch.equal(s_p, s_d)


def test_no_final_state_zero_initial_state_and_empty(kda):
    x = W.batched(2, 200, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=None, seed=45)
    o_h, s_h = _host(kda, x, "channel", 64, output_final_state=False)
    assert s_h is None
    o_d, _ = _device_piece_loop(kda, x, "channel", 64)
    assert torch.equal(o_h, o_d)
    # T = 0: the final state is the initial one; B = 0: nothing at all
    s0 = torch.randn(2, 3, 64, 64)
    e = torch.empty(2, 0, 3, 64)
    _, s = kda.prefill(e, e, e, e, torch.empty(2, 0, 3), s0)
    assert torch.equal(s, s0)
    _, s = kda.prefill(e, e, e, e, torch.empty(2, 0, 3), None)
    assert torch.count_nonzero(s) == 0
    z = torch.empty(0, 5, 3, 64)
    o, s = kda.prefill(z, z, z, z, torch.empty(0, 5, 3), None)
    assert o.shape == (0, 5, 3, 64) and s.shape == (0, 3, 64, 64)


def test_device_buffers_are_refused(kda):
    """A device pointer where a host buffer belongs is an argument error,
    reported before anything is queued."""
    from kda_gated_delta_chunkwise_gb300 import _binding
    lib = kda.load()
    d = torch.device("cuda")
    t = torch.zeros(1, 64, 1, 64, device=d)
    b = torch.zeros(1, 64, 1, device=d)
    h = torch.zeros(1, 64, 1, 64, pin_memory=True)
    ws = torch.empty(lib.kda_prefill_host_workspace_bytes(1, 64, 1, 64, 64, 0, 0, 0), dtype=torch.uint8, device=d)
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    st = lib.kda_prefill_host(p(t), p(t), p(t), 0, p(t), 0, p(b), None, p(h), None, 1, 64, 1, 64, 64, 0, 0,
                              p(ws), ws.numel(), None)
    assert st == _binding.KDA_ERR_INVALID_ARG and b"host pointer" in lib.kda_last_error()
    # a host workspace is refused too
    hw = torch.empty(ws.numel(), dtype=torch.uint8, pin_memory=True)
    st = lib.kda_prefill_host(p(h), p(h), p(h), 0, p(h), 0, p(h), None, p(h), None, 1, 64, 1, 64, 64, 0, 0,
                              p(hw), hw.numel(), None)
    assert st == _binding.KDA_ERR_INVALID_ARG and b"device memory" in lib.kda_last_error()


def test_full_size_workload_through_host_buffers(kda):
    """The 4x16x4096 workload from page-locked host memory: in pieces of 384
    tokens it is the device piece loop bit for bit; with the library's own
    piece size it meets the parity tolerance against the single device call's
    oracle-checked result."""
    x = W.prefill_4x16x4096()
    o_h, s_h = _host(kda, x, "channel", 384)
    o_d, s_d = _device_piece_loop(kda, x, "channel", 384)
    assert torch.equal(o_h, o_d) and torch.equal(s_h, s_d)
    del o_d, s_d
    o_a, s_a = _host(kda, x, "channel", 0)
    d = torch.device("cuda")
    o_1, s_1 = kda.prefill(*[t.to(d) for t in x.tensors()], None)
    tol = tol_for(torch.bfloat16)
    assert_close("o", o_a, o_1.cpu(), tol)
    assert_close("final_state", s_a, s_1.cpu(), tol)


def test_back_to_back_calls_share_a_workspace_on_one_stream(kda):
    """Two kda_prefill_host calls queued on one stream with one workspace and
    no synchronisation between them: the second call's copies wait for the
    first call's work, so both results are the single calls' bits."""
    from kda_gated_delta_chunkwise_gb300 import _binding
    lib = kda.load()
    xs = [W.batched(2, 300, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=s) for s in (51, 52)]
    ref = [_host(kda, x, "channel", 128) for x in xs]
    d = torch.device("cuda")
    nbytes = lib.kda_prefill_host_workspace_bytes(2, 300, 2, 128, 128, 1, 0, 128)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=d)
    stream = torch.cuda.Stream()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    outs = []
    for x in xs:
        h = [t.pin_memory() for t in (x.q, x.k, x.v, x.alpha, x.beta, x.initial_state)]
        o = torch.empty(x.v.shape, dtype=x.v.dtype, pin_memory=True)
        s = torch.empty(x.initial_state.shape, pin_memory=True)
        st = lib.kda_prefill_host(p(h[0]), p(h[1]), p(h[2]), 1, p(h[3]), 0, p(h[4]), p(h[5]), p(o), p(s),
                                  2, 300, 2, 128, 128, 0, 128, p(ws), nbytes, ctypes.c_void_p(stream.cuda_stream))
        assert st == _binding.KDA_OK, lib.kda_last_error()
        outs.append((o, s, h))
    stream.synchronize()
    for (o, s, _), (o_r, s_r) in zip(outs, ref):
        assert torch.equal(o, o_r) and torch.equal(s, s_r)


def test_concurrent_host_calls_from_two_threads(kda):
    """Host threads each running prefill on host buffers on their own stream
    (the library serialises the queueing, the copies share its streams): every
    result is the bits of the same call made alone."""
    import threading
    xs = [W.batched(2, 260, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=s) for s in (61, 62, 63)]
    ref = [_host(kda, x, "channel", 64) for x in xs]
    got = [None] * len(xs)
    errors = []

    def work(i):
        try:
            with torch.cuda.stream(torch.cuda.Stream()):
                for _ in range(3):
                    got[i] = _host(kda, xs[i], "channel", 64)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(xs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (o, s), (o_r, s_r) in zip(got, ref):
        assert torch.equal(o, o_r) and torch.equal(s, s_r)


def _fp8(x, d):
    out = []
    for t in (x.q, x.k, x.v):
        c, sc, _ = W.to_mxfp8(t)
        out += [c.to(d), sc.to(d)]
    return out  # cq, sq, ck, sk, cv, sv


@pytest.mark.parametrize("gate", ["channel", "none"])
def test_fp8_pieces_are_the_device_piece_loop_bit_for_bit(kda, gate):
    """FP8 inputs from host memory in pieces of 128 tokens over T = 300: the
    bits of kda_prefill_fp8 run piece by piece on the device."""
    x = W.batched(2, 300, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=71)
    cq, sq, ck, sk, cv, sv = _fp8(x, torch.device("cpu"))
    a = _alpha(x, gate)
    pin = lambda t: None if t is None else t.pin_memory()  # noqa: E731
    o_h, s_h = kda.prefill_fp8(pin(cq), pin(ck), pin(cv), pin(sq), pin(sk), pin(sv), pin(a), pin(x.beta),
                               pin(x.initial_state), gate=gate, piece_tokens=128)
    assert o_h.is_pinned() and s_h.is_pinned()
    d = torch.device("cuda")
    s = x.initial_state.to(d)
    outs = []
    for t0 in range(0, 300, 128):
        sl = slice(t0, min(300, t0 + 128))
        part = [t[:, sl].contiguous().to(d) for t in (cq, ck, cv, sq, sk, sv)]
        ap = None if a is None else a[:, sl].contiguous().to(d)
        o, s = kda.prefill_fp8(*part, ap, x.beta[:, sl].contiguous().to(d), s, gate=gate)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(o_h, torch.cat(outs, 1).cpu()) and torch.equal(s_h, s.cpu())
    # one piece: the single device call
    o1, s1 = kda.prefill_fp8(pin(cq), pin(ck), pin(cv), pin(sq), pin(sk), pin(sv), pin(a), pin(x.beta),
                             pin(x.initial_state), gate=gate, piece_tokens=0)
    part = [t.to(d) for t in (cq, ck, cv, sq, sk, sv)]
    o_d, s_d = kda.prefill_fp8(*part, None if a is None else a.to(d), x.beta.to(d), x.initial_state.to(d), gate=gate)
    assert torch.equal(o1, o_d.cpu()) and torch.equal(s1, s_d.cpu())
