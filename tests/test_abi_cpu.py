"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/kda.h declares, and argument checks reject bad calls before
any CUDA work (no kernel is launched by these tests)."""
import ctypes
import os
import re

import pytest

import kda_gated_delta_chunkwise_gb300 as kda
from kda_gated_delta_chunkwise_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kda.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kda_prefill", "kda_varlen_prefill", "kda_decode_step", "kda_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    for name in kda.EXPORTS:
        assert hasattr(lib, name)


def test_abi_version(lib):
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    ver = int(re.search(r"#define KDA_ABI_VERSION (\d+)", text).group(1))
    assert lib.kda_abi_version() == ver


def _prefill(lib, dk=128, dv=128, B=1, T=4, H=1, ptr=0x1000, algo=0, dtype=1, beta_ptr=None):
    p = ctypes.c_void_p(ptr)
    b = ctypes.c_void_p(ptr if beta_ptr is None else beta_ptr)
    return lib.kda_prefill_ex(p, p, p, dtype, p, b, None, p, None, B, T, H, dk, dv, algo, None)


def test_unsupported_head_size_is_rejected_before_launch(lib):
    assert _prefill(lib, dk=96) == 2
    assert b"64 or 128" in lib.kda_last_error()
    assert _prefill(lib, dv=256) == 2


def test_null_and_misaligned_pointers_are_rejected(lib):
    assert _prefill(lib, ptr=0) == 1
    assert b"must not be NULL" in lib.kda_last_error()
    assert _prefill(lib, ptr=0x1004) == 1
    assert b"16-byte aligned" in lib.kda_last_error()
    assert _prefill(lib, beta_ptr=0x1002) == 1


def test_bad_sizes_and_enums(lib):
    assert _prefill(lib, B=-1) == 1
    assert _prefill(lib, H=0) == 1
    assert _prefill(lib, dtype=7) == 1
    assert _prefill(lib, algo=9) == 1


def test_tensor_core_path_rejects_fp32(lib):
    assert _prefill(lib, algo=2, dtype=0) == 2


def test_empty_batches_are_no_ops(lib):
    # B = 0 or T = 0 without a final state: nothing to do, nothing launched
    assert _prefill(lib, B=0) == 0
    assert _prefill(lib, T=0) == 0


def test_varlen_argument_checks(lib):
    p = ctypes.c_void_p(0x1000)
    ws = lib.kda_varlen_workspace_bytes(64, 16, 128, 128)
    assert ws >= 64 * 4 and ws % 256 == 0
    # no workspace
    st = lib.kda_varlen_prefill(p, p, p, 1, p, p, None, p, None, p, 64, 1000, 16, 128, 128,
                                None, 0, None, None)
    assert st == 5
    # misaligned workspace
    st = lib.kda_varlen_prefill(p, p, p, 1, p, p, None, p, None, p, 64, 1000, 16, 128, 128,
                                ctypes.c_void_p(0x1010), ws, None, None)
    assert st == 5
    # missing cu_seqlens
    st = lib.kda_varlen_prefill(p, p, p, 1, p, p, None, p, None, None, 64, 1000, 16, 128, 128,
                                p, ws, None, None)
    assert st == 1
    # zero sequences: nothing to do
    st = lib.kda_varlen_prefill(None, None, None, 1, None, None, None, None, None, None, 0, 0, 16,
                                128, 128, None, 0, None, None)
    assert st == 0


def test_decode_argument_checks(lib):
    p = ctypes.c_void_p(0x1000)
    assert lib.kda_decode_step(p, p, p, 1, p, p, None, p, 4, 2, 128, 128, None) == 1
    assert lib.kda_decode_step(p, p, p, 1, p, p, p, p, 4, 2, 80, 128, None) == 2
    assert lib.kda_decode_step(p, p, p, 1, p, p, p, p, 0, 2, 128, 128, None) == 0


def test_gate_and_slot_argument_checks(lib):
    """The gate-kind and slot entry points reject bad arguments before any
    launch (no GPU is touched here)."""
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    ws = 4096
    # unknown gate kind
    assert lib.kda_prefill_gate(p, p, p, 1, p, 7, p, None, p, None, 1, 8, 2, 128, 128, 0, None) == 1
    # per-channel gate needs a 16-byte aligned alpha; a scalar gate 4-byte; no gate none at all
    assert lib.kda_prefill_gate(p, p, p, 1, odd, 0, p, None, p, None, 1, 8, 2, 128, 128, 0, None) == 1
    assert lib.kda_prefill_gate(p, p, p, 1, ctypes.c_void_p(0x1001), 1, p, None, p, None, 1, 8, 2, 128, 128, 0,
                                None) == 1
    assert lib.kda_prefill_gate(p, p, p, 1, None, 1, p, None, p, None, 1, 8, 2, 128, 128, 0, None) == 1
    # empty batch: nothing to do whatever the gate
    assert lib.kda_prefill_gate(None, None, None, 1, None, 2, None, None, None, None, 0, 8, 2, 128, 128, 0,
                                None) == 0
    # slots: pool and slot map required, pool_size positive
    assert lib.kda_varlen_prefill_slots(p, p, p, 1, p, 0, p, None, p, 4, p, p, 2, 100, 2, 128, 128, p, ws,
                                        None, None) == 1
    assert lib.kda_varlen_prefill_slots(p, p, p, 1, p, 0, p, p, None, 4, p, p, 2, 100, 2, 128, 128, p, ws,
                                        None, None) == 1
    assert lib.kda_varlen_prefill_slots(p, p, p, 1, p, 0, p, p, p, 0, p, p, 2, 100, 2, 128, 128, p, ws,
                                        None, None) == 1
    assert lib.kda_varlen_prefill_slots(p, p, p, 1, p, 9, p, p, p, 4, p, p, 2, 100, 2, 128, 128, p, ws,
                                        None, None) == 1
    assert lib.kda_varlen_prefill_slots(None, None, None, 1, None, 0, None, None, None, 0, None, None, 0, 0, 2,
                                        128, 128, None, 0, None, None) == 0
    assert lib.kda_decode_step_slots(p, p, p, 1, p, 0, p, None, p, 4, p, 3, 2, 128, 128, None, None) == 1
    assert lib.kda_decode_step_slots(p, p, p, 1, p, 0, p, p, None, 4, p, 3, 2, 128, 128, None, None) == 1
    assert lib.kda_decode_step_slots(p, p, p, 1, p, 0, p, p, p, 0, p, 3, 2, 128, 128, None, None) == 1
    assert lib.kda_decode_step_slots(p, p, p, 1, p, 0, p, p, p, 4, p, 3, 2, 128, 128, odd, None) == 1
    assert lib.kda_decode_step_slots(p, p, p, 1, p, 0, p, p, p, 4, p, 0, 2, 128, 128, None, None) == 0


def test_fp8_argument_checks(lib):
    p = ctypes.c_void_p(0x1000)
    # scales required, d = 128 only, gate checked
    assert lib.kda_prefill_fp8(p, p, p, None, p, p, p, 0, p, None, p, None, 1, 8, 2, 128, 128, None) == 1
    assert lib.kda_prefill_fp8(p, p, p, p, p, p, p, 0, p, None, p, None, 1, 8, 2, 64, 64, None) == 2
    assert lib.kda_prefill_fp8(p, p, p, p, p, p, p, 5, p, None, p, None, 1, 8, 2, 128, 128, None) == 1
    assert lib.kda_prefill_fp8(p, p, p, ctypes.c_void_p(0x1001), p, p, p, 0, p, None, p, None, 1, 8, 2, 128, 128,
                               None) == 1
    assert lib.kda_prefill_fp8(None, None, None, None, None, None, None, 0, None, None, None, None, 0, 8, 2, 128,
                               128, None) == 0


def test_host_prefill_argument_checks(lib):
    """kda_prefill_host checks its arguments and workspace before any CUDA call."""
    p = ctypes.c_void_p(0x1000)

    def call(dtype=1, gate=0, B=1, T=64, H=1, dk=64, dv=64, algo=0, piece=0, ws=p, nbytes=1 << 30, q=p, a=p):
        return lib.kda_prefill_host(q, p, p, dtype, a, gate, p, None, p, None, B, T, H, dk, dv, algo, piece,
                                    ws, nbytes, None)

    assert call(dtype=5) == 1
    assert call(gate=3) == 1
    assert call(algo=7) == 1
    assert call(dk=96) == 2
    assert call(piece=100) == 1 and b"multiple of 64" in lib.kda_last_error()
    assert call(piece=-64) == 1
    assert call(q=None) == 1
    assert call(a=None) == 1                # the channel gate needs alpha
    assert call(ws=None) == 5               # no workspace
    assert call(nbytes=16) == 5             # too small
    assert call(ws=ctypes.c_void_p(0x1008)) == 1  # misaligned workspace
    assert call(B=0) == 0                   # nothing to do
    assert call(T=0) == 0                   # no tokens and no final state


def test_host_prefill_workspace_size(lib):
    """Three piece buffers of q, k, v, alpha, beta and o (each rounded up to
    256 bytes) plus one set of states."""
    f = lib.kda_prefill_host_workspace_bytes
    # B=1, T=64, H=1, d=64, fp32, channel gate, pieces of 64 tokens:
    # q, k, v, alpha, o 64*64*4 = 16384 bytes each, beta 256; state 16384
    assert f(1, 64, 1, 64, 64, 0, 0, 64) == 3 * (5 * 16384 + 256) + 16384
    # no gate: no alpha buffer; a piece longer than T holds T tokens
    assert f(1, 64, 1, 64, 64, 0, 2, 512) == 3 * (4 * 16384 + 256) + 16384
    # invalid arguments give 0
    assert f(1, 64, 1, 96, 64, 0, 0, 0) == 0
    assert f(1, 64, 1, 64, 64, 0, 0, 65) == 0
    # the library's own piece size stays within about 32 MiB of input per piece
    B, T, H = 4, 4096, 16
    full_in = B * T * H * (3 * 128 * 2 + 128 * 4 + 4)
    ws = f(B, T, H, 128, 128, 1, 0, 0)
    assert 0 < ws < full_in


def test_fp8_host_prefill_argument_checks(lib):
    """kda_prefill_fp8_host checks its arguments and workspace before any CUDA call."""
    p = ctypes.c_void_p(0x1000)

    def call(gate=0, B=1, T=64, H=1, dk=128, dv=128, piece=0, ws=p, nbytes=1 << 30, qs=p):
        return lib.kda_prefill_fp8_host(p, p, p, qs, p, p, p, gate, p, None, p, None, B, T, H, dk, dv, piece,
                                        ws, nbytes, None)

    assert call(gate=5) == 1
    assert call(dk=64) == 2 and b"128" in lib.kda_last_error()
    assert call(piece=96) == 1
    assert call(qs=None) == 1
    assert call(ws=None) == 5
    assert call(B=0) == 0
    f = lib.kda_prefill_fp8_host_workspace_bytes
    # B=1, T=64, H=1, d=128, channel gate, pieces of 64: q, k, v 64*128 = 8192 B
    # each; scales 64*4 = 256 each; alpha 64*512 = 32768; beta 256; o (bf16)
    # 16384; state 65536
    assert f(1, 64, 1, 128, 128, 0, 64) == 3 * (3 * 8192 + 3 * 256 + 32768 + 256 + 16384) + 65536
    assert f(1, 64, 1, 64, 128, 0, 64) == 0


def test_host_prefill_picks_pieces_of_about_32_mib(lib):
    """The library's own piece size on the benchmark shape (4 x 16 x 4096,
    bf16, per-channel gate): 20,544 input bytes per token row, so eleven
    pieces of at most 32 MiB, each 384 tokens (whole chunks); the workspace is
    that of explicit 384-token pieces."""
    f = lib.kda_prefill_host_workspace_bytes
    assert f(4, 4096, 16, 128, 128, 1, 0, 0) == f(4, 4096, 16, 128, 128, 1, 0, 384)
    assert f(4, 4096, 16, 128, 128, 1, 0, 0) != f(4, 4096, 16, 128, 128, 1, 0, 448)
    row = 4 * (3 * 16 * 128 * 2 + 16 * 128 * 4 + 16 * 4)
    assert 384 * row <= 32 << 20 < 448 * row
    # a small input is one piece: the workspace holds T tokens
    assert f(1, 300, 2, 128, 128, 1, 0, 0) == f(1, 300, 2, 128, 128, 1, 0, 320)


def test_grid_size_limit_is_checked_before_launch(lib):
    """One CTA per (sequence, head, value half): N * H * 2 beyond 2^31 - 1
    blocks is rejected as unsupported on every prefill entry point."""
    p = ctypes.c_void_p(0x1000)
    big_h = 1 << 20  # B * H * 2 = 2^31 with B = 1024
    assert lib.kda_prefill_ex(p, p, p, 1, p, p, None, p, None, 1024, 1, big_h, 128, 128, 0, None) == 2
    assert b"N * H * 2" in lib.kda_last_error()
    assert lib.kda_prefill_fp8(p, p, p, p, p, p, p, 0, p, None, p, None, 1024, 1, big_h, 128, 128, None) == 2
    ws = lib.kda_varlen_workspace_bytes(1024, big_h, 128, 128)
    st = lib.kda_varlen_prefill(p, p, p, 1, p, p, None, p, None, p, 1024, 1024, big_h, 128, 128,
                                ctypes.c_void_p(0x100000), ws, None, None)
    assert st == 2
    # just below the limit passes the check (and fails later on the pointers)
    assert lib.kda_prefill_ex(None, p, p, 1, p, p, None, p, None, 1023, 1, big_h, 128, 128, 0, None) == 1


def test_equal_length_prefill_needs_no_workspace(lib):
    assert lib.kda_prefill_workspace_bytes(4, 4096, 16, 128, 128) == 0
    assert kda.prefill_workspace_bytes(1, 1 << 20, 32) == 0


def test_selftest_argument_checks(lib):
    p = ctypes.c_void_p(0x1000)
    assert lib.kda_selftest_bounded_wait(p, p, p, p, p, p, None, 0, 0, None) == 1      # T = 0
    assert lib.kda_selftest_bounded_wait(p, p, p, p, p, p, None, 256, 4, None) == 1    # chunk 4 of 4
    assert b"stall_chunk" in lib.kda_last_error()
    assert lib.kda_selftest_bounded_wait(p, p, p, p, p, p, None, 256, -1, None) == 1
    assert lib.kda_selftest_bounded_wait(None, p, p, p, p, p, None, 256, 0, None) == 1


def test_backward_argument_checks(lib):
    p = ctypes.c_void_p(0x1000)
    ws = lib.kda_prefill_backward_workspace_bytes(2, 130, 3, 128, 128)
    chunks = 2 * 3 * 3
    # per chunk: the state, the state gradient, the chunk tables (Kr, Qr, Kc,
    # T, P, mu, beta and a flag) and four 64 x d_v work tiles (U, V - X, dU, dR)
    assert ws == chunks * (2 * 128 * 128 + 3 * 64 * 128 + 2 * 64 * 64 + 128 + 64 + 4 + 4 * 64 * 128) * 4
    args = [p, p, p, 1, p, p, None, p, None, p, p, p, p, p, None, 2, 130, 3, 128, 128]
    assert lib.kda_prefill_backward(*args, None, 0, None) == 5           # no workspace
    assert lib.kda_prefill_backward(*args, ctypes.c_void_p(0x1008), ws, None) == 5  # misaligned
    bad = list(args)
    bad[9] = None                                                        # dq
    assert lib.kda_prefill_backward(*bad, p, ws, None) == 1
    bad = list(args)
    bad[18] = 96                                                         # d_k
    assert lib.kda_prefill_backward(*bad, p, ws, None) == 2
    # nothing to do for B = 0
    z = list(args)
    z[15] = 0
    assert lib.kda_prefill_backward(*z, None, 0, None) == 0


def _plan(lib, B, T, H, dk=128, dv=128, dtype=1, segments=0):
    g, f, n = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = lib.kda_prefill_segment_plan(B, T, H, dk, dv, dtype, segments, ctypes.byref(g), ctypes.byref(f),
                                      ctypes.byref(n))
    return st, g.value, f.value, n.value


def test_segment_plan(lib):
    # the long-context workload (2048 chunks, 32 heads): segment 0 runs alone
    # on 32 of the 76 cluster slots while the 4 later segments run twice
    # (local, then transition) on the other 44, each launch in 3 waves (w = 6)
    # with a start-up of 16 chunk steps per wave
    st, G, first, seg = _plan(lib, 1, 131072, 32)
    assert (st, G) == (0, 5)
    assert seg == ((2048 + 16 - 6 * 16) // (6 + 4)) * 64 and first == 131072 - 4 * seg
    # fewer heads leave room for more segments; every plan covers T
    for T, H in ((131072, 16), (131072, 1), (4096, 16), (100_000, 8), (65 * 64 + 5, 4)):
        st, G, first, seg = _plan(lib, 1, T, H)
        assert st == 0 and G >= 1
        if G > 1:
            assert first % 64 == 0 and seg % 64 == 0
            assert first + (G - 2) * seg < T <= first + (G - 1) * seg
            assert seg >= 8 * 64 and first >= seg
    # no split where it cannot pay or cannot run
    assert _plan(lib, 1, 131072, 39)[1] == 1          # more than 38 heads
    assert _plan(lib, 1, 64 * 9, 32)[1] == 1          # too short
    assert _plan(lib, 2, 131072, 8)[1] == 1           # a batch
    assert _plan(lib, 1, 131072, 8, dtype=0)[1] == 1  # fp32 inputs
    assert _plan(lib, 1, 131072, 8, dk=64)[1] == 1
    assert _plan(lib, 1, 131072, 8, segments=1)[1:] == (1, 131072, 0)
    # forced splits
    assert _plan(lib, 1, 1000, 2, segments=3) == (0, 3, 512, 256)
    assert _plan(lib, 1, 130, 2, segments=8) == (0, 2, 128, 64)  # three chunks: the last segment has 2 tokens
    assert _plan(lib, 1, 1000, 2, dtype=0, segments=2)[0] == 2
    assert _plan(lib, 2, 1000, 2, segments=2)[0] == 2
    assert _plan(lib, 1, 1000, 2, segments=4097)[0] == 2
    assert _plan(lib, 1, 1000, 65536, segments=2)[0] == 2


def test_segmented_workspace_and_argument_checks(lib):
    T, H = 131072, 32
    _, G, first, seg = _plan(lib, 1, T, H)
    T1 = T - first
    mat = 128 * 128

    def up(x):
        return (x + 255) // 256 * 256

    want = (up(4 * G) + up(lib.kda_varlen_workspace_bytes(G - 1, H, 128, 128)) + up(4 * H * mat)
            + 3 * up(4 * (G - 1) * H * mat) + up(2 * (G - 1) * H * mat) + 2 * up(2 * T1 * H * 128))
    assert lib.kda_prefill_segmented_workspace_bytes(1, T, H, 128, 128, 1, 0) == want
    assert lib.kda_prefill_segmented_workspace_bytes(1, T, 39, 128, 128, 1, 0) == 0  # no split
    p = ctypes.c_void_p(0x1000)
    args = [p, p, p, 1, p, 0, p, None, p, None, 1, 1000, 2, 128, 128, 3]
    ws = lib.kda_prefill_segmented_workspace_bytes(1, 1000, 2, 128, 128, 1, 3)
    assert lib.kda_prefill_segmented(*args, None, 0, None) == 5                     # no workspace
    assert lib.kda_prefill_segmented(*args, ctypes.c_void_p(0x1010), ws, None) == 5  # misaligned
    assert lib.kda_prefill_segmented(*args, p, ws - 1, None) == 5                    # too small
    bad = list(args)
    bad[0] = None
    assert lib.kda_prefill_segmented(*bad, p, ws, None) == 1
    bad = list(args)
    bad[6] = ctypes.c_void_p(0x1002)                                                 # beta
    assert lib.kda_prefill_segmented(*bad, p, ws, None) == 1
    bad = list(args)
    bad[3] = 0                                                                       # fp32, forced split
    assert lib.kda_prefill_segmented(*bad, p, ws, None) == 2
    bad = list(args)
    bad[5] = 7                                                                       # gate kind
    assert lib.kda_prefill_segmented(*bad, p, ws, None) == 1
    bad = list(args)
    bad[4] = ctypes.c_void_p(0x1004)                                                 # per-channel alpha: 16 bytes
    assert lib.kda_prefill_segmented(*bad, p, ws, None) == 1
    bad[5] = 1                                                                       # a scalar gate: 4 bytes do
    assert lib.kda_prefill_segmented(*bad, None, 0, None) == 5
    bad[4], bad[5] = None, 2                                                         # no gate: alpha unused
    assert lib.kda_prefill_segmented(*bad, None, 0, None) == 5
