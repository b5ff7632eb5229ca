"""GPU parity of kda_prefill_segmented (one long sequence cut into segments
that run at once, joined through the segments' transition products) against
the float64 oracle, on every output and the final state."""
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import TOL_BF16, assert_close, rel_l2

pytestmark = pytest.mark.gpu


def _dev(x: W.Inputs):
    d = torch.device("cuda")
    s0 = None if x.initial_state is None else x.initial_state.to(d)
    return [t.to(d) for t in x.tensors()] + [s0]


def _oracle(x: W.Inputs):
    return oracle.run(*x.tensors(), initial_state=x.initial_state)


def _check_split(kda, x: W.Inputs, segments, want_segments=None):
    q, k, v, a, b, s0 = _dev(x)
    o, s = kda.prefill_segmented(q, k, v, a, b, s0, segments=segments)
    torch.cuda.synchronize()
    assert kda.device_errors() == 0
    G, first, seg = kda.segment_plan(x.q.shape[1], x.q.shape[2], segments=segments)
    if want_segments is not None:
        assert G == want_segments
    ro, rs = _oracle(x)
    assert_close("o", o.cpu(), ro, TOL_BF16)
    assert_close("final_state", s.cpu(), rs, TOL_BF16)
    # against the unsplit tensor-core prefill: the same bf16 error budget
    o1, s1 = kda.prefill(q, k, v, a, b, s0, algo="tc")
    assert_close("o vs prefill", o, o1, TOL_BF16)
    assert_close("S vs prefill", s, s1, TOL_BF16)
    return o, s, (G, first, seg), (ro, rs)


@pytest.mark.parametrize("T,H,segments,s0", [(1000, 2, 2, True), (1000, 2, 3, False), (4133, 3, 5, True),
                                             (130, 2, 8, True), (64 * 40, 4, 16, True)])
def test_forced_splits(kda, T, H, segments, s0):
    """Forced splits over several chunks and a ragged tail, segments of one
    chunk included; with and without an initial state."""
    x = W.batched(1, T, H, dtype="bf16", alpha_scale=0.1, s0_std=0.05 if s0 else None, seed=T + segments)
    _, _, (G, first, seg), _ = _check_split(kda, x, segments)
    assert G >= 2 and first + (G - 2) * seg < T <= first + (G - 1) * seg


def test_long_memory_carries_across_segments(kda):
    """Slow gates (alpha ~ 0.999) and weak writes (beta / 20) keep the state of
    one segment alive through the next ones, so the correction carries most
    of the later segments' outputs: a later segment run alone from zero is far
    from the oracle, the split is not."""
    x = W.batched(1, 3000, 2, dtype="bf16", alpha_scale=1e-3, s0_std=0.5, seed=77)
    x.beta.mul_(0.05)
    _, _, (G, first, seg), (ro, _) = _check_split(kda, x, 4, want_segments=4)
    q, k, v, a, b, _ = _dev(x)
    sl = slice(first, first + seg)
    alone, _ = kda.prefill(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                           a[:, sl].contiguous(), b[:, sl].contiguous(), None)
    assert rel_l2(alone.cpu(), ro[:, sl]) > 0.2


def test_strong_decay_across_segment_boundaries(kda):
    """Token-by-token chunks (alpha = 0, e^-138 channels, e^-103 chunks) in
    segment 0, at a segment boundary and inside later segments."""
    x = W.batched(1, 1500, 2, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=15)
    G, first, seg = kda.segment_plan(1500, 2, segments=3)
    x.alpha[0, 10, 0, :] = 0.0
    x.alpha[0, first - 3:first + 20, 1, 5] = 1e-3
    x.alpha[0, first + seg:first + seg + 64, 1, :64] = 0.2
    x.alpha[0, first + seg + 100, :, :] = 0.0
    _check_split(kda, x, 3, want_segments=3)


def test_automatic_plan_1x16x16384(kda):
    """The library's own plan on a 16-head sequence of 16,384 tokens."""
    x = W.batched(1, 16384, 16, dtype="bf16", alpha_scale=W.split_scales(128), s0_std=0.01, seed=3)
    G, _, _ = kda.segment_plan(16384, 16)
    assert G >= 2
    _check_split(kda, x, 0, want_segments=G)


def test_in_place_state_optional_outputs_and_repeat(kda):
    x = W.batched(1, 2000, 2, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=31)
    q, k, v, a, b, s0 = _dev(x)
    o_ref, s_ref = kda.prefill_segmented(q, k, v, a, b, s0, segments=3)
    o2, s2 = kda.prefill_segmented(q, k, v, a, b, s0, segments=3)
    torch.testing.assert_close(o2, o_ref, rtol=0, atol=0)          # two calls, the same bits
    torch.testing.assert_close(s2, s_ref, rtol=0, atol=0)
    st = s0.clone()
    o3, s3 = kda.prefill_segmented(q, k, v, a, b, st, segments=3, final_state=st)
    assert s3.data_ptr() == st.data_ptr()
    torch.testing.assert_close(st, s_ref, rtol=0, atol=0)
    torch.testing.assert_close(o3, o_ref, rtol=0, atol=0)
    o4, s4 = kda.prefill_segmented(q, k, v, a, b, s0, segments=3, output_final_state=False)
    assert s4 is None
    torch.testing.assert_close(o4, o_ref, rtol=0, atol=0)
    o5, s5 = kda.prefill_segmented(q, k, v, a, b, None, segments=3)
    o6, s6 = kda.prefill_segmented(q, k, v, a, b, torch.zeros_like(s0), segments=3)
    torch.testing.assert_close(o5, o6, rtol=0, atol=0)
    torch.testing.assert_close(s5, s6, rtol=0, atol=0)
    torch.cuda.synchronize()
    assert kda.device_errors() == 0


@pytest.mark.parametrize("gate", ["scalar", "none"])
def test_gate_kinds(kda, gate):
    """A scalar gate (Gated DeltaNet) and no gate (the delta rule) through a
    forced split: against the oracle on the per-channel gate each stands for,
    and against the unsplit prefill of the same gate kind."""
    x = W.batched(1, 2500, 3, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=41)
    lead = tuple(x.beta.shape)
    a_g = x.alpha[..., 0].contiguous() if gate == "scalar" else None
    full = torch.from_numpy(oracle.expand_gate(None if a_g is None else a_g.numpy(), gate, lead, 128)).float()
    ro, rs = oracle.run(x.q, x.k, x.v, full, x.beta, initial_state=x.initial_state)
    q, k, v, _, b, s0 = _dev(x)
    ad = None if a_g is None else a_g.cuda()
    o, s = kda.prefill_segmented(q, k, v, ad, b, s0, segments=4, gate=gate)
    assert_close("o", o.cpu(), ro, TOL_BF16)
    assert_close("final_state", s.cpu(), rs, TOL_BF16)
    o1, s1 = kda.prefill(q, k, v, ad, b, s0, gate=gate, algo="tc")
    assert_close("o vs prefill", o, o1, TOL_BF16)
    assert_close("S vs prefill", s, s1, TOL_BF16)


def test_no_split_is_the_plain_prefill(kda):
    """segments = 1, and configurations the split does not take (fp32 inputs,
    d = 64, more than 38 heads under the automatic plan), are kda_prefill
    bit for bit."""
    for x, segs in ((W.batched(1, 700, 2, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=1), 1),
                    (W.batched(1, 700, 2, dtype="fp32", alpha_scale=0.1, s0_std=0.05, seed=2), 0),
                    (W.batched(1, 700, 2, 64, 64, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=3), 0),
                    (W.batched(1, 1024, 40, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=4), 0)):
        q, k, v, a, b, s0 = _dev(x)
        assert kda.segment_plan(x.q.shape[1], x.q.shape[2], x.q.shape[3], x.v.shape[3], q.dtype, segs)[0] == 1
        o, s = kda.prefill_segmented(q, k, v, a, b, s0, segments=segs)
        o1, s1 = kda.prefill(q, k, v, a, b, s0)
        torch.testing.assert_close(o, o1, rtol=0, atol=0)
        torch.testing.assert_close(s, s1, rtol=0, atol=0)
    with pytest.raises(kda.KdaError):
        x = W.batched(1, 700, 2, dtype="fp32", alpha_scale=0.1, seed=5)
        q, k, v, a, b, _ = _dev(x)
        kda.prefill_segmented(q, k, v, a, b, None, segments=2)


def test_cuda_graph_capture_and_side_stream(kda):
    """The call forks onto the library's own streams and joins back, so it is
    captured whole into a CUDA graph (the replay matches the eager call bit for
    bit) and it orders correctly on a caller's non-default stream."""
    x = W.batched(1, 3000, 4, dtype="bf16", alpha_scale=W.split_scales(128), s0_std=0.05, seed=51)
    q, k, v, a, b, s0 = _dev(x)
    T, H = q.shape[1], q.shape[2]
    ws = torch.empty(kda.prefill_segmented_workspace_bytes(T, H, segments=4), dtype=torch.uint8, device="cuda")
    o_ref, s_ref = kda.prefill_segmented(q, k, v, a, b, s0, segments=4, workspace=ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        o1, s1 = kda.prefill_segmented(q, k, v, a, b, s0, segments=4, workspace=ws)
        o1c, s1c = o1.clone(), s1.clone()  # ordered after the call on the same stream
    torch.cuda.current_stream().wait_stream(side)
    torch.testing.assert_close(o1c, o_ref, rtol=0, atol=0)
    torch.testing.assert_close(s1c, s_ref, rtol=0, atol=0)
    o = torch.empty_like(o_ref)
    st = torch.empty_like(s_ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        kda.prefill_segmented(q, k, v, a, b, s0, segments=4, out=o, final_state=st, workspace=ws)
    o.zero_()
    st.zero_()
    g.replay()
    torch.cuda.synchronize()
    torch.testing.assert_close(o, o_ref, rtol=0, atol=0)
    torch.testing.assert_close(st, s_ref, rtol=0, atol=0)
    assert kda.device_errors() == 0
