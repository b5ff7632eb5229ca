"""GPU tests of the gate kinds (per-channel KDA, scalar Gated DeltaNet, no gate:
the delta rule; the K3 essay's §三 and §四) and of the state pool indexed by
slots (prefill a prompt in pieces, then decode from the same slot).

Each gate kind is compared with the float64 oracle run on the per-channel
gate it stands for (oracle.expand_gate), and bit for bit with the library's
own per-channel path fed that expanded gate: the kinds differ only in how
alpha is read. Slots are compared bit for bit with the slot-free entry
points on gathered states, and against the oracle over the whole prompt."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _gate_inputs(x: W.Inputs, gate: str):
    """alpha for the gate kind (scalar: channel 0 of the drawn gates, one per
    token-head) and the per-channel alpha it stands for, on the host."""
    lead = tuple(x.beta.shape)
    dk = x.q.shape[-1]
    if gate == "channel":
        a = x.alpha
    elif gate == "scalar":
        a = x.alpha[..., 0].contiguous()
    else:
        a = None
    full = torch.from_numpy(oracle.expand_gate(None if a is None else a.numpy(), gate, lead, dk)).float()
    return a, full


@pytest.mark.parametrize("gate", ["scalar", "none"])
@pytest.mark.parametrize("algo,dtype,d", [("tc", "bf16", 128), ("simt", "fp32", 64), ("simt", "bf16", 128)])
def test_prefill_gate_kinds(kda, gate, algo, dtype, d):
    x = W.batched(2, 300, 3, d, d, dtype=dtype, alpha_scale=0.1, s0_std=0.05, seed=31)
    a, full = _gate_inputs(x, gate)
    q, k, v, b, s0 = (t.to(DEV) for t in (x.q, x.k, x.v, x.beta, x.initial_state))
    ag = None if a is None else a.to(DEV)
    o, s = kda.prefill(q, k, v, ag, b, s0, algo=algo, gate=gate)
    # the same arithmetic as the per-channel path on the expanded gate
    oc, sc = kda.prefill(q, k, v, full.to(DEV), b, s0, algo=algo)
    assert torch.equal(o, oc) and torch.equal(s, sc)
    ro, rs = oracle.run(x.q, x.k, x.v, full.numpy(), x.beta, initial_state=x.initial_state)
    tol = tol_for(x.q.dtype)
    assert_close("o", o, ro, tol)
    assert_close("state", s, rs, tol)


def test_prefill_scalar_gate_strong_decay_runs_token_by_token(kda):
    """A scalar gate of 0 in one token (every channel at once) and a stretch of
    small gates: those chunks take the exact token loop."""
    x = W.batched(1, 200, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=32)
    a, _ = _gate_inputs(x, "scalar")
    a[0, 10, 0] = 0.0
    a[0, 70:100, 1] = 1e-3
    full = torch.from_numpy(oracle.expand_gate(a.numpy(), "scalar", tuple(x.beta.shape), 128)).float()
    q, k, v, b, s0 = (t.to(DEV) for t in (x.q, x.k, x.v, x.beta, x.initial_state))
    o, s = kda.prefill(q, k, v, a.to(DEV), b, s0, algo="tc", gate="scalar")
    ro, rs = oracle.run(x.q, x.k, x.v, full.numpy(), x.beta, initial_state=x.initial_state)
    assert_close("o", o, ro, tol_for(torch.bfloat16))
    assert_close("state", s, rs, tol_for(torch.bfloat16))


def _slots_prefill(kda, x, gate, pool, slots, lo_hi):
    """varlen_prefill_slots over the token ranges lo_hi of each sequence of x."""
    a, _ = _gate_inputs(x, gate)
    parts, cu = [], [0]
    for n, (lo, hi) in enumerate(lo_hi):
        parts.append(n)
        cu.append(cu[-1] + (hi - lo))
    sel = lambda t: torch.cat([t[n, lo:hi] for n, (lo, hi) in enumerate(lo_hi)]).contiguous()
    q, k, v, b = (sel(t).to(DEV) for t in (x.q, x.k, x.v, x.beta))
    ag = None if a is None else sel(a).to(DEV)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    status = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    o = kda.varlen_prefill_slots(q, k, v, ag, b, cu_t, pool, torch.tensor(slots, dtype=torch.int32, device=DEV),
                                 gate=gate, device_status=status)
    torch.cuda.synchronize()
    return o, cu, int(status.item())


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_prompt_prefilled_in_pieces_through_the_pool(kda, gate):
    """A prompt prefilled in three pieces, each piece continuing from the slot's
    state, matches the oracle over the whole prompt; the states land in their
    own slots and the other slots keep their bits."""
    B, T, H = 3, 333, 2
    x = W.batched(B, T, H, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=33)
    P = 6
    pool = torch.randn(P, H, 128, 128, device=DEV) * 0.05
    slots = [4, 1, 5]
    pool[slots] = x.initial_state.to(DEV)
    keep = pool[[0, 2, 3]].clone()
    o_parts = []
    for lo, hi in ((0, 100), (100, 229), (229, T)):
        o, cu, st = _slots_prefill(kda, x, gate, pool, slots, [(lo, hi)] * B)
        assert st == kda.KDA_DEV_OK
        o_parts.append([o[cu[n]:cu[n + 1]] for n in range(B)])
    o_all = torch.stack([torch.cat([p[n] for p in o_parts]) for n in range(B)])
    _, full = _gate_inputs(x, gate)
    ro, rs = oracle.run(x.q, x.k, x.v, full.numpy(), x.beta, initial_state=x.initial_state)
    tol = tol_for(torch.bfloat16)
    assert_close("o", o_all, ro, tol)
    assert_close("state", pool[slots], rs, tol)
    assert torch.equal(pool[[0, 2, 3]], keep)


def test_fresh_slots_start_from_zero_and_match_the_slot_free_call(kda):
    """slots[n] = -1 - s starts slot s from the zero state: bit for bit the
    slot-free prefill without an initial state, written into slot s."""
    x = W.batched(2, 150, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.0, seed=34)
    pool = torch.full((3, 2, 128, 128), 123.0, device=DEV)  # junk that must not be read
    o, cu, st = _slots_prefill(kda, x, "channel", pool, [-1 - 2, -1 - 0], [(0, 150)] * 2)
    assert st == kda.KDA_DEV_OK
    q, k, v, a, b = (t.to(DEV) for t in x.tensors())
    for n, slot in enumerate((2, 0)):
        on, sn = kda.prefill(q[n:n + 1], k[n:n + 1], v[n:n + 1], a[n:n + 1], b[n:n + 1], None)
        assert torch.equal(o[cu[n]:cu[n + 1]], on[0])
        assert torch.equal(pool[slot], sn[0])
    assert torch.all(pool[1] == 123.0)


def test_bad_slot_writes_nothing(kda):
    x = W.batched(2, 70, 2, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.05, seed=35)
    pool = torch.randn(2, 2, 128, 128, device=DEV)
    before = pool.clone()
    o, cu, st = _slots_prefill(kda, x, "channel", pool, [0, 2], [(0, 70)] * 2)  # slot 2 of a pool of 2
    assert st == kda.KDA_DEV_BAD_SLOT
    assert torch.equal(pool, before)


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_decode_slots_match_gathered_decode(kda, gate):
    """decode_step_slots on pool[slots] is bit for bit decode_step on the
    gathered states (gate kinds through their expanded per-channel gate), and
    the other slots keep their bits; a fresh slot starts from zeros."""
    N, H = 5, 3
    q, k, v, a, b, s0 = W.draw((N,), H, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.1, seed=36)
    if gate == "scalar":
        ag = a[..., 0].contiguous()
    elif gate == "none":
        ag = None
    else:
        ag = a
    full = torch.from_numpy(oracle.expand_gate(None if ag is None else ag.numpy(), gate, (N, H), 128)).float()
    P = 8
    pool = torch.randn(P, H, 128, 128, device=DEV) * 0.1
    slots = [6, 0, 3, -1 - 5, 1]
    pool[[6, 0, 3, 1]] = s0[[0, 1, 2, 4]].to(DEV)
    untouched = pool[[2, 4, 7]].clone()
    qd, kd, vd, bd = (t.to(DEV) for t in (q, k, v, b))
    status = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    o = kda.decode_step_slots(qd, kd, vd, None if ag is None else ag.to(DEV), bd, pool,
                              torch.tensor(slots, dtype=torch.int32, device=DEV), gate=gate, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_OK
    st = s0.clone()
    st[3] = 0.0
    st0 = st.clone()
    st = st.to(DEV)
    o_ref = kda.decode_step(qd, kd, vd, full.to(DEV), bd, st)
    assert torch.equal(o, o_ref)
    assert torch.equal(pool[[6, 0, 3, 5, 1]], st)
    assert torch.equal(pool[[2, 4, 7]], untouched)
    # and the oracle (one-token sequences)
    ro, rs = oracle.run(q[:, None], k[:, None], v[:, None], full.numpy()[:, None], b[:, None],
                        initial_state=st0)
    assert_close("o", o, ro[:, 0], tol_for(torch.bfloat16))


def test_decode_bad_slot_skips_only_its_heads(kda):
    N, H = 3, 2
    q, k, v, a, b, s0 = W.draw((N,), H, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.1, seed=37)
    pool = s0.to(DEV).clone()
    before = pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = torch.full((N, H, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    kda.decode_step_slots(q.to(DEV), k.to(DEV), v.to(DEV), a.to(DEV), b.to(DEV), pool,
                          torch.tensor([0, 9, 2], dtype=torch.int32, device=DEV), out=o, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_BAD_SLOT
    assert torch.all(o[1] == 7.0)           # skipped
    assert torch.equal(pool[1], before[1])  # slot 1 belongs to nobody here
    assert not torch.equal(pool[0], before[0]) and not torch.equal(pool[2], before[2])


def test_serving_loop_prefill_then_decode(kda):
    """Prefill a prompt into a slot, then decode token after token from the
    same slot: the outputs follow the oracle over the whole sequence."""
    H, T0, steps = 2, 190, 6
    x = W.batched(1, T0 + steps, H, 128, 128, dtype="bf16", alpha_scale=0.1, s0_std=0.0, seed=38)
    pool = torch.zeros(3, H, 128, 128, device=DEV)
    o_pre, cu, st = _slots_prefill(kda, x, "channel", pool, [-1 - 1], [(0, T0)])
    assert st == kda.KDA_DEV_OK
    outs = [o_pre]
    slot = torch.tensor([1], dtype=torch.int32, device=DEV)
    for t in range(T0, T0 + steps):
        q, k, v, a, b = (u[:, t].contiguous().to(DEV) for u in x.tensors())
        outs.append(kda.decode_step_slots(q, k, v, a, b, pool, slot))
    o_all = torch.cat([outs[0]] + [u for u in outs[1:]])
    ro, rs = oracle.run(*x.tensors())
    tol = tol_for(torch.bfloat16)
    assert_close("o", o_all, ro[0], tol)
    assert_close("state", pool[1], rs[0], tol)


def test_slots_identity_map_is_the_packed_prefill_bit_for_bit(kda):
    """The 64-sequence packed workload through the slot entry point with slot
    n for sequence n (the pool holding the initial states) gives the bits of
    kda_varlen_prefill."""
    x = W.varlen_64seq()
    q, k, v, a, b = (t.to(DEV) for t in x.tensors())
    cu = x.cu_seqlens.to(DEV)
    s0 = x.initial_state.to(DEV)
    o_ref, s_ref = kda.varlen_prefill(q, k, v, a, b, cu, s0)
    pool = s0.clone()
    slots = torch.arange(x.num_seqs, dtype=torch.int32, device=DEV)
    status = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    o = kda.varlen_prefill_slots(q, k, v, a, b, cu, pool, slots, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == kda.KDA_DEV_OK
    assert torch.equal(o, o_ref)
    assert torch.equal(pool, s_ref)


def test_long_prompt_prefilled_in_pieces(kda):
    """The 131,072-token workload (32 heads) prefilled through a slot in four
    pieces equals one prefill of the whole sequence to rounding (the state
    carries everything between the pieces)."""
    x = W.prefill_long_131k()
    q, k, v, a, b = (t.to(DEV) for t in x.tensors())
    s0 = x.initial_state.to(DEV)
    o_ref, s_ref = kda.prefill(q, k, v, a, b, s0)
    pool = torch.zeros(2, 32, 128, 128, device=DEV)
    pool[1] = s0[0]
    T = q.shape[1]
    outs = []
    for lo in range(0, T, T // 4):
        hi = lo + T // 4
        cu = torch.tensor([0, hi - lo], dtype=torch.int32, device=DEV)
        outs.append(kda.varlen_prefill_slots(q[0, lo:hi].contiguous(), k[0, lo:hi].contiguous(),
                                             v[0, lo:hi].contiguous(), a[0, lo:hi].contiguous(),
                                             b[0, lo:hi].contiguous(), cu, pool,
                                             torch.tensor([1], dtype=torch.int32, device=DEV)))
    o = torch.cat(outs)[None]
    tol = tol_for(torch.bfloat16)
    assert_close("o", o, o_ref, tol)
    assert_close("state", pool[1:2], s_ref, tol)
