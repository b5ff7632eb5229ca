"""Every wait of the tensor-core prefill is bounded. kda_selftest_bounded_wait
runs that kernel with its state chain stalled on a barrier that nothing ever
completes; the stuck wait must give up (about a second), the kernel's other
groups must wind down, the kernel must return with a nonzero device error
word, and the same CUDA context must then run an ordinary call that matches
the oracle. The failure is made on purpose without any fault: a wait that
never completes, ended by its own iteration bound."""
import time

import pytest
import torch

import oracle
from kda_gated_delta_chunkwise_gb300 import workloads as W
from _parity import assert_close, tol_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("stall_chunk", [0, 2])
def test_stuck_wait_ends_in_an_error_and_the_context_stays_usable(kda, stall_chunk):
    x = W.batched(1, 256, 1, 128, 128, dtype="bf16", alpha_scale=0.1, seed=41)
    q, k, v, a, b = (t[0, :, 0].contiguous().cuda() for t in x.tensors())
    assert kda.device_errors(reset=True) == 0
    t0 = time.perf_counter()
    kda.selftest_bounded_wait(q, k, v, a, b, stall_chunk)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    errs = kda.device_errors(reset=True)
    assert errs != 0, "the stalled kernel returned without reporting its timeout"
    assert waited < 60.0, f"the wind-down took {waited:.1f} s"
    # the context is intact: an ordinary call on the same inputs is correct
    o, s = kda.prefill(q[None, :, None], k[None, :, None], v[None, :, None], a[None, :, None],
                       b[None, :, None], None)
    torch.cuda.synchronize()
    assert kda.device_errors(reset=True) == 0
    ro, rs = oracle.run(*x.tensors())
    tol = tol_for(x.q.dtype)
    assert_close("o", o.cpu(), ro, tol)
    assert_close("final_state", s.cpu(), rs, tol)
