"""A bounded pipeline wait that runs out, on the GPU, without a fault.

Every mbarrier wait in the kernels gives up after the wait bound
(fa_set_wait_timeout_ns).  With the bound set to 1 ns, a wait that is not
satisfied within one poll of its barrier (a poll may suspend the thread for
a short, hardware-chosen time) gives up at once: the kernel records
FA_ERR_TIMEOUT with the site of the wait in the per-device error word, lets
the copies and tensor-core operations it has issued complete, frees its
tensor memory and returns.  Nothing is injected: the same kernels run on
valid inputs, only the bound differs.  Each main kernel (forward, the d = 64
and the d = 128 backward) is made to give up once on a small problem, and
the persistent kernels on one with more work items than SMs; the
status is read back, the bound restored, and a normal call on the same
device then matches the oracle.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from io_aware_exact_10_gb300 import workloads as W
from parity import check_heads, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def gives_up(fn):
    """Run fn() with a 1 ns wait bound; return (status, raw error word)."""
    assert fa.fa_last_device_error() == fa.FA_OK  # a clean word to start from
    fa.fa_set_wait_timeout_ns(1)
    try:
        fn()
        word = fa.fa_device_error_word()
        st = fa.fa_last_device_error()  # synchronises, reads and clears the word
    finally:
        fa.fa_set_wait_timeout_ns(0)  # back to the default bound
    return st, word


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 4096, 64, False), (1, 2, 4096, 128, False),
    # more work items than SMs: the persistent kernels, at d = 64 the
    # forward that stages O through its second Q buffers, at d = 128 the
    # backward with three Q slots and one dO slot, and (causal, 19 heads of 16
    # units: two full waves on 152 SMs) both backward kernels walking units
    # of two key tiles
    (8, 20, 1024, 64, False), (8, 20, 1024, 128, False),
    (1, 19, 4096, 64, True), (1, 19, 4096, 128, True)])
def test_wait_bound_runs_out_then_a_normal_call_succeeds(B, H, N, d, causal):
    # long enough that the pipelines' producers wait for free slots (a wait
    # that ends within one poll of the barrier cannot run out)
    w = W.Workload("timeout", B, H, N, d, causal=causal, seed=40 + d + N)
    cpu = W.make_inputs(w)
    q, k, v, dO = (t.cuda() for t in cpu)

    # forward
    st, word = gives_up(lambda: fa.forward(q, k, v, w.scale, causal))
    assert st == fa.FA_ERR_TIMEOUT, (st, hex(word))
    assert word & 0xFF == 4  # the timeout code, then the site and the block index

    # backward, on a forward computed with the normal bound
    o, lse = fa.forward(q, k, v, w.scale, causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    st, word = gives_up(lambda: fa.backward(q, k, v, o, lse, dO, w.scale, causal))
    assert st == fa.FA_ERR_TIMEOUT, (st, hex(word))

    # the device is still usable: a normal forward and backward match the oracle
    out = run_gpu(*cpu, w.scale, causal)
    check_heads(*cpu, out, w.scale, causal, [(0, 0), (0, 1)])
    assert fa.fa_last_device_error() == fa.FA_OK
