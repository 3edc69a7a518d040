"""The allocation-free backward entry point (fa_bwd_noalloc).

Callers that cannot allocate device memory (a plugin whose host framework
owns all GPU memory, a loop that must not call cudaMalloc) use this entry
point instead of fa_bwd; its scratch is a fixed array inside the library.
These tests call it through the C ABI and check that it gives the same
gradients as fa_bwd with a caller workspace, on two calls in a row with
different problems (so nothing left in the shared array by the first call
leaks into the second), and that it refuses problems that do not fit.

The file is named to be collected last: if it fails, a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from io_aware_exact_10_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_GRAD = 3e-2  # the relative Frobenius bound every gradient test uses


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def rel_fro(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def one_call(w):
    q, k, v, dO = (t.cuda() for t in W.make_inputs(w))
    o, lse = fa.forward(q, k, v, w.scale, w.causal)
    ref = fa.backward(q, k, v, o, lse, dO, w.scale, w.causal)      # fa_bwd + workspace
    B, H, N, d = q.shape
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    st = fa.fa_bwd_noalloc(q, k, v, o, lse, dO, *got, B, H, N, d, w.scale, int(w.causal))
    torch.cuda.synchronize()
    assert st == fa.FA_OK
    assert fa.fa_last_device_error() == fa.FA_OK
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert torch.isfinite(g).all(), name
        e = rel_fro(g, r)
        assert e <= TOL_GRAD, f"{name}: {e}"


def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    # first call: causal, d=128, ragged N; second call: a different, smaller
    # non-causal d=64 problem that reuses the same static scratch
    one_call(W.Workload("noalloc1", 2, 4, 1000, 128, causal=True, seed=21))
    one_call(W.Workload("noalloc2", 1, 8, 512, 64, causal=False, seed=22))


def test_noalloc_refuses_problems_beyond_its_scratch():
    L = fa.lib()
    A = 0x10000  # aligned placeholder addresses: the size check comes first
    # B*H*N = 262144 rows at d=128 needs ~135 MB of scratch > 64 MiB
    st = L.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, 1, 64, 4096, 128,
                          ctypes.c_float(0.088), 1, None)
    assert st == fa.FA_ERR_INVALID_ARG
    assert fa.fa_bwd_workspace_size(1, 64, 4096, 128) > (64 << 20)
