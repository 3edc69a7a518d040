"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small shapes are compared in full (several tiles, ragged tails, degenerate
sizes); the full-size workloads are run in the launch configuration the
benchmark times and compared on seeded heads (full fwd + bwd), on sampled
rows, and on exact gradient identities over every head.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from io_aware_exact_10_gb300 import workloads as W
from parity import (check_bwd_rows, check_heads, check_invariants, check_rows, f64, run_gpu,
                    seeded_heads)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_single_head_config():
    """B=1, H=1, N=128, d=64, non-causal: every output compared."""
    w = W.SINGLE_HEAD
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, w.causal)
    check_heads(q, k, v, dO, out, w.scale, w.causal, [(0, 0)])


SMALL = [
    # B, H, N, d, causal
    (1, 2, 256, 64, False), (1, 2, 256, 64, True),
    (2, 3, 384, 128, False), (2, 3, 384, 128, True),
    (1, 2, 512, 128, True), (2, 1, 640, 64, False),
    (1, 1, 200, 64, False), (1, 1, 200, 128, True),     # ragged tail
    (1, 2, 1000, 64, True), (1, 1, 1000, 128, False),   # several tiles + tail
    (1, 1, 64, 128, False), (1, 2, 100, 64, True),      # shorter than one tile
    (1, 1, 1, 64, False), (1, 1, 1, 128, True),          # one row
    (1, 1, 129, 64, True), (1, 1, 255, 128, False),     # one past / one short of a tile
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_small_shapes(B, H, N, d, causal):
    w = W.Workload("small", B, H, N, d, causal=causal, seed=N + d)
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, causal)
    heads = [(b, h) for b in range(B) for h in range(H)]
    check_heads(q, k, v, dO, out, w.scale, causal, heads)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_persistent_staged_ragged(causal, d):
    """More query-tile pairs than SMs and short heads (persistent launches;
    at d = 64 the CTAs stage O through shared memory for every item but
    their last) and a ragged last tile whose last three warps hold no row
    (N = 900 = 7 * 128 + 4): six seeded heads in full, identities on all 160."""
    w = W.Workload("persistent_staged", 8, 20, 900, d, causal=causal, seed=77 + d)
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, causal)
    check_heads(q, k, v, dO, out, w.scale, causal, seeded_heads(w.B, w.H, 6, seed=8))
    check_invariants(dO, out)


def test_nonstandard_scale():
    """scale is an argument, not fixed to 1/sqrt(d)."""
    q, k, v, dO = W.make_inputs(W.Workload("s", 1, 2, 384, 64, causal=True, seed=3))
    for scale in (0.03, 0.4):
        out = run_gpu(q, k, v, dO, scale, True)
        check_heads(q, k, v, dO, out, scale, True, [(0, 0), (0, 1)])


def test_forward_deterministic_and_fully_written():
    """The forward has no atomics: two runs agree bit for bit; outputs that
    start as NaN are fully overwritten; guard bands around them are intact."""
    w = W.Workload("det", 2, 2, 384, 128, causal=True, seed=11)
    q, k, v = W.make_inputs(w, with_grad=False)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    B, H, N, d = q.shape
    n = B * H * N * d
    pad = 4096
    obuf = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    obuf[:pad] = 7.0
    obuf[-pad:] = 7.0
    lbuf = torch.full((B * H * N + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    lbuf[:pad] = 7.0
    lbuf[-pad:] = 7.0
    o = obuf[pad:pad + n].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    fa.fa_fwd(qd, kd, vd, o, lse, B, H, N, d, w.scale, 1)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert (obuf[:pad] == 7.0).all() and (obuf[-pad:] == 7.0).all()
    assert (lbuf[:pad] == 7.0).all() and (lbuf[-pad:] == 7.0).all()
    o2, lse2 = fa.forward(qd, kd, vd, w.scale, True)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_backward_outputs_fully_written():
    """dq/dk/dv that start as NaN are fully overwritten, guard bands intact."""
    w = W.Workload("bw", 1, 2, 200, 64, causal=False, seed=5)
    q, k, v, dO = (t.cuda() for t in W.make_inputs(w))
    o, lse = fa.forward(q, k, v, w.scale, False)
    B, H, N, d = q.shape
    n, pad = B * H * N * d, 2048
    bufs = []
    for _ in range(3):
        b = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
        b[:pad] = 3.0
        b[-pad:] = 3.0
        bufs.append(b)
    dq, dk, dv = (b[pad:pad + n].view(B, H, N, d) for b in bufs)
    ws = torch.full((fa.fa_bwd_workspace_size(B, H, N, d),), 255, dtype=torch.uint8, device="cuda")
    fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, w.scale, 0, ws, ws.numel())
    torch.cuda.synchronize()
    for b, t in zip(bufs, (dq, dk, dv)):
        assert torch.isfinite(t).all()
        assert (b[:pad] == 3.0).all() and (b[-pad:] == 3.0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_gpt2_medium(causal):
    """B=64, H=16, N=1024, d=64 (the GPT-2-medium attention shape): 6 seeded
    heads in full, 64 rows on 24 more heads, identities on all 1024 heads."""
    w = W.GPT2_MEDIUM_CAUSAL if causal else W.GPT2_MEDIUM
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, causal)
    check_heads(q, k, v, dO, out, w.scale, causal, seeded_heads(w.B, w.H, 6, seed=1))
    rows = np.random.default_rng(2).choice(w.N, 64, replace=False)
    check_rows(q, k, v, out, w.scale, causal, seeded_heads(w.B, w.H, 24, seed=3), rows)
    check_invariants(dO, out)


def test_long_causal():
    """B=4, H=32, N=8192, d=128, causal: 1 head in full (fwd + bwd), 64 rows on
    6 more heads, identities on all heads."""
    w = W.LONG_CAUSAL
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, True)
    check_heads(q, k, v, dO, out, w.scale, True, seeded_heads(w.B, w.H, 1, seed=4))
    rows = np.concatenate([[0, 1, 127, 128, 8191], np.random.default_rng(5).choice(8192, 59, replace=False)])
    check_rows(q, k, v, out, w.scale, True, seeded_heads(w.B, w.H, 6, seed=6), rows)
    check_invariants(dO, out)


@pytest.mark.parametrize("causal", [True, False])
def test_stress(causal):
    """Q, K ~ N(0, 4^2), every 97th key row x8: LSE reaches O(100); 2 heads in
    full, and the rows right after each boosted key on 4 more heads."""
    w = W.STRESS_CAUSAL if causal else W.STRESS
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, causal)
    check_heads(q, k, v, dO, out, w.scale, causal, seeded_heads(w.B, w.H, 2, seed=7))
    boosted = np.arange(96, w.N, 97)
    rows = np.unique(np.clip(np.concatenate([boosted, boosted + 1]), 0, w.N - 1))[:96]
    check_rows(q, k, v, out, w.scale, causal, seeded_heads(w.B, w.H, 4, seed=8), rows)
    check_invariants(dO, out)


def sampled_rows(N, n, seed):
    """n distinct rows of [0, N): the first and last rows of the first two
    tiles and of the sequence, the middle one, and seeded random rows."""
    fixed = [r for r in (0, 1, 127, 128, N // 2, N - 2, N - 1) if 0 <= r < N]
    rest = np.setdiff1d(np.arange(N), fixed)
    pick = np.random.default_rng(seed).choice(rest, n - len(fixed), replace=False)
    return np.sort(np.concatenate([fixed, pick])).astype(np.int64)


@pytest.mark.parametrize("d", W.SWEEP_D)
@pytest.mark.parametrize("N", W.SWEEP_N)
def test_sweep(N, d):
    """Sequence-length sweep (H=16, B*N=65536, causal): one head in full,
    forward and backward, up to N=8192; beyond that, on one head, dq on 48
    query rows and dk, dv on 48 key rows (the key rows include the first
    tile's, whose sums run over every query).  O and LSE on 48 rows of two
    more heads, and the gradient identities on every head."""
    w = W.sweep(N, d)
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, True)
    head = seeded_heads(w.B, w.H, 1, seed=N)
    if N <= 8192:
        check_heads(q, k, v, dO, out, w.scale, True, head)
    else:
        check_bwd_rows(q, k, v, dO, out, w.scale, True, head, sampled_rows(N, 48, N + 2),
                       sampled_rows(N, 48, N + 3))
    rows = np.concatenate([[0, N - 1], np.random.default_rng(N).choice(N, 46, replace=False)])
    check_rows(q, k, v, out, w.scale, True, seeded_heads(w.B, w.H, 2, seed=N + 1), rows)
    check_invariants(dO, out)


@pytest.mark.parametrize("B,H,N,d", [(2, 2, 1024, 64), (1, 2, 512, 128)])
def test_one_query_tile_per_cta_matches_two(B, H, N, d):
    """The tile-size sweep's Br = 128 layout (every 128-row query tile its own
    query head of the same key/value head, non-causal) computes each row as
    the standard Br = 256 layout does: o and lse bit for bit."""
    g = torch.Generator().manual_seed(N + d)
    q, k, v = (torch.randn((B, H, N, d), generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    scale = d ** -0.5
    o, lse = fa.forward(q, k, v, scale, False)
    nt = N // 128
    o1, lse1 = torch.empty_like(q), torch.empty((B, H, N), device="cuda")
    fa.fa_fwd_ex(q, k, v, o1, lse1, B, H * nt, H, 128, N, d, scale, 0)
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(lse, lse1)


@pytest.mark.parametrize("d", [64, 128])
def test_longest_sequence(d):
    """B=1, H=2, N=131072, causal: 1024 key tiles per head (launches of one
    CTA per tile; dK and dV of the first key tiles accumulate over 131072
    queries).  On one head: O, LSE and dq on 48 query rows spread over the
    sequence, dk and dv on 48 key rows among the last 1024 (the oracle's
    statistics are then needed for those rows only); gradient identities on
    both heads."""
    N = 131072
    w = W.Workload(f"longest_N{N}_d{d}", 1, 2, N, d, causal=True, seed=d + 1)
    q, k, v, dO = W.make_inputs(w)
    out = run_gpu(q, k, v, dO, w.scale, True)
    rows = sampled_rows(N, 48, 11)
    check_rows(q, k, v, out, w.scale, True, [(0, 1)], rows)
    krows = np.sort(N - 1024 + np.random.default_rng(12).choice(1024, 48, replace=False))
    check_bwd_rows(q, k, v, dO, out, w.scale, True, [(0, 1)], rows, krows)
    check_invariants(dO, out)
