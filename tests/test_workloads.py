"""Host-side checks of the seeded workloads and their FLOP accounting (CPU)."""
import numpy as np
import pytest
import torch

from io_aware_exact_10_gb300 import workloads as W


def visible_pairs(Nq, Nk, causal):
    """Brute-force count of (query, key) pairs under the causal rule that
    aligns the last query with the last key."""
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    return int((j <= i + (Nk - Nq)).sum()) if causal else Nq * Nk


@pytest.mark.parametrize("Nq,Nk,causal", [(8, 8, True), (8, 8, False), (5, 17, True),
                                          (17, 5, False), (1, 9, True), (64, 1000, True)])
def test_fwd_flops_counts_visible_pairs(Nq, Nk, causal):
    """fwd = 4*B*H*d per pair; causal counts N^2/2 for the square part (the
    convention of the square workloads), i.e. the exact count less Nq/2."""
    w = W.Workload("t", 2, 3, Nq, 16, causal=causal, N_k=Nk)
    pairs = visible_pairs(Nq, Nk, causal) - (Nq / 2 if causal else 0)
    assert w.fwd_flops() == pytest.approx(4 * 2 * 3 * 16 * pairs)
    assert w.bwd_flops() == pytest.approx(2.5 * w.fwd_flops())


def test_inputs_follow_shapes_and_seed():
    w = W.Workload("t", 1, 4, 3, 8, causal=True, H_kv=2, N_k=5, seed=4)
    q, k, v, dO = W.make_inputs(w)
    assert q.shape == dO.shape == (1, 4, 3, 8) and k.shape == v.shape == (1, 2, 5, 8)
    assert all(t.dtype == torch.bfloat16 for t in (q, k, v, dO))
    again = W.make_inputs(w)
    assert all(torch.equal(a, b) for a, b in zip((q, k, v, dO), again))
    # with N_k = N and H_kv = H the draw is the square workload's
    sq = W.make_inputs(W.Workload("t", 1, 2, 6, 8, causal=False, seed=1))
    ex = W.make_inputs(W.Workload("t", 1, 2, 6, 8, causal=False, seed=1, H_kv=2, N_k=6))
    assert all(torch.equal(a, b) for a, b in zip(sq, ex))


def test_named_workloads():
    p = W.WORKLOADS["prefill_chunk"]
    assert (p.N, p.kv_len, p.H, p.kv_heads, p.d, p.causal) == (1024, 8192, 32, 8, 128, True)
    assert W.WORKLOADS["gqa_causal"].kv_len == 4096


@pytest.mark.parametrize("Nq,Nk,causal", [(300, 300, False), (300, 300, True), (130, 700, True),
                                          (700, 130, False)])
def test_visible_pairs_brute_force(Nq, Nk, causal):
    """The block-sparse pair count equals a count over the expanded element mask."""
    g = torch.Generator().manual_seed(Nq + Nk)
    bm = (torch.rand(((Nq + 127) // 128, (Nk + 127) // 128), generator=g) < 0.5).to(torch.uint8)
    elem = torch.kron(bm, torch.ones(128, 128, dtype=torch.uint8))[:Nq, :Nk].bool()
    if causal:
        elem &= torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    assert W.visible_pairs(bm.numpy(), Nq, Nk, causal) == int(elem.sum())


def test_block_pattern():
    w = W.Workload("t", 1, 1, 128 * 40 + 5, 64, causal=False, block_pattern="local2_global1_random0.1",
                   seed=3)
    m = W.block_mask(w)
    assert m.shape == (41, 41) and m.dtype.name == "uint8"
    i, j = np.meshgrid(np.arange(41), np.arange(41), indexing="ij")
    assert m[np.abs(i - j) <= 2].all() and m[0].all() and m[:, 0].all()
    off = (np.abs(i - j) > 2) & (i > 0) & (j > 0)
    assert 0.03 < m[off].mean() < 0.2  # the random blocks
    assert np.array_equal(m, W.block_mask(w))  # seeded
    with pytest.raises(ValueError):
        W.block_mask(W.Workload("t", 1, 1, 128, 64, causal=False, block_pattern="butterfly"))
