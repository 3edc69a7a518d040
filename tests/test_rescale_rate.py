"""How often the forward's lazy rescale of O runs (CPU only).

The forward keeps one running maximum m per query row (log2 units) and
adopts a new one only when a key tile's maximum exceeds it by more than
tau = 8; only then is the unnormalised O of the row rescaled in tensor
memory, and the warp that holds the row (32 consecutive rows of a 128-row
query tile) runs the rescale loop when any of its rows needs it.  The first
tile of a row sets m without a rescale (O is still empty).

This computes, for one head of the measured workloads, the fraction of
(warp, key tile) steps that run the rescale loop, from the same bf16 inputs
and the same rule, with fp32 scores: it is the evidence that the rescale
can stay inline in the softmax warps (no separate correction warps) for
inputs like these, and that the stress workload does exercise it.
"""
import math

import pytest
import torch

from io_aware_exact_10_gb300 import workloads as W

TAU = 8.0
BM = BN = 128


def rescale_fraction(w, head=(0, 0)):
    """(fraction of warp steps with a rescale, fraction of row steps with
    one) over one head of w, rows processed in 128-key tiles."""
    q, k, _ = W.make_inputs(w, with_grad=False)
    b, h = head
    s = (q[b, h].float() @ k[b, h].float().T) * (w.scale / math.log(2.0))  # log2 units
    N, Nk = s.shape
    if w.causal:
        off = Nk - N
        keep = torch.ones(N, Nk, dtype=torch.bool).tril(diagonal=off)
        s = s.masked_fill(~keep, float("-inf"))
    nt = -(-Nk // BN)
    tile_max = torch.stack([s[:, j * BN:(j + 1) * BN].max(dim=1).values for j in range(nt)], 1)
    m = torch.full((N,), float("-inf"))
    row_steps = row_rescales = warp_steps = warp_rescales = 0
    for j in range(nt):
        tm = tile_max[:, j]
        active = tm > float("-inf")  # the row sees a key of this tile (causal bound)
        need = active & (tm > m + TAU)
        rescale = need & (m > float("-inf"))  # not the row's first tile
        m = torch.where(need, tm, m)
        row_steps += int(active.sum())
        row_rescales += int(rescale.sum())
        # a warp steps through tile j when any of its rows sees it
        a = active.view(-1, 32).any(dim=1) if N % 32 == 0 else None
        r = rescale.view(-1, 32).any(dim=1) if N % 32 == 0 else None
        warp_steps += int(a.sum())
        warp_rescales += int(r.sum())
    return warp_rescales / warp_steps, row_rescales / row_steps


@pytest.mark.parametrize("w,bound", [(W.LONG_CAUSAL, 1e-3), (W.GPT2_MEDIUM, 1e-3),
                                     (W.GPT2_MEDIUM_CAUSAL, 1e-3), (W.sweep(32768, 128), 1e-3)])
def test_rescale_is_rare_on_normal_inputs(w, bound):
    fw, fr = rescale_fraction(w)
    print(f"{w.name}: rescale in {100 * fw:.4f} % of warp steps, {100 * fr:.5f} % of row steps")
    assert fw <= bound


def test_stress_inputs_exercise_the_rescale():
    fw, fr = rescale_fraction(W.STRESS_CAUSAL)
    print(f"{W.STRESS_CAUSAL.name}: rescale in {100 * fw:.3f} % of warp steps, "
          f"{100 * fr:.4f} % of row steps")
    assert fw > 0.01
