"""Grouped key/value heads (GQA, MQA): GPU path against the fp64 oracle.

k and v have H_kv heads; query head h attends with key/value head
h // (H // H_kv), and dk, dv of a key/value head sum over its query heads.
Tolerances as in parity.py.
"""
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from parity import check_groups, f64, gqa_inputs, rel_fro, run_gpu

pytestmark = pytest.mark.gpu


GQA_SHAPES = [
    # B, H, H_kv, N, d, causal
    (1, 4, 2, 256, 64, False), (1, 4, 1, 200, 128, True),      # GQA; MQA with a ragged tail
    (2, 6, 2, 384, 64, True), (1, 8, 2, 1000, 128, False),     # several tiles + tail
    (1, 2, 2, 128, 64, True), (2, 4, 4, 129, 128, True),       # one query head per group
    (1, 16, 1, 64, 64, True), (1, 4, 2, 1, 64, False),         # MQA short; a single row
]


@pytest.mark.parametrize("B,H,H_kv,N,d,causal", GQA_SHAPES)
def test_gqa_shapes(B, H, H_kv, N, d, causal):
    q, k, v, dO = gqa_inputs(B, H, H_kv, N, d, seed=N + d + H_kv)
    scale = d ** -0.5
    out = run_gpu(q, k, v, dO, scale, causal)
    assert out["dk"].shape == k.shape and out["dv"].shape == v.shape
    check_groups(q, k, v, dO, out, scale, causal, [(b, hk) for b in range(B) for hk in range(H_kv)])


def test_gqa_with_all_heads_equals_multi_head():
    """H_kv = H through fa_fwd_gqa / fa_bwd_gqa gives fa_fwd / fa_bwd: O, LSE,
    dK, dV bit for bit; dQ (fp32 reduce-adds from several key-tile CTAs, in
    run-dependent order) to rounding."""
    B, H, N, d = 1, 3, 384, 64
    q, k, v, dO = gqa_inputs(B, H, H, N, d, seed=5)
    dev = "cuda"
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    scale = d ** -0.5
    res = []
    for gqa in (False, True):
        o, lse = torch.empty_like(qd), torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
        if gqa:
            fa.fa_fwd_gqa(qd, kd, vd, o, lse, B, H, H, N, d, scale, 1)
            fa.fa_bwd_gqa(qd, kd, vd, o, lse, dOd, dq, dk, dv, B, H, H, N, d, scale, 1, ws, ws.numel())
        else:
            fa.fa_fwd(qd, kd, vd, o, lse, B, H, N, d, scale, 1)
            fa.fa_bwd(qd, kd, vd, o, lse, dOd, dq, dk, dv, B, H, N, d, scale, 1, ws, ws.numel())
        torch.cuda.synchronize()
        res.append([t.cpu() for t in (o, lse, dq, dk, dv)])
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), *res):
        if name == "dq":
            assert rel_fro(f64(a), f64(b)) <= 1e-3, name
        else:
            assert torch.equal(a, b), name


def test_gqa_long_causal_sampled():
    """A grouped-query shape of current decoder models (32 query heads on 8
    key/value heads, d=128, N=4096, causal): two key/value groups in full, and
    the group identities of the gradients on every head (sum_j dk_j = 0;
    sum_j dv_j = the sum of dO over the group's query rows)."""
    B, H, H_kv, N, d = 1, 32, 8, 4096, 128
    q, k, v, dO = gqa_inputs(B, H, H_kv, N, d, seed=77)
    scale = d ** -0.5
    out = run_gpu(q, k, v, dO, scale, True)
    check_groups(q, k, v, dO, out, scale, True, [(0, 0), (0, 5)])
    G = H // H_kv
    dk, dv = out["dk"].double(), out["dv"].double()
    sdo = dO.double().sum(dim=2).reshape(B, H_kv, G, d).sum(dim=2)
    fro = lambda t: t.pow(2).sum(dim=(-1, -2)).sqrt().clamp_min(1e-12)
    err_v = ((dv.sum(dim=2) - sdo).norm(dim=-1) / fro(dv)).max().item()
    err_k = (dk.sum(dim=2).norm(dim=-1) / fro(dk)).max().item()
    assert err_v <= 3e-2 and err_k <= 3e-2, (err_v, err_k)


@pytest.mark.parametrize("causal", [False, True])
def test_persistent_d64_grouped_cross(causal):
    """d = 64 with grouped key/value heads, more queries than fit one tile
    pair and keys that differ in length (N_q = 640, N_k = 1000), on enough
    heads that both main kernels run persistent CTAs over several items: the
    forward staging O through shared memory, the backward copying the next
    item's K and V into tensor memory before the current item ends.  Three
    key/value groups in full."""
    B, H, H_kv, Nq, Nk, d = 8, 16, 4, 640, 1000, 64
    q, k, v, dO = gqa_inputs(B, H, H_kv, Nq, d, seed=88 + causal, N_k=Nk)
    scale = d ** -0.5
    out = run_gpu(q, k, v, dO, scale, causal)
    check_groups(q, k, v, dO, out, scale, causal, [(0, 0), (3, 2), (7, 3)])
