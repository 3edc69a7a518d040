"""Query and key lengths that differ (N_q != N_k): GPU path against the fp64
oracle, through fa_fwd_ex / fa_bwd_ex.

Causal masking aligns the last query row with the last key: query i sees key
j iff j <= i + N_k - N_q.  The shapes put that boundary on and off the
128-row tiles, make either length ragged, and cover a single query row (one
decoding step), a single key, more queries than keys (unmasked only) and
grouped key/value heads.  Tolerances as in parity.py.
"""
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from parity import check_groups, gqa_inputs, run_gpu

pytestmark = pytest.mark.gpu

CROSS_SHAPES = [
    # B, H, H_kv, N_q, N_k, d, causal
    (1, 2, 2, 128, 384, 64, True), (1, 2, 1, 100, 333, 128, True),    # offset on / off a tile
    (2, 4, 2, 257, 1000, 64, True), (1, 2, 2, 129, 4096, 128, True),  # several tiles; long keys
    (1, 2, 2, 255, 256, 64, True), (1, 2, 2, 127, 255, 128, True),    # offsets 1 and 128
    (1, 2, 2, 1, 777, 128, True), (1, 2, 2, 1, 777, 64, False),       # one query row
    (1, 2, 2, 384, 128, 64, False), (1, 3, 3, 200, 50, 128, False),   # more queries than keys
    (1, 4, 2, 640, 130, 128, False), (1, 2, 2, 300, 1, 64, False),    # ... ; a single key
    (1, 2, 2, 1, 1, 128, True), (1, 2, 2, 513, 513, 64, True),        # equal lengths
]


@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,d,causal", CROSS_SHAPES)
def test_cross_shapes(B, H, H_kv, Nq, Nk, d, causal):
    q, k, v, dO = gqa_inputs(B, H, H_kv, Nq, d, seed=Nq + 3 * Nk + d, N_k=Nk)
    scale = d ** -0.5
    out = run_gpu(q, k, v, dO, scale, causal)
    assert out["o"].shape == q.shape and out["lse"].shape == q.shape[:-1]
    assert out["dk"].shape == k.shape and out["dv"].shape == v.shape
    check_groups(q, k, v, dO, out, scale, causal, [(b, hk) for b in range(B) for hk in range(H_kv)])


def test_cross_chunked_prefill_sampled():
    """A chunk of 1024 new queries after 7168 cached positions (N_k = 8192),
    32 query heads on 8 key/value heads, d = 128, causal: one key/value group
    in full, and on every head the identities sum_j dk_j = 0 and sum_j dv_j =
    the sum of dO over the group's query rows."""
    B, H, H_kv, Nq, Nk, d = 1, 32, 8, 1024, 8192, 128
    q, k, v, dO = gqa_inputs(B, H, H_kv, Nq, d, seed=91, N_k=Nk)
    scale = d ** -0.5
    out = run_gpu(q, k, v, dO, scale, True)
    check_groups(q, k, v, dO, out, scale, True, [(0, 3)])
    G = H // H_kv
    dk, dv = out["dk"].double(), out["dv"].double()
    sdo = dO.double().sum(dim=2).reshape(B, H_kv, G, d).sum(dim=2)
    fro = lambda t: t.pow(2).sum(dim=(-1, -2)).sqrt().clamp_min(1e-12)
    err_v = ((dv.sum(dim=2) - sdo).norm(dim=-1) / fro(dv)).max().item()
    err_k = (dk.sum(dim=2).norm(dim=-1) / fro(dk)).max().item()
    assert err_v <= 3e-2 and err_k <= 3e-2, (err_v, err_k)


def test_cross_no_query_rows_zeroes_key_gradients():
    """N_q = 0: the forward does nothing; the backward sets dk, dv to zero."""
    B, H, H_kv, Nk, d = 1, 4, 2, 300, 64
    dev = "cuda"
    q = torch.empty((B, H, 0, d), dtype=torch.bfloat16, device=dev)
    k = torch.randn((B, H_kv, Nk, d), device=dev).to(torch.bfloat16)
    v = torch.randn((B, H_kv, Nk, d), device=dev).to(torch.bfloat16)
    o, lse = fa.forward(q, k, v, causal=True)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    fa.fa_bwd_ex(q, k, v, o, lse, q, q, dk, dv, B, H, H_kv, 0, Nk, d, d ** -0.5, 1, ws, 256)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    assert o.shape == q.shape and lse.shape == (B, H, 0)
    assert torch.count_nonzero(dk).item() == 0 and torch.count_nonzero(dv).item() == 0
