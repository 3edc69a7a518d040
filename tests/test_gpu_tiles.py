"""GPU parity of the forward with 64-key tiles (fa_fwd_tiled, key_tile = 64).

The 64-key forward streams K and V in tiles of 64 keys and keeps its own
tensor-memory plan (S of 64 columns per query tile); the arithmetic per key
is that of the 128-key forward, the online softmax only groups the keys
differently.  Compared with the fp64 oracle element by element on small
shapes (several tiles, ragged tails, one row, causal and not, N_q != N_k,
grouped key/value heads) and on seeded heads of a larger causal problem; the
backward takes its o and lse like those of the 128-key forward.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_10_gb300 as fa
import oracle
from parity import TOL_LSE, TOL_O, check_groups, f64, gqa_inputs, record

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def fwd64(q, k, v, scale, causal):
    B, H, Nq, d = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa.fa_fwd_tiled(q, k, v, o, lse, B, H, H_kv, Nq, Nk, d, scale, int(causal), 64)
    return o, lse


SHAPES = [
    # B, H, H_kv, N_q, N_k, d, causal
    (1, 2, 2, 256, 256, 64, False), (1, 2, 2, 256, 256, 64, True),
    (1, 2, 2, 384, 384, 128, False), (1, 2, 2, 384, 384, 128, True),
    (1, 1, 1, 200, 200, 64, True), (1, 1, 1, 1000, 1000, 128, True),     # ragged tails
    (1, 1, 1, 1, 1, 64, False), (1, 1, 1, 63, 63, 128, True),            # shorter than a tile
    (1, 1, 1, 65, 65, 64, True), (1, 1, 1, 129, 129, 128, False),        # one past a tile
    (2, 4, 2, 300, 1000, 128, True), (1, 4, 1, 1000, 260, 64, False),    # N_q != N_k, GQA, MQA
]


@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,d,causal", SHAPES)
def test_key_tile_64_matches_the_oracle(B, H, H_kv, Nq, Nk, d, causal):
    q, k, v, dO = gqa_inputs(B, H, H_kv, Nq, d, seed=Nq + Nk + d, N_k=Nk)
    scale = d ** -0.5
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = fwd64(qd, kd, vd, scale, causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale, causal)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    out = {n: t.cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    check_groups(q, k, v, dO, out, scale, causal, [(b, hk) for b in range(B) for hk in range(H_kv)])


def test_key_tile_64_long_causal_heads():
    """B=2, H=8, N=4096, d=128, causal: two heads in full against the oracle;
    every head within rounding of the 128-key forward."""
    B, H, N, d = 2, 8, 4096, 128
    q, k, v, _ = gqa_inputs(B, H, H, N, d, seed=77)
    scale = d ** -0.5
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o64, lse64 = fwd64(qd, kd, vd, scale, True)
    o128, lse128 = fa.forward(qd, kd, vd, scale, True)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    d_o = (o64.float() - o128.float()).abs().max().item()
    d_l = (lse64 - lse128).abs().max().item()
    assert d_o <= TOL_O and d_l <= TOL_LSE, (d_o, d_l)
    record("o max-abs, 64 vs 128 keys per tile", d_o, TOL_O)
    record("lse max-abs, 64 vs 128 keys per tile", d_l, TOL_LSE)
    wo = wl = 0.0
    for b, h in ((0, 3), (1, 6)):
        o_ref, lse_ref = oracle.attn_fwd(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), scale, True)
        eo = float(np.abs(f64(o64[b, h]) - o_ref).max())
        el = float(np.abs(f64(lse64[b, h]) - lse_ref).max())
        assert eo <= TOL_O and el <= TOL_LSE, (b, h, eo, el)
        wo, wl = max(wo, eo), max(wl, el)
    record("o max-abs", wo, TOL_O, heads=2)
    record("lse max-abs", wl, TOL_LSE, heads=2)


def test_key_tile_other_values_are_refused():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), device="cuda")
    for kt in (32, 96, 256, 0):
        st = fa.fa_fwd_tiled(q, q, q, o, lse, 1, 1, 1, 128, 128, 64, 0.125, 0, kt, check=False)
        assert st == fa.FA_ERR_UNSUPPORTED
