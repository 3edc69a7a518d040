"""Block-sparse attention: GPU path (fa_fwd_sparse / fa_bwd_sparse) against
the fp64 oracle with the same block mask.

The mask keeps or drops 128 x 128 blocks of (query rows, keys), on top of the
causal rule.  Rows that see no key must come out as o = 0, lse = -inf with
zero gradients; keys that no row sees get dk = dv = 0.  Tolerances as in
parity.py; -inf entries of the LSE must match exactly.
"""
import numpy as np
import pytest
import torch

import io_aware_exact_10_gb300 as fa
import oracle
from parity import TOL_GRAD, TOL_LSE, TOL_O, f64, gqa_inputs, record, rel_fro

pytestmark = pytest.mark.gpu


def run_sparse(q, k, v, dO, scale, causal, bm):
    dev = "cuda"
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    mask = torch.from_numpy(bm).to(dev)
    o, lse = fa.forward(qd, kd, vd, scale, causal, block_mask=mask)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale, causal, block_mask=mask)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    return {n: t.cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}


def check_sparse(q, k, v, dO, out, scale, causal, bm):
    """Every key/value group of every batch against the oracle."""
    B, H, Nq, d = q.shape
    H_kv = k.shape[1]
    G = H // H_kv
    worst = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    for b in range(B):
        for hk in range(H_kv):
            hs = slice(hk * G, hk * G + G)
            qg, dOg = f64(q[b, hs]), f64(dO[b, hs])
            kg, vg = f64(k[b, hk:hk + 1]), f64(v[b, hk:hk + 1])
            o_ref, lse_ref = oracle.attn_fwd(qg, kg, vg, scale, causal, block_mask=bm)
            o_g, lse_g = f64(out["o"][b, hs]), f64(out["lse"][b, hs])
            assert np.all(np.isfinite(o_g)), "non-finite O"
            eo = float(np.abs(o_g - o_ref).max())
            assert eo <= TOL_O, f"O max-abs {eo} at {(b, hk)}"
            worst["o"] = max(worst["o"], eo)
            empty = np.isneginf(lse_ref)
            assert np.array_equal(np.isneginf(lse_g), empty), f"-inf LSE rows differ at {(b, hk)}"
            if (~empty).any():
                el = float(np.abs(lse_g[~empty] - lse_ref[~empty]).max())
                assert el <= TOL_LSE, f"LSE max-abs {el} at {(b, hk)}"
                worst["lse"] = max(worst["lse"], el)
            refs = oracle.attn_bwd(qg, kg, vg, dOg, scale, causal, block_mask=bm)
            for g in range(G):
                e = rel_fro(f64(out["dq"][b, hk * G + g]), refs[0][g])
                assert e <= TOL_GRAD, f"dq rel-Frobenius {e} at query head {(b, hk * G + g)}"
                worst["dq"] = max(worst["dq"], e)
            for name, r in (("dk", refs[1][0]), ("dv", refs[2][0])):
                gv = f64(out[name][b, hk])
                assert np.all(np.isfinite(gv)), f"non-finite {name}"
                e = rel_fro(gv, r)
                assert e <= TOL_GRAD, f"{name} rel-Frobenius {e} at {(b, hk)}"
                worst[name] = max(worst[name], e)
    record("o max-abs", worst["o"], TOL_O)
    record("lse max-abs", worst["lse"], TOL_LSE)
    for name in ("dq", "dk", "dv"):
        record(f"{name} rel-Frobenius", worst[name], TOL_GRAD)


def random_mask(Nq, Nk, density, seed, keep_col0=True):
    g = np.random.default_rng(seed)
    bm = (g.random(((Nq + 127) // 128, (Nk + 127) // 128)) < density).astype(np.uint8)
    if keep_col0:
        bm[:, 0] = 1
    return bm


SPARSE_SHAPES = [
    # B, H, H_kv, N_q, N_k, d, causal, density
    (1, 2, 2, 640, 640, 64, False, 0.5), (1, 2, 2, 640, 640, 128, False, 0.5),
    (1, 2, 2, 700, 700, 64, True, 0.6), (1, 2, 2, 700, 700, 128, True, 0.6),   # ragged, causal
    (2, 4, 2, 300, 1000, 64, True, 0.5), (1, 4, 1, 1000, 260, 128, False, 0.4),  # GQA / MQA, N_q != N_k
    (1, 2, 2, 1024, 1024, 128, True, 0.25),
]


@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,d,causal,density", SPARSE_SHAPES)
def test_sparse_random_masks(B, H, H_kv, Nq, Nk, d, causal, density):
    q, k, v, dO = gqa_inputs(B, H, H_kv, Nq, d, seed=Nq + Nk + d + int(causal), N_k=Nk)
    bm = random_mask(Nq, Nk, density, seed=Nq * 7 + Nk)
    scale = d ** -0.5
    out = run_sparse(q, k, v, dO, scale, causal, bm)
    check_sparse(q, k, v, dO, out, scale, causal, bm)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_sparse_empty_tiles(d, causal):
    """Dropped query tiles (whole rows of the mask), dropped key tiles (whole
    columns) and a pair of query tiles of which one keeps nothing."""
    N = 5 * 128 + 17
    bm = random_mask(N, N, 0.6, seed=3 + d)
    bm[1, :] = 0          # query tile 1 keeps nothing: o = 0, lse = -inf
    bm[4, :] = 0          # ... and tile 4, paired with a busy tile 5
    bm[:, 3] = 0          # key tile 3: dk = dv = 0
    q, k, v, dO = gqa_inputs(1, 2, 2, N, d, seed=11 + d)
    scale = d ** -0.5
    out = run_sparse(q, k, v, dO, scale, causal, bm)
    assert torch.count_nonzero(out["o"][:, :, 128:256]).item() == 0
    assert torch.isneginf(out["lse"][:, :, 128:256]).all()
    assert torch.count_nonzero(out["dq"][:, :, 128:256]).item() == 0
    assert torch.count_nonzero(out["dk"][:, :, 384:512]).item() == 0
    assert torch.count_nonzero(out["dv"][:, :, 384:512]).item() == 0
    check_sparse(q, k, v, dO, out, scale, causal, bm)


@pytest.mark.parametrize("d", [64, 128])
def test_sparse_rows_empty_inside_kept_tile(d):
    """Causal with N_k - N_q = 72 and only key tile 1 kept: rows i < 56 see
    keys <= i + 72 < 128, all dropped, although their tile computes."""
    Nq, Nk = 128, 200
    bm = np.array([[0, 1]], dtype=np.uint8)
    q, k, v, dO = gqa_inputs(1, 2, 2, Nq, d, seed=21 + d, N_k=Nk)
    scale = d ** -0.5
    out = run_sparse(q, k, v, dO, scale, True, bm)
    assert torch.isneginf(out["lse"][:, :, :56]).all() and torch.isfinite(out["lse"][:, :, 56:]).all()
    check_sparse(q, k, v, dO, out, scale, True, bm)


@pytest.mark.parametrize("d", [64, 128])
def test_sparse_all_kept_equals_dense(d):
    """An all-ones mask gives the dense result: O, LSE, dK and dV bit for bit
    (one CTA computes each, in the same order); dQ is summed by several
    key-tile CTAs whose fp32 reduce-adds land in run-dependent order, so it
    agrees to rounding."""
    B, H, N = 1, 2, 384
    q, k, v, dO = (t.cuda() for t in gqa_inputs(B, H, H, N, d, seed=5))
    ones = torch.ones((3, 3), dtype=torch.uint8, device="cuda")
    for causal in (False, True):
        a = fa.forward(q, k, v, causal=causal)
        b = fa.forward(q, k, v, causal=causal, block_mask=ones)
        ga = fa.backward(q, k, v, *a, dO, causal=causal)
        gb = fa.backward(q, k, v, *b, dO, causal=causal, block_mask=ones)
        torch.cuda.synchronize()
        for name, x, y in zip(("o", "lse", "dq", "dk", "dv"), a + ga, b + gb):
            if name == "dq":
                e = rel_fro(f64(x), f64(y))
                assert e <= 1e-3, (name, causal, e)
            else:
                assert torch.equal(x, y), (name, causal)


def test_sparse_local_window_long():
    """A banded (local) mask with a global first block column at N = 8192,
    d = 128, causal: two heads against the oracle."""
    N, d = 8192, 128
    nb = N // 128
    i, j = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    bm = ((np.abs(i - j) <= 2) | (j == 0)).astype(np.uint8)
    q, k, v, dO = gqa_inputs(1, 2, 2, N, d, seed=31)
    scale = d ** -0.5
    out = run_sparse(q, k, v, dO, scale, True, bm)
    check_sparse(q, k, v, dO, out, scale, True, bm)
