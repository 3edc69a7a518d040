"""Helpers for GPU-vs-oracle parity tests.

Tolerances (fixed by the accuracy contract of the library):
  O: max |gpu - oracle| <= 2e-2          LSE: max |gpu - oracle| <= 1e-3
  dQ, dK, dV: ||gpu - oracle||_F / ||oracle||_F <= 3e-2, per tensor, per head
The oracle runs in fp64 on the same bf16-rounded inputs widened to fp64.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import io_aware_exact_10_gb300 as fa
import oracle

TOL_O = 2e-2
TOL_LSE = 1e-3
TOL_GRAD = 3e-2

# Worst error of every comparison made in this process, for the margin
# report (tests/conftest.py prints it and, when FA_PARITY_REPORT names a
# file, writes it there as JSON lines).
MARGINS: list = []


def record(what: str, err: float, tol: float, **extra) -> None:
    """Note the worst error `err` of one comparison (`what`: the tensor and
    the kind of check) against its tolerance, under the running test's id."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    MARGINS.append({"test": test, "what": what, "err": float(err), "tol": float(tol), **extra})


def f64(t) -> np.ndarray:
    return t.detach().to("cpu").double().numpy()


def run_gpu(q, k, v, dO, scale, causal, bwd=True, dev="cuda"):
    """Run fa_fwd (+ fa_bwd) through the C ABI; returns CPU tensors."""
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, scale, causal)
    out = {"o": o, "lse": lse}
    if bwd:
        dOd = dO.to(dev)
        dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale, causal)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    return {k_: v_.cpu() for k_, v_ in out.items()}


def rel_fro(g: np.ndarray, r: np.ndarray) -> float:
    den = np.linalg.norm(r)
    return float(np.linalg.norm(g - r) / den) if den > 0 else float(np.linalg.norm(g))


def check_heads(q, k, v, dO, out, scale, causal, heads, bwd=True):
    """Full per-head comparison of GPU outputs with the oracle on `heads`
    (a list of (b, h)).  Returns the worst errors seen."""
    worst = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    for b, h in heads:
        qh, kh, vh = f64(q[b, h]), f64(k[b, h]), f64(v[b, h])
        o_ref, lse_ref = oracle.attn_fwd(qh, kh, vh, scale, causal)
        eo = float(np.abs(f64(out["o"][b, h]) - o_ref).max())
        el = float(np.abs(f64(out["lse"][b, h]) - lse_ref).max())
        assert np.isfinite(f64(out["o"][b, h])).all()
        assert eo <= TOL_O, f"O max-abs {eo} at head {(b, h)}"
        assert el <= TOL_LSE, f"LSE max-abs {el} at head {(b, h)}"
        worst["o"] = max(worst["o"], eo)
        worst["lse"] = max(worst["lse"], el)
        if bwd:
            refs = oracle.attn_bwd(qh, kh, vh, f64(dO[b, h]), scale, causal)
            for name, r in zip(("dq", "dk", "dv"), refs):
                e = rel_fro(f64(out[name][b, h]), r)
                assert e <= TOL_GRAD, f"{name} rel-Frobenius {e} at head {(b, h)}"
                worst[name] = max(worst[name], e)
    record("o max-abs", worst["o"], TOL_O, heads=len(heads))
    record("lse max-abs", worst["lse"], TOL_LSE, heads=len(heads))
    if bwd:
        for name in ("dq", "dk", "dv"):
            record(f"{name} rel-Frobenius", worst[name], TOL_GRAD, heads=len(heads))
    return worst


def check_rows(q, k, v, out, scale, causal, heads, rows):
    """O and LSE on selected query rows of selected heads (any size)."""
    wo = wl = 0.0
    for b, h in heads:
        o_r, lse_r = oracle.attn_fwd_rows(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), rows,
                                          scale, causal)
        eo = float(np.abs(f64(out["o"][b, h][rows]) - o_r).max())
        el = float(np.abs(f64(out["lse"][b, h][rows]) - lse_r).max())
        assert eo <= TOL_O, f"O max-abs {eo} at head {(b, h)} rows"
        assert el <= TOL_LSE, f"LSE max-abs {el} at head {(b, h)} rows"
        wo, wl = max(wo, eo), max(wl, el)
    record("o max-abs (rows)", wo, TOL_O, heads=len(heads), rows=len(rows))
    record("lse max-abs (rows)", wl, TOL_LSE, heads=len(heads), rows=len(rows))


def check_bwd_rows(q, k, v, dO, out, scale, causal, heads, qrows, krows):
    """dq on selected query rows and dk, dv on selected key rows of selected
    heads (any size), against the oracle's backward rows entry: relative
    Frobenius error over the selected rows of each tensor, per head."""
    worst = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    for b, h in heads:
        refs = oracle.attn_bwd_rows(f64(q[b, h]), f64(k[b, h]), f64(v[b, h]), f64(dO[b, h]),
                                    qrows, krows, scale, causal)
        for name, rows, r in zip(("dq", "dk", "dv"), (qrows, krows, krows), refs):
            g = f64(out[name][b, h][rows])
            assert np.isfinite(g).all(), f"{name} not finite at head {(b, h)} rows"
            e = rel_fro(g, r)
            assert e <= TOL_GRAD, f"{name} rel-Frobenius {e} at head {(b, h)} rows"
            worst[name] = max(worst[name], e)
    for name in ("dq", "dk", "dv"):
        record(f"{name} rel-Frobenius (rows)", worst[name], TOL_GRAD, heads=len(heads),
               rows=len(qrows if name == "dq" else krows))
    return worst


def check_invariants(dO, out, tol=3e-2):
    """Exact identities of the gradients, on every head: sum_j dv_j =
    sum_i dO_i (rows of P sum to 1) and sum_j dk_j = 0 (softmax ignores a
    common shift of the keys).  A sum of N rounded rows has an error that
    scales with the head's Frobenius norm, so each residual is measured
    against it: ||sum_j dk_j|| / ||dk||_F and ||sum_j dv_j - sum_i dO_i|| /
    ||dv||_F."""
    dv = out["dv"].double()
    dk = out["dk"].double()
    sdo = dO.double().sum(dim=2)
    fro = lambda t: t.pow(2).sum(dim=(-1, -2)).sqrt().clamp_min(1e-12)
    err_v = ((dv.sum(dim=2) - sdo).norm(dim=-1) / fro(dv)).max().item()
    err_k = (dk.sum(dim=2).norm(dim=-1) / fro(dk)).max().item()
    assert err_v <= tol, f"sum dv != sum dO: {err_v}"
    assert err_k <= tol, f"sum dk != 0: {err_k}"
    record("sum_j dv_j - sum_i dO_i (all heads)", err_v, tol)
    record("sum_j dk_j (all heads)", err_k, tol)
    return err_v, err_k


def seeded_heads(B, H, n, seed=0):
    g = np.random.default_rng(seed)
    idx = g.choice(B * H, size=min(n, B * H), replace=False)
    return [(int(i) // H, int(i) % H) for i in sorted(idx)]


def gqa_inputs(B, H, H_kv, N, d, seed, N_k=None):
    """Seeded fp32 N(0,1) draws rounded to bf16: q, k, v, dO in that order
    (k, v with H_kv heads and N_k rows, N_k = N unless given)."""
    N_k = N if N_k is None else N_k
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H_kv, N_k, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H_kv, N_k, d), generator=g).to(torch.bfloat16)
    dO = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    return q, k, v, dO


def check_groups(q, k, v, dO, out, scale, causal, kv_heads):
    """Every query head of each listed key/value head (b, hk), and dk, dv of
    that head, against the oracle run on the group."""
    H, H_kv = q.shape[1], k.shape[1]
    G = H // H_kv
    worst = {"o": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    for b, hk in kv_heads:
        hs = slice(hk * G, hk * G + G)
        qg, dOg = f64(q[b, hs]), f64(dO[b, hs])
        kg, vg = f64(k[b, hk:hk + 1]), f64(v[b, hk:hk + 1])
        o_ref, lse_ref = oracle.attn_fwd(qg, kg, vg, scale, causal)
        eo = float(np.abs(f64(out["o"][b, hs]) - o_ref).max())
        el = float(np.abs(f64(out["lse"][b, hs]) - lse_ref).max())
        assert eo <= TOL_O, f"O max-abs {eo} at key/value head {(b, hk)}"
        assert el <= TOL_LSE, f"LSE max-abs {el} at key/value head {(b, hk)}"
        dq_ref, dk_ref, dv_ref = oracle.attn_bwd(qg, kg, vg, dOg, scale, causal)
        for g in range(G):
            e = rel_fro(f64(out["dq"][b, hk * G + g]), dq_ref[g])
            assert e <= TOL_GRAD, f"dq rel-Frobenius {e} at query head {(b, hk * G + g)}"
            worst["dq"] = max(worst["dq"], e)
        for name, r in (("dk", dk_ref[0]), ("dv", dv_ref[0])):
            e = rel_fro(f64(out[name][b, hk]), r)
            assert e <= TOL_GRAD, f"{name} rel-Frobenius {e} at key/value head {(b, hk)}"
            worst[name] = max(worst[name], e)
        worst["o"], worst["lse"] = max(worst["o"], eo), max(worst["lse"], el)
    record("o max-abs", worst["o"], TOL_O, kv_heads=len(kv_heads))
    record("lse max-abs", worst["lse"], TOL_LSE, kv_heads=len(kv_heads))
    for name in ("dq", "dk", "dv"):
        record(f"{name} rel-Frobenius", worst[name], TOL_GRAD, kv_heads=len(kv_heads))
    return worst
