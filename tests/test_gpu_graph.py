"""CUDA graphs: the C-ABI calls can be captured on a stream and replayed, and
a replay computes what an eager call computes on the inputs then in the
buffers (o, lse, dk, dv bit for bit; dq up to the order of its fp32
additions).  The first call of each entry point runs eagerly before the
capture (it resolves the device and the driver's tensor-map encoder once)."""
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from parity import gqa_inputs

pytestmark = pytest.mark.gpu


def same(a, b):
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(a[name], b[name]), name
    err = ((a["dq"].double() - b["dq"].double()).norm() / b["dq"].double().norm()).item()
    assert err <= 1e-3, err


def test_capture_and_replay_device_entry_points():
    B, H, H_kv, Nq, Nk, d, causal = 2, 4, 2, 600, 700, 64, True
    scale = d ** -0.5
    q, k, v, dO = (t.cuda() for t in gqa_inputs(B, H, H_kv, Nq, d, seed=31, N_k=Nk))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = fa.fa_bwd_workspace_size(B, H, Nq, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")

    def step(stream=None):
        fa.fa_fwd_ex(q, k, v, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal, stream)
        fa.fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, Nq, Nk, d, scale, causal, ws,
                     wsb, stream)

    def outputs():
        return {"o": o.clone(), "lse": lse.clone(), "dq": dq.clone(), "dk": dk.clone(),
                "dv": dv.clone()}

    step()
    torch.cuda.synchronize()
    eager = outputs()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    same(outputs(), eager)
    # new inputs in the same buffers: the replay follows them
    q2, k2, v2, dO2 = (t.cuda() for t in gqa_inputs(B, H, H_kv, Nq, d, seed=32, N_k=Nk))
    for dst, src in ((q, q2), (k, k2), (v, v2), (dO, dO2)):
        dst.copy_(src)
    g.replay()
    torch.cuda.synchronize()
    replayed = outputs()
    step()
    torch.cuda.synchronize()
    same(replayed, outputs())


def test_capture_and_replay_host_entry_point():
    """The host-memory entry point's two internal copy streams join the
    capture through the caller's stream (its start and done events), so the
    whole pipeline of copies and kernels becomes one graph."""
    B, H, H_kv, N, d = 2, 4, 4, 384, 128
    scale = d ** -0.5
    q, k, v, dO = (t.pin_memory() for t in gqa_inputs(B, H, H_kv, N, d, seed=33))
    ho, hdq = torch.empty_like(q).pin_memory(), torch.empty_like(q).pin_memory()
    hl = torch.empty((B, H, N)).pin_memory()
    hdk, hdv = torch.empty_like(k).pin_memory(), torch.empty_like(v).pin_memory()
    nbytes = fa.fa_fwd_bwd_host_device_bytes(B, H, H_kv, N, N, d, 3)
    stage = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    def step():
        fa.fa_fwd_bwd_host(q, k, v, dO, ho, hl, hdq, hdk, hdv, B, H, H_kv, N, N, d, scale, False,
                           stage, nbytes, 3)

    def outputs():
        return {"o": ho.clone(), "lse": hl.clone(), "dq": hdq.clone(), "dk": hdk.clone(),
                "dv": hdv.clone()}

    step()
    torch.cuda.synchronize()
    eager = outputs()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (ho, hl, hdq, hdk, hdv):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    same(outputs(), eager)
