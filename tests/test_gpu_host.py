"""Host-memory entry points on the GPU: fa_fwd_bwd_host and fa_fwd_host
against the fp64 oracle, and against the device entry points on the same
inputs (o, lse, dk, dv bit for bit; dq to the order of its fp32 additions).

The shapes cut the key/value heads into groups of unequal size, give a group
an odd number of query rows (its lse slice then starts off a 16-byte
boundary), and cover the empty-query case, group counts above the number of
heads, and back-to-back calls on one stream that reuse the staging area.
"""
import pytest
import torch

import io_aware_exact_10_gb300 as fa
from parity import check_groups, gqa_inputs

pytestmark = pytest.mark.gpu


def pinned(t):
    return t.contiguous().pin_memory()


def host_step(q, k, v, dO, scale, causal, chunks, stream=None, dev_buf=None):
    """fa_fwd_bwd_host on pinned copies of the inputs; returns the host outputs
    (synchronised) and the staging buffer."""
    B, H, Nq, d = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    hq, hk, hv, hdO = (pinned(t) for t in (q, k, v, dO))
    ho, hdq = torch.full_like(hq, 7.0).pin_memory(), torch.full_like(hq, 7.0).pin_memory()
    hl = torch.full((B, H, Nq), 7.0).pin_memory()
    hdk, hdv = torch.full_like(hk, 7.0).pin_memory(), torch.full_like(hv, 7.0).pin_memory()
    nbytes = fa.fa_fwd_bwd_host_device_bytes(B, H, H_kv, Nq, Nk, d, chunks)
    if dev_buf is None:
        dev_buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    fa.fa_fwd_bwd_host(hq, hk, hv, hdO, ho, hl, hdq, hdk, hdv, B, H, H_kv, Nq, Nk, d, scale,
                       causal, dev_buf, nbytes, chunks, stream)
    (stream or torch.cuda.current_stream()).synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    return {"o": ho, "lse": hl, "dq": hdq, "dk": hdk, "dv": hdv}, dev_buf


def device_step(q, k, v, dO, scale, causal):
    """The device entry points on the same inputs (reference for bitwise checks)."""
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = fa.forward(qd, kd, vd, scale, causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale, causal)
    torch.cuda.synchronize()
    return {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}


def same_as_device(out, ref):
    for name in ("o", "lse", "dk", "dv"):
        assert torch.equal(out[name], ref[name]), name
    dq, dq_ref = out["dq"].double(), ref["dq"].double()
    err = ((dq - dq_ref).norm() / dq_ref.norm().clamp_min(1e-30)).item()
    assert err <= 1e-3, err


HOST_SHAPES = [
    # B, H, H_kv, N_q, N_k, d, causal, chunks
    (2, 4, 2, 200, 200, 64, True, 3),     # groups of 1, 1 and 2 key/value heads; ragged tiles
    (1, 6, 3, 77, 301, 128, False, 3),    # odd N_q: each group's lse starts off 16 bytes
    (1, 8, 2, 256, 640, 64, True, 0),     # the default group count, capped at B * H_kv = 2
    (3, 2, 2, 130, 130, 128, False, 64),  # more groups asked for than heads
    (1, 4, 4, 384, 384, 64, False, 1),    # one group: no overlap, same result
]


@pytest.mark.parametrize("B,H,H_kv,Nq,Nk,d,causal,chunks", HOST_SHAPES)
def test_host_step(B, H, H_kv, Nq, Nk, d, causal, chunks):
    q, k, v, dO = gqa_inputs(B, H, H_kv, Nq, d, seed=11 * Nq + Nk + d, N_k=Nk)
    scale = d ** -0.5
    out, _ = host_step(q, k, v, dO, scale, causal, chunks)
    check_groups(q, k, v, dO, out, scale, causal, [(b, hk) for b in range(B) for hk in range(H_kv)])
    same_as_device(out, device_step(q, k, v, dO, scale, causal))


def test_host_forward_only():
    B, H, H_kv, Nq, Nk, d = 2, 4, 1, 199, 513, 128
    q, k, v, _ = gqa_inputs(B, H, H_kv, Nq, d, seed=5, N_k=Nk)
    scale = d ** -0.5
    hq, hk, hv = (pinned(t) for t in (q, k, v))
    ho = torch.full_like(hq, 7.0).pin_memory()
    hl = torch.full((B, H, Nq), 7.0).pin_memory()
    nbytes = fa.fa_fwd_host_device_bytes(B, H, H_kv, Nq, Nk, d)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    fa.fa_fwd_host(hq, hk, hv, ho, hl, B, H, H_kv, Nq, Nk, d, scale, True, buf, nbytes, 2)
    torch.cuda.synchronize()
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), scale, True)
    assert torch.equal(ho, o.cpu()) and torch.equal(hl, lse.cpu())


def test_host_block_sparse():
    """A block mask passes through to every group: the host call equals the
    block-sparse device entry points, and the oracle on two groups."""
    import numpy as np
    B, H, H_kv, N, d = 2, 4, 2, 640, 128
    q, k, v, dO = gqa_inputs(B, H, H_kv, N, d, seed=17)
    scale = d ** -0.5
    nt = -(-N // 128)
    rng = np.random.default_rng(5)
    mask = (rng.random((nt, nt)) < 0.5) | np.eye(nt, dtype=bool)
    mask[2, :] = False  # a query block that sees no key: o = 0, lse = -inf
    m_dev = torch.from_numpy(mask.astype(np.uint8)).cuda()
    hq, hk, hv, hdO = (pinned(t) for t in (q, k, v, dO))
    ho, hdq = torch.empty_like(hq).pin_memory(), torch.empty_like(hq).pin_memory()
    hl = torch.empty((B, H, N)).pin_memory()
    hdk, hdv = torch.empty_like(hk).pin_memory(), torch.empty_like(hv).pin_memory()
    nbytes = fa.fa_fwd_bwd_host_device_bytes(B, H, H_kv, N, N, d, 3)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    fa.fa_fwd_bwd_host(hq, hk, hv, hdO, ho, hl, hdq, hdk, hdv, B, H, H_kv, N, N, d, scale, True,
                       buf, nbytes, 3, block_mask=m_dev)
    torch.cuda.synchronize()
    assert fa.fa_last_device_error() == fa.FA_OK
    out = {"o": ho, "lse": hl, "dq": hdq, "dk": hdk, "dv": hdv}
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = fa.forward(qd, kd, vd, scale, True, block_mask=m_dev)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dOd, scale, True, block_mask=m_dev)
    torch.cuda.synchronize()
    same_as_device(out, {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(),
                         "dv": dv.cpu()})
    assert torch.isneginf(hl[:, :, 256:384]).all() and not ho[:, :, 256:384].any()
    import oracle
    from parity import f64, rel_fro, TOL_GRAD, TOL_O
    G = H // H_kv
    for b, hk_ in ((0, 1), (1, 0)):
        hs = slice(hk_ * G, hk_ * G + G)
        o_ref, _ = oracle.attn_fwd(f64(q[b, hs]), f64(k[b, hk_:hk_ + 1]), f64(v[b, hk_:hk_ + 1]),
                                   scale, True, block_mask=mask)
        assert float(np.abs(f64(ho[b, hs]) - o_ref).max()) <= TOL_O
        _, dk_ref, dv_ref = oracle.attn_bwd(f64(q[b, hs]), f64(k[b, hk_:hk_ + 1]),
                                            f64(v[b, hk_:hk_ + 1]), f64(dO[b, hs]), scale, True,
                                            block_mask=mask)
        assert rel_fro(f64(hdk[b, hk_]), dk_ref[0]) <= TOL_GRAD
        assert rel_fro(f64(hdv[b, hk_]), dv_ref[0]) <= TOL_GRAD


def test_host_no_query_rows_zeroes_key_gradients():
    B, H, H_kv, Nk, d = 1, 4, 2, 300, 64
    _, k, v, _ = gqa_inputs(B, H, H_kv, 1, d, seed=3, N_k=Nk)
    q = torch.empty((B, H, 0, d), dtype=torch.bfloat16)
    out, _ = host_step(q, k, v, q.clone(), d ** -0.5, True, 2)
    assert not out["dk"].any() and not out["dv"].any()


def test_host_back_to_back_on_one_stream():
    """Two calls enqueued on one stream with one staging area and no
    synchronisation between them: the second must not overwrite the first's
    device inputs before its kernels ran, nor its outputs before they were
    copied back."""
    B, H, H_kv, N, d = 2, 4, 4, 512, 64
    scale = d ** -0.5
    a = gqa_inputs(B, H, H_kv, N, d, seed=21)
    b = gqa_inputs(B, H, H_kv, N, d, seed=22)
    s = torch.cuda.Stream()
    nbytes = fa.fa_fwd_bwd_host_device_bytes(B, H, H_kv, N, N, d, 4)
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ha = [pinned(t) for t in a]
    hb = [pinned(t) for t in b]
    outs = []
    for src in (ha, hb):
        o = {n: torch.empty_like(src[0]).pin_memory() for n in ("o", "dq")}
        o["lse"] = torch.empty((B, H, N)).pin_memory()
        o["dk"], o["dv"] = torch.empty_like(src[1]).pin_memory(), torch.empty_like(src[2]).pin_memory()
        fa.fa_fwd_bwd_host(*src, o["o"], o["lse"], o["dq"], o["dk"], o["dv"], B, H, H_kv, N, N, d,
                           scale, False, buf, nbytes, 4, s)
        outs.append(o)
    s.synchronize()
    same_as_device(outs[0], device_step(*a, scale, False))
    same_as_device(outs[1], device_step(*b, scale, False))
