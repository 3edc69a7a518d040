"""Checks that pin the fp64 oracle to facts other than itself.

Each function takes an ``oracle.OracleLib`` and raises AssertionError when the
oracle disagrees with a closed form, an invariant, brute force, an independent
formulation or a library routine.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` runs them on oracles with planted
mistakes and expects at least one of them to fail for every mistake.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def read_four_scores():
    """Parse tests/golden/four_scores.txt into {key: [hand values...]}."""
    out = {}
    with open(os.path.join(GOLDEN, "four_scores.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key = line.split()[0]
            out[key] = line
    scores = [float(x) for x in out["scores"].split()[1:]]
    hand = {}
    for key in ("block1_sum", "final_sum", "lse"):
        hand[key] = float(out[key].split()[-1])
    hand["softmax"] = [float(x) for x in out["softmax"].split()[-4:]]
    return scores, hand


# ----------------------------------------------------------------------------
# forward pins
# ----------------------------------------------------------------------------

def check_four_scores(orc):
    """The worked four-score example: oracle softmax row and LSE equal the
    closed forms, which equal the hand values to 4 digits, and the online
    recurrence over the two blocks reaches the same sum."""
    x, hand = read_four_scores()
    e = math.exp
    final_sum = 1 + e(-1) + e(-2) + e(-3)
    soft = [e(xi - 4) / final_sum for xi in x]
    lse = 4 + math.log(final_sum)
    # closed forms against the hand values written in the golden file
    assert abs((1 + e(-1)) - hand["block1_sum"]) < 1e-4
    assert abs(final_sum - hand["final_sum"]) < 1e-4
    assert np.allclose(soft, hand["softmax"], atol=1e-4)
    assert abs(lse - hand["lse"]) < 1e-4
    # the recurrence of the page on the two blocks
    m, s = -math.inf, 0.0
    for blk in ((1.0, 2.0), (3.0, 4.0)):
        for xi in blk:
            m_new = max(m, xi)
            s = s * (e(m - m_new) if m > -math.inf else 0.0) + e(xi - m_new)
            m = m_new
        if blk == (1.0, 2.0):
            assert m == 2.0 and abs(s - (1 + e(-1))) < 1e-15
    assert m == 4.0 and abs(s - final_sum) < 1e-15
    # the oracle: d = 4, q_i = e_0, k_j = x_j e_0, v_j = e_j, so o_i = p_i
    N = d = 4
    q = np.zeros((N, d)); q[:, 0] = 1.0
    k = np.zeros((N, d)); k[:, 0] = x
    v = np.eye(N)
    o, l = orc.attn_fwd(q, k, v, 1.0, False)
    for i in range(N):
        assert np.allclose(o[i], soft, rtol=0, atol=1e-14)
        assert abs(l[i] - lse) < 1e-13


def check_rows_sum_to_one(orc):
    """With V = I (N <= d) the output is P itself: rows sum to 1, entries >= 0,
    causal entries above the diagonal are exactly 0.  With V = ones, O = 1."""
    r = _rng(1)
    for causal in (False, True):
        N, d = 16, 16
        q, k = r.normal(size=(2, N, d)), r.normal(size=(2, N, d))
        v = np.broadcast_to(np.eye(N), (2, N, d)).copy()
        P, _ = orc.attn_fwd(q, k, v, 0.3, causal)
        assert np.all(P >= 0)
        assert np.allclose(P.sum(-1), 1.0, atol=1e-14)
        if causal:
            assert np.all(np.triu(P[0], 1) == 0) and np.all(np.triu(P[1], 1) == 0)
        N, d = 40, 8
        q, k = r.normal(size=(N, d)), r.normal(size=(N, d))
        o, _ = orc.attn_fwd(q, k, np.ones((N, d)), 0.5, causal)
        assert np.allclose(o, 1.0, atol=1e-13)


def check_softmax_of_scores(orc):
    """O = P with V = I equals the textbook softmax of scale*q.k computed by
    brute force in numpy, and LSE equals log(sum(exp)) of the same scores."""
    r = _rng(2)
    for causal in (False, True):
        N, d, scale = 12, 12, 0.7
        q, k = r.normal(size=(N, d)), r.normal(size=(N, d))
        P, lse = orc.attn_fwd(q, k, np.eye(N), scale, causal)
        for i in range(N):
            s = [scale * sum(q[i, c] * k[j, c] for c in range(d))
                 for j in range(N) if (not causal or j <= i)]
            ex = [math.exp(t) for t in s]
            tot = sum(ex)
            assert np.allclose(P[i, :len(ex)], [t / tot for t in ex], atol=1e-14)
            assert abs(lse[i] - math.log(tot)) < 1e-12


def check_identical_keys(orc):
    """All k_j equal: p_ij = 1/N, O_i = mean_j V_j, LSE_i = scale q_i.k + ln N;
    causal: O_i = mean_{j<=i} V_j, LSE_i = scale q_i.k + ln(i+1)."""
    r = _rng(3)
    N, d, scale = 24, 8, 0.25
    q = r.normal(size=(N, d))
    k = np.tile(r.normal(size=(1, d)), (N, 1))
    v = r.normal(size=(N, d))
    o, lse = orc.attn_fwd(q, k, v, scale, False)
    assert np.allclose(o, v.mean(0, keepdims=True), atol=1e-13)
    assert np.allclose(lse, scale * q @ k[0] + math.log(N), atol=1e-12)
    o, lse = orc.attn_fwd(q, k, v, scale, True)
    pref = np.cumsum(v, 0) / np.arange(1, N + 1)[:, None]
    assert np.allclose(o, pref, atol=1e-13)
    assert np.allclose(lse, scale * q @ k[0] + np.log(np.arange(1, N + 1)),
                       atol=1e-12)


def check_causal_row0(orc):
    """Causal row 0 sees key 0 only: O_0 = V_0, LSE_0 = scale q_0.k_0."""
    r = _rng(4)
    N, d, scale = 32, 16, 0.125
    q, k, v = (r.normal(size=(N, d)) for _ in range(3))
    o, lse = orc.attn_fwd(q, k, v, scale, True)
    assert np.allclose(o[0], v[0], atol=1e-15)
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-13


def check_zero_queries(orc):
    """Q = 0: all scores 0, O = column mean of V, LSE = ln N (causal: prefix)."""
    r = _rng(5)
    N, d = 20, 6
    q = np.zeros((N, d))
    k, v = r.normal(size=(N, d)), r.normal(size=(N, d))
    o, lse = orc.attn_fwd(q, k, v, 1.0, False)
    assert np.allclose(o, v.mean(0, keepdims=True), atol=1e-13)
    assert np.allclose(lse, math.log(N), atol=1e-13)
    o, lse = orc.attn_fwd(q, k, v, 1.0, True)
    assert np.allclose(o, np.cumsum(v, 0) / np.arange(1, N + 1)[:, None], atol=1e-13)
    assert np.allclose(lse, np.log(np.arange(1, N + 1)), atol=1e-13)


def check_dominant_key(orc):
    """One key whose score exceeds every other by >= 60: O_i = V_{j*} to
    within e^-60 * N * max|V|, LSE_i = s_{i j*} up to the same."""
    r = _rng(6)
    N, d = 16, 4
    q = np.zeros((N, d)); q[:, 0] = 1.0
    k = r.uniform(-1, 1, size=(N, d)); k[:, 0] = r.uniform(-1, 1, size=N)
    jstar = 11
    k[jstar, 0] = 62.0
    v = r.normal(size=(N, d))
    o, lse = orc.attn_fwd(q, k, v, 1.0, False)
    assert np.allclose(o, v[jstar][None, :], atol=1e-20 + N * math.exp(-60) * 4)
    assert np.allclose(lse, 62.0, atol=1e-20 + N * math.exp(-60))


def _online_blocked(q, k, v, scale, causal, bounds):
    """Independent blocked forward: the per-block recurrence with an
    unnormalised output and one final divide, per query row (Flash Attention,
    "Core Flash Attention Algorithm", in the one-divide form its Flash
    Attention 2 section describes).  Pure numpy, no oracle code."""
    N, d = q.shape
    o = np.zeros((N, d))
    lse = np.zeros(N)
    for i in range(N):
        m, l, acc = -np.inf, 0.0, np.zeros(d)
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            js = [j for j in range(lo, hi) if not causal or j <= i]
            if not js:
                continue
            s = scale * (k[js] @ q[i])
            m_new = max(m, s.max())
            alpha = math.exp(m - m_new) if m > -np.inf else 0.0
            p = np.exp(s - m_new)
            l = l * alpha + p.sum()
            acc = acc * alpha + p @ v[js]
            m = m_new
        o[i] = acc / l
        lse[i] = m + math.log(l)
    return o, lse


def check_blocked_online_softmax(orc):
    """Block-sum invariant: any partition of the keys into blocks, run through
    the online recurrence, reproduces the oracle to 1e-12 (Flash Attention,
    "Mathematical Correctness")."""
    r = _rng(7)
    for causal in (False, True):
        for trial in range(4):
            N, d = int(r.integers(5, 40)), int(r.integers(1, 9))
            q, k, v = (r.normal(size=(N, d)) * 2 for _ in range(3))
            cuts = sorted(set(r.integers(1, N, size=int(r.integers(0, 6))).tolist()))
            bounds = [0] + cuts + [N]
            ob, lb = _online_blocked(q, k, v, 0.6, causal, bounds)
            o, l = orc.attn_fwd(q, k, v, 0.6, causal)
            assert np.allclose(o, ob, atol=1e-12, rtol=0)
            assert np.allclose(l, lb, atol=1e-12, rtol=0)


def check_multi_head_independent(orc):
    """Heads are independent: a [B, H] batch equals each head run alone."""
    r = _rng(8)
    B, H, N, d = 2, 3, 10, 4
    q, k, v = (r.normal(size=(B, H, N, d)) for _ in range(3))
    o, lse = orc.attn_fwd(q, k, v, 0.5, True)
    for b in range(B):
        for h in range(H):
            o1, l1 = orc.attn_fwd(q[b, h], k[b, h], v[b, h], 0.5, True)
            assert np.array_equal(o1, o[b, h]) and np.array_equal(l1, lse[b, h])


def check_rows_entry(orc):
    """The sampled-rows entry equals the full forward on those rows."""
    r = _rng(9)
    N, d = 33, 8
    q, k, v = (r.normal(size=(N, d)) for _ in range(3))
    rows = [0, 5, 17, 32]
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, 0.4, causal)
        o_r, l_r = orc.attn_fwd_rows(q, k, v, rows, 0.4, causal)
        assert np.allclose(o_r, o[rows], atol=1e-14)
        assert np.allclose(l_r, lse[rows], atol=1e-14)


def check_torch_sdpa_fwd(orc):
    """torch's CPU scaled_dot_product_attention in fp64 (a library routine
    sharing no code with the oracle) agrees to 1e-12."""
    import torch
    import torch.nn.functional as F
    r = _rng(10)
    for causal in (False, True):
        B, H, N, d = 2, 2, 37, 16
        q, k, v = (r.normal(size=(B, H, N, d)) for _ in range(3))
        o, _ = orc.attn_fwd(q, k, v, 0.3, causal)
        ot = F.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
            is_causal=causal, scale=0.3).numpy()
        assert np.allclose(o, ot, atol=1e-12, rtol=0)


# ----------------------------------------------------------------------------
# backward pins
# ----------------------------------------------------------------------------

def _loss(orc, q, k, v, dO, scale, causal):
    o, _ = orc.attn_fwd(q, k, v, scale, causal)
    return float((o * dO).sum())


def check_finite_differences(orc):
    """Central differences of L = sum(dO * O) w.r.t. every entry of Q, K, V on
    tiny shapes agree with the analytic gradients to 1e-6 relative."""
    r = _rng(11)
    h = 1e-6
    for causal in (False, True):
        for N, d in ((1, 1), (2, 2), (3, 4), (5, 1), (8, 2)):
            q, k, v, dO = (r.normal(size=(N, d)) for _ in range(4))
            scale = 0.9
            g = orc.attn_bwd(q, k, v, dO, scale, causal)
            for which, x in enumerate((q, k, v)):
                num = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    xp, xm = x.copy(), x.copy()
                    xp[idx] += h
                    xm[idx] -= h
                    args_p = [q, k, v]; args_p[which] = xp
                    args_m = [q, k, v]; args_m[which] = xm
                    num[idx] = (_loss(orc, *args_p, dO, scale, causal)
                                - _loss(orc, *args_m, dO, scale, causal)) / (2 * h)
                err = np.abs(num - g[which]).max()
                ref = max(np.abs(num).max(), 1e-3)
                assert err / ref < 1e-6, (causal, N, d, which, err, ref)


def check_gradient_invariants(orc):
    """sum_j dk_j = 0 (softmax ignores a shift of all keys), sum_j dv_j =
    sum_i dO_i (rows of P sum to 1), and D_i = dO_i . o_i."""
    r = _rng(12)
    for causal in (False, True):
        B, H, N, d = 1, 2, 30, 8
        q, k, v, dO = (r.normal(size=(B, H, N, d)) for _ in range(4))
        dq, dk, dv, D = orc.attn_bwd(q, k, v, dO, 0.5, causal, return_D=True)
        o, _ = orc.attn_fwd(q, k, v, 0.5, causal)
        assert np.allclose(dk.sum(-2), 0.0, atol=1e-12)
        assert np.allclose(dv.sum(-2), dO.sum(-2), atol=1e-12)
        assert np.allclose(D, (dO * o).sum(-1), atol=1e-12)


def check_torch_autograd(orc):
    """torch autograd through fp64 CPU scaled_dot_product_attention agrees with
    the oracle's gradients to 1e-11."""
    import torch
    import torch.nn.functional as F
    r = _rng(13)
    for causal in (False, True):
        B, H, N, d = 1, 2, 29, 8
        q, k, v, dO = (r.normal(size=(B, H, N, d)) for _ in range(4))
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
        out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.35)
        out.backward(torch.from_numpy(dO))
        dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.35, causal)
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-11, rtol=0)
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-11, rtol=0)
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-11, rtol=0)


def _rows_cases():
    """(Nq, Nk, causal) shapes for the backward rows entry: equal lengths
    with and without the causal mask, fewer queries than keys (causal,
    bottom-right aligned) and more queries than keys (unmasked)."""
    return ((33, 33, False), (33, 33, True), (20, 45, True), (40, 17, False))


def check_bwd_rows_entry(orc):
    """The backward rows entry equals the full backward on those rows: dq of
    the chosen query rows, dk and dv of the chosen key rows."""
    r = _rng(14)
    d = 8
    for Nq, Nk, causal in _rows_cases():
        q, dO = (r.normal(size=(Nq, d)) for _ in range(2))
        k, v = (r.normal(size=(Nk, d)) for _ in range(2))
        qrows = [0, 3, Nq // 2, Nq - 1]
        krows = [0, 1, Nk // 3, Nk - 2, Nk - 1]
        dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.45, causal)
        dq_r, dk_r, dv_r = orc.attn_bwd_rows(q, k, v, dO, qrows, krows, 0.45, causal)
        assert np.allclose(dq_r, dq[qrows], atol=1e-13, rtol=0), (Nq, Nk, causal)
        assert np.allclose(dk_r, dk[krows], atol=1e-13, rtol=0), (Nq, Nk, causal)
        assert np.allclose(dv_r, dv[krows], atol=1e-13, rtol=0), (Nq, Nk, causal)


def check_bwd_rows_torch(orc):
    """The backward rows entry against torch autograd in fp64 (explicit
    mask: key j visible to query i iff j <= i + Nk - Nq when causal) on the
    chosen rows, to 1e-11."""
    import torch
    r = _rng(15)
    d = 8
    for Nq, Nk, causal in _rows_cases():
        q, dO = (r.normal(size=(Nq, d)) for _ in range(2))
        k, v = (r.normal(size=(Nk, d)) for _ in range(2))
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
        s = (tq @ tk.T) * 0.6
        if causal:
            s = s.masked_fill(~_bottom_right_mask(Nq, Nk), float("-inf"))
        (torch.softmax(s, dim=-1) @ tv).backward(torch.from_numpy(dO))
        qrows = [1, Nq // 3, Nq - 1]
        krows = [Nk // 2 + 1, Nk - 1]  # no key 0 (which every causal row sees)
        dq_r, dk_r, dv_r = orc.attn_bwd_rows(q, k, v, dO, qrows, krows, 0.6, causal)
        assert np.allclose(dq_r, tq.grad.numpy()[qrows], atol=1e-11, rtol=0), (Nq, Nk, causal)
        assert np.allclose(dk_r, tk.grad.numpy()[krows], atol=1e-11, rtol=0), (Nq, Nk, causal)
        assert np.allclose(dv_r, tv.grad.numpy()[krows], atol=1e-11, rtol=0), (Nq, Nk, causal)


# ----------------------------------------------------------------------------
# grouped key/value heads (GQA / MQA)
# ----------------------------------------------------------------------------

def check_gqa_torch(orc):
    """Grouped key/value heads against torch in fp64: K, V repeated over each
    group with repeat_interleave (query head h takes key/value head h // G),
    scaled_dot_product_attention forward, and autograd back through the
    repeat, which sums dk, dv over each group.  Covers MQA (one key/value
    head) and a batch of two."""
    import torch
    import torch.nn.functional as F
    r = _rng(14)
    for causal in (False, True):
        for B, H, Hkv in ((2, 4, 2), (1, 6, 1), (1, 3, 3)):
            N, d, G = 23, 8, H // Hkv
            q, dO = (r.normal(size=(B, H, N, d)) for _ in range(2))
            k, v = (r.normal(size=(B, Hkv, N, d)) for _ in range(2))
            tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
            out = F.scaled_dot_product_attention(
                tq, torch.repeat_interleave(tk, G, dim=1), torch.repeat_interleave(tv, G, dim=1),
                is_causal=causal, scale=0.4)
            out.backward(torch.from_numpy(dO))
            o, _ = orc.attn_fwd(q, k, v, 0.4, causal)
            dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.4, causal)
            assert dk.shape == k.shape and dv.shape == v.shape
            assert np.allclose(o, out.detach().numpy(), atol=1e-12, rtol=0)
            assert np.allclose(dq, tq.grad.numpy(), atol=1e-11, rtol=0)
            assert np.allclose(dk, tk.grad.numpy(), atol=1e-11, rtol=0)
            assert np.allclose(dv, tv.grad.numpy(), atol=1e-11, rtol=0)


def check_gqa_finite_differences(orc):
    """Central differences of L = sum(dO * O) w.r.t. every entry of the shared
    K and V (two query heads per key/value head) agree with dk, dv."""
    r = _rng(15)
    h = 1e-6
    for causal in (False, True):
        N, d = 5, 2
        q, dO = (r.normal(size=(1, 2, N, d)) for _ in range(2))
        k, v = (r.normal(size=(1, 1, N, d)) for _ in range(2))
        _, dk, dv = orc.attn_bwd(q, k, v, dO, 0.8, causal)
        for which, (x, g) in enumerate(((k, dk), (v, dv))):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                kp, vp = (xp, v) if which == 0 else (k, xp)
                km, vm = (xm, v) if which == 0 else (k, xm)
                num[idx] = (_loss(orc, q, kp, vp, dO, 0.8, causal)
                            - _loss(orc, q, km, vm, dO, 0.8, causal)) / (2 * h)
            err = np.abs(num - g).max()
            assert err / max(np.abs(num).max(), 1e-3) < 1e-6, (causal, which, err)


# ----------------------------------------------------------------------------
# query and key lengths that differ (Nq != Nk)
# ----------------------------------------------------------------------------

def _bottom_right_mask(Nq, Nk):
    """Boolean [Nq, Nk]: query i may see key j iff j <= i + Nk - Nq."""
    import torch
    return torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)


def check_cross_torch(orc):
    """Nq != Nk against torch in fp64: scaled_dot_product_attention with no
    mask, or with an explicit bottom-right causal mask built by tril, forward
    and autograd; grouped key/value heads and several heads so that a head
    stride taken from the wrong length shows.  The first case has Nq < Nk."""
    import torch
    import torch.nn.functional as F
    r = _rng(16)
    for Nq, Nk, causal in ((7, 19, True), (7, 19, False), (19, 7, False), (1, 9, True),
                           (13, 13, True), (5, 130, True), (130, 5, False)):
        B, H, Hkv, d = 1, 4, 2, 8
        G = H // Hkv
        q, dO = (r.normal(size=(B, H, Nq, d)) for _ in range(2))
        k, v = (r.normal(size=(B, Hkv, Nk, d)) for _ in range(2))
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
        mask = _bottom_right_mask(Nq, Nk) if causal else None
        out = F.scaled_dot_product_attention(
            tq, torch.repeat_interleave(tk, G, dim=1), torch.repeat_interleave(tv, G, dim=1),
            attn_mask=mask, scale=0.45)
        out.backward(torch.from_numpy(dO))
        o, lse = orc.attn_fwd(q, k, v, 0.45, causal)
        assert o.shape == q.shape and lse.shape == q.shape[:-1]
        assert np.allclose(o, out.detach().numpy(), atol=1e-12, rtol=0), (Nq, Nk, causal)
        dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.45, causal)
        assert dk.shape == k.shape and dv.shape == v.shape
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-11, rtol=0), (Nq, Nk, causal)
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-11, rtol=0), (Nq, Nk, causal)
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-11, rtol=0), (Nq, Nk, causal)
        rows = np.array([0, Nq - 1, Nq // 2], dtype=np.int32)
        o_r, l_r = orc.attn_fwd_rows(q[0, 1], k[0, 0], v[0, 0], rows, 0.45, causal)
        assert np.allclose(o_r, o[0, 1, rows], atol=1e-13, rtol=0)
        assert np.allclose(l_r, lse[0, 1, rows], atol=1e-13, rtol=0)


def check_cross_causal_is_suffix(orc):
    """Causal attention of Nq queries on Nk >= Nq keys is the last Nq rows of
    square causal attention over Nk queries whose last Nq rows are those
    queries (a chunk of queries appended after Nk - Nq earlier positions).
    dq is the suffix of the square problem's dq, and dk, dv equal the square
    problem's with dO zero on the first Nk - Nq rows."""
    r = _rng(17)
    for Nq, Nk in ((3, 11), (1, 6), (8, 8), (9, 40)):
        d = 4
        q_full, dO_full = (r.normal(size=(2, Nk, d)) for _ in range(2))
        k, v = (r.normal(size=(2, Nk, d)) for _ in range(2))
        dO_full[:, :Nk - Nq] = 0.0
        q, dO = q_full[:, Nk - Nq:], dO_full[:, Nk - Nq:]
        o_f, lse_f = orc.attn_fwd(q_full, k, v, 0.7, True)
        o, lse = orc.attn_fwd(q, k, v, 0.7, True)
        assert np.allclose(o, o_f[:, Nk - Nq:], atol=1e-13, rtol=0), (Nq, Nk)
        assert np.allclose(lse, lse_f[:, Nk - Nq:], atol=1e-13, rtol=0), (Nq, Nk)
        dq_f, dk_f, dv_f = orc.attn_bwd(q_full, k, v, dO_full, 0.7, True)
        dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.7, True)
        assert np.allclose(dq, dq_f[:, Nk - Nq:], atol=1e-12, rtol=0), (Nq, Nk)
        assert np.allclose(dk, dk_f, atol=1e-12, rtol=0), (Nq, Nk)
        assert np.allclose(dv, dv_f, atol=1e-12, rtol=0), (Nq, Nk)


def check_cross_finite_differences(orc):
    """Central differences of L = sum(dO * O) w.r.t. every entry of Q, K, V
    with Nq != Nk (bottom-right causal and unmasked) agree with the analytic
    gradients to 1e-6 relative."""
    r = _rng(18)
    h = 1e-6
    for Nq, Nk, causal in ((2, 5, True), (2, 5, False), (4, 3, False), (1, 4, True)):
        d = 2
        q, dO = (r.normal(size=(Nq, d)) for _ in range(2))
        k, v = (r.normal(size=(Nk, d)) for _ in range(2))
        g = orc.attn_bwd(q, k, v, dO, 0.9, causal)
        for which, x in enumerate((q, k, v)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]; args_p[which] = xp
                args_m = [q, k, v]; args_m[which] = xm
                num[idx] = (_loss(orc, *args_p, dO, 0.9, causal)
                            - _loss(orc, *args_m, dO, 0.9, causal)) / (2 * h)
            err = np.abs(num - g[which]).max()
            assert err / max(np.abs(num).max(), 1e-3) < 1e-6, (Nq, Nk, causal, which, err)


# ----------------------------------------------------------------------------
# block-sparse attention (a block mask over (query, key) blocks)
# ----------------------------------------------------------------------------

def _element_mask(block_mask, bq, bk, Nq, Nk, causal):
    """Boolean [Nq, Nk] element mask: the block mask expanded by kron with
    ones(bq, bk), cut to Nq x Nk, and the bottom-right causal rule."""
    import torch
    m = torch.from_numpy(np.kron(np.asarray(block_mask, dtype=np.uint8),
                                 np.ones((bq, bk), dtype=np.uint8))[:Nq, :Nk] != 0)
    if causal:
        m &= torch.ones(Nq, Nk, dtype=torch.bool).tril(diagonal=Nk - Nq)
    return m


def check_block_sparse_torch(orc):
    """Random block masks against torch in fp64: SDPA with the element mask
    (kron expansion of the block mask, and the causal rule), forward and
    autograd, grouped heads, ragged last blocks, blocks taller or wider than
    they are long.  Every row keeps a key (block column 0 stays on), so the
    masked softmax is defined everywhere.  The first case has fewer query
    blocks than key blocks and bq < bk."""
    import torch
    import torch.nn.functional as F
    r = _rng(19)
    for Nq, Nk, bq, bk, causal in ((10, 29, 4, 8, False), (10, 29, 4, 8, True),
                                   (21, 21, 8, 4, True), (17, 9, 5, 3, False),
                                   (1, 40, 1, 7, True), (33, 64, 16, 16, True)):
        B, H, Hkv, d = 1, 4, 2, 8
        G = H // Hkv
        nbq, nbk = -(-Nq // bq), -(-Nk // bk)
        bm = (r.random((nbq, nbk)) < 0.5).astype(np.uint8)
        bm[:, 0] = 1
        q, dO = (r.normal(size=(B, H, Nq, d)) for _ in range(2))
        k, v = (r.normal(size=(B, Hkv, Nk, d)) for _ in range(2))
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
        out = F.scaled_dot_product_attention(
            tq, torch.repeat_interleave(tk, G, dim=1), torch.repeat_interleave(tv, G, dim=1),
            attn_mask=_element_mask(bm, bq, bk, Nq, Nk, causal), scale=0.5)
        out.backward(torch.from_numpy(dO))
        case = (Nq, Nk, bq, bk, causal)
        o, _ = orc.attn_fwd(q, k, v, 0.5, causal, block_mask=bm, block=(bq, bk))
        assert np.allclose(o, out.detach().numpy(), atol=1e-12, rtol=0), case
        dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.5, causal, block_mask=bm, block=(bq, bk))
        assert np.allclose(dq, tq.grad.numpy(), atol=1e-11, rtol=0), case
        assert np.allclose(dk, tk.grad.numpy(), atol=1e-11, rtol=0), case
        assert np.allclose(dv, tv.grad.numpy(), atol=1e-11, rtol=0), case


def check_block_sparse_empty_rows(orc):
    """A row that sees no key: o = 0, lse = -inf, dq = 0, D = 0, and dk, dv
    are those of the same problem without that row.  Unmasked: block row 1
    of three is all zero (rows 4..7 of 12).  Causal: block (0, 0) off leaves
    the rows of block row 0 whose visible keys all lie in it empty."""
    r = _rng(20)
    Nq, Nk, b, d = 12, 12, 4, 3
    q, k, v, dO = (r.normal(size=(Nq if i in (0, 3) else Nk, d)) for i in range(4))
    bm = np.ones((3, 3), dtype=np.uint8)
    bm[1] = 0
    o, lse = orc.attn_fwd(q, k, v, 0.6, False, block_mask=bm, block=(b, b))
    dq, dk, dv, D = orc.attn_bwd(q, k, v, dO, 0.6, False, return_D=True, block_mask=bm,
                                 block=(b, b))
    assert np.all(o[4:8] == 0) and np.all(np.isneginf(lse[4:8])) and np.all(np.isfinite(lse[:4]))
    assert np.all(dq[4:8] == 0) and np.all(D[4:8] == 0)
    keep = np.r_[0:4, 8:12]
    o2, lse2 = orc.attn_fwd(q[keep], k, v, 0.6, False)
    _, dk2, dv2 = orc.attn_bwd(q[keep], k, v, dO[keep], 0.6, False)
    assert np.allclose(o[keep], o2, atol=1e-14, rtol=0) and np.allclose(lse[keep], lse2, atol=1e-14)
    assert np.allclose(dk, dk2, atol=1e-13, rtol=0) and np.allclose(dv, dv2, atol=1e-13, rtol=0)
    # causal, square: rows 0..3 see only keys <= i, all in block (0, 0)
    bm = np.ones((3, 3), dtype=np.uint8)
    bm[0, 0] = 0
    o, lse = orc.attn_fwd(q, k, v, 0.6, True, block_mask=bm, block=(b, b))
    dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.6, True, block_mask=bm, block=(b, b))
    assert np.all(o[:4] == 0) and np.all(np.isneginf(lse[:4])) and np.all(dq[:4] == 0)
    assert np.all(np.isfinite(lse[4:])) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def check_block_diagonal_is_independent(orc):
    """A block-diagonal mask splits attention into independent problems:
    query block i attends only to key block i, so every output equals the
    unmasked oracle run on that pair of blocks alone."""
    r = _rng(21)
    for causal in (False, True):
        b, nb, d = 5, 3, 4
        N = b * nb
        q, k, v, dO = (r.normal(size=(2, N, d)) for _ in range(4))
        bm = np.eye(nb, dtype=np.uint8)
        o, lse = orc.attn_fwd(q, k, v, 0.8, causal, block_mask=bm, block=(b, b))
        dq, dk, dv = orc.attn_bwd(q, k, v, dO, 0.8, causal, block_mask=bm, block=(b, b))
        for i in range(nb):
            s = slice(i * b, i * b + b)
            ob, lb = orc.attn_fwd(q[:, s], k[:, s], v[:, s], 0.8, causal)
            gb = orc.attn_bwd(q[:, s], k[:, s], v[:, s], dO[:, s], 0.8, causal)
            assert np.allclose(o[:, s], ob, atol=1e-14, rtol=0) and np.allclose(lse[:, s], lb, atol=1e-14)
            for g, ref in zip((dq, dk, dv), gb):
                assert np.allclose(g[:, s], ref, atol=1e-13, rtol=0), (causal, i)


def check_block_sparse_finite_differences(orc):
    """Central differences of L = sum(dO * O) w.r.t. every entry of Q, K, V
    under a block mask agree with the analytic gradients to 1e-6 relative."""
    r = _rng(22)
    h = 1e-6
    for causal in (False, True):
        Nq, Nk, bq, bk, d = 4, 6, 2, 3, 2
        bm = np.array([[1, 0], [1, 1]], dtype=np.uint8)
        q, dO = (r.normal(size=(Nq, d)) for _ in range(2))
        k, v = (r.normal(size=(Nk, d)) for _ in range(2))
        g = orc.attn_bwd(q, k, v, dO, 0.9, causal, block_mask=bm, block=(bq, bk))
        loss = lambda *a: float((orc.attn_fwd(*a, 0.9, causal, block_mask=bm,
                                               block=(bq, bk))[0] * dO).sum())
        for which, x in enumerate((q, k, v)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]; args_p[which] = xp
                args_m = [q, k, v]; args_m[which] = xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.abs(num - g[which]).max()
            assert err / max(np.abs(num).max(), 1e-3) < 1e-6, (causal, which, err)


FWD_CHECKS = (check_four_scores, check_rows_sum_to_one, check_softmax_of_scores,
              check_identical_keys, check_causal_row0, check_zero_queries,
              check_dominant_key, check_blocked_online_softmax,
              check_multi_head_independent, check_rows_entry, check_torch_sdpa_fwd)
BWD_CHECKS = (check_finite_differences, check_gradient_invariants, check_torch_autograd,
              check_bwd_rows_entry, check_bwd_rows_torch)
GQA_CHECKS = (check_gqa_torch, check_gqa_finite_differences)
CROSS_CHECKS = (check_cross_torch, check_cross_causal_is_suffix, check_cross_finite_differences)
SPARSE_CHECKS = (check_block_sparse_torch, check_block_sparse_empty_rows,
                 check_block_diagonal_is_independent, check_block_sparse_finite_differences)
ALL_CHECKS = FWD_CHECKS + BWD_CHECKS + GQA_CHECKS + CROSS_CHECKS + SPARSE_CHECKS
