"""Pins of the fp64 oracle against things other than itself (CPU only).

The oracle restates the backward equations of the page "CANN ops-transformer FlashAttnGrad
算子详解" (discosf.com/news/4863418), §一.  These tests check it against:
  * central finite differences of L = Σ dY ⊙ Y(q, k, v) (the backward is the derivative of the
    forward: a dropped term, wrong sign or transposed operand anywhere breaks it);
  * torch fp64 autograd through a plain softmax attention (a library differentiation);
  * an exact sympy differentiation stored in tests/golden/exact_causal_gqa.json;
  * closed forms (one key, q = 0, two keys), invariants (Σ_j dS_ij = 0), GQA == repeated-KV MHA
    and TND == per-sequence BSND;
and finally plant mistakes in the oracle to show each pin family catches them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import fabwd_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "exact_causal_gqa.json")


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def make(layout, B, S1, S2, N1, N2, D, Dv, seed, cu_q=None, cu_kv=None):
    if layout == "BSND":
        shp = lambda S, N, d: (B, S, N, d)
    elif layout == "BNSD":
        shp = lambda S, N, d: (B, N, S, d)
    else:
        shp = lambda S, N, d: (S, N, d)
        S1, S2 = int(cu_q[-1]), int(cu_kv[-1])
    q = rand(shp(S1, N1, D), seed)
    k = rand(shp(S2, N2, D), seed + 1)
    v = rand(shp(S2, N2, Dv), seed + 2)
    dy = rand(shp(S1, N1, Dv), seed + 3)
    return q, k, v, dy


def loss(q, k, v, dy, kw):
    y, _ = orc.forward(q, k, v, **kw)
    return float((dy * y).sum())


def fd_grad(x, f, h=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


CASES = [
    # name, layout, B, S1, S2, N1, N2, D, Dv, kw, cu_q, cu_kv
    ("dense", "BSND", 1, 5, 5, 2, 2, 3, 2, dict(), None, None),
    ("dense_scale", "BSND", 2, 4, 6, 2, 1, 4, 3, dict(softmax_scale=0.3), None, None),
    ("causal_s1_lt_s2_gqa", "BSND", 1, 4, 6, 4, 2, 4, 3, dict(mask_mode=1), None, None),
    ("causal_s1_gt_s2_empty_rows", "BSND", 1, 6, 4, 2, 1, 3, 3, dict(mask_mode=1), None, None),
    ("band", "BSND", 1, 7, 7, 2, 2, 3, 2, dict(mask_mode=2, win_left=1, win_right=1), None, None),
    ("causal_window", "BSND", 1, 7, 7, 2, 1, 3, 2, dict(mask_mode=1, win_left=2, win_right=0), None, None),
    ("band_right_only", "BSND", 1, 5, 7, 2, 2, 2, 2, dict(mask_mode=2, win_left=-1, win_right=0), None, None),
    ("bnsd_causal", "BNSD", 2, 4, 4, 2, 2, 3, 2, dict(mask_mode=1), None, None),
    ("tnd_causal_gqa", "TND", 3, 0, 0, 4, 2, 3, 2, dict(mask_mode=1),
     np.array([0, 3, 8, 9]), np.array([0, 4, 9, 11])),
    ("tnd_window", "TND", 2, 0, 0, 2, 2, 2, 3, dict(mask_mode=1, win_left=1, win_right=0),
     np.array([0, 5, 8]), np.array([0, 5, 8])),
]


def case_inputs(case, seed=11):
    name, layout, B, S1, S2, N1, N2, D, Dv, kw, cu_q, cu_kv = case
    q, k, v, dy = make(layout, B, S1, S2, N1, N2, D, Dv, seed, cu_q, cu_kv)
    kw = dict(kw, layout=layout)
    if layout == "TND":
        kw.update(cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv)
    return q, k, v, dy, kw


def fd_check(q, k, v, dy, kw, rtol=1e-6):
    y, lse = orc.forward(q, k, v, **kw)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, **kw)
    f = lambda: loss(q, k, v, dy, kw)
    ok = True
    for got, x in ((dq, q), (dk, k), (dv, v)):
        ref = fd_grad(x, f)
        ok &= np.allclose(got, ref, rtol=rtol, atol=rtol * max(1.0, np.abs(ref).max()))
    return ok


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_finite_differences(case):
    q, k, v, dy, kw = case_inputs(case)
    assert fd_check(q, k, v, dy, kw)


# ---------------------------------------------------------------------------------------------
# torch fp64 autograd of a plain softmax attention (an independent differentiation)
# ---------------------------------------------------------------------------------------------


def torch_grads(q, k, v, dy, *, scale, ok):
    """BSND, one batch: per head softmax attention in torch fp64, differentiated by autograd."""
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    N1, N2 = q.shape[2], k.shape[2]
    G = N1 // N2
    tot = 0
    for n1 in range(N1):
        s = scale * tq[0, :, n1, :] @ tk[0, :, n1 // G, :].T
        s = s.masked_fill(~torch.tensor(ok), float("-inf"))
        p = torch.softmax(s, dim=1)
        y = p @ tv[0, :, n1 // G, :]
        tot = tot + (torch.tensor(dy[0, :, n1, :]) * y).sum()
    tot.backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


TORCH_CASES = [
    (6, 6, 2, 2, 4, 4, dict(), 0.0),
    (5, 9, 4, 2, 8, 5, dict(mask_mode=1), 0.25),
    (9, 9, 3, 1, 6, 6, dict(mask_mode=2, win_left=2, win_right=3), 0.0),
    (9, 9, 2, 2, 6, 6, dict(mask_mode=1, win_left=3, win_right=0), 0.0),
]


@pytest.mark.parametrize("S1,S2,N1,N2,D,Dv,mkw,sc", TORCH_CASES)
def test_torch_autograd(S1, S2, N1, N2, D, Dv, mkw, sc):
    q, k, v, dy = make("BSND", 1, S1, S2, N1, N2, D, Dv, 21)
    kw = dict(mkw, softmax_scale=sc)
    y, lse = orc.forward(q, k, v, **kw)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, **kw)
    ok = orc.visible(S1, S2, kw.get("mask_mode", 0), kw.get("win_left", -1), kw.get("win_right", -1))
    assert ok.any(axis=1).all()
    gq, gk, gv = torch_grads(q, k, v, dy, scale=orc.resolve_scale(sc, D), ok=ok)
    np.testing.assert_allclose(dq, gq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, gk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, gv, rtol=1e-10, atol=1e-12)
    # forward against torch softmax too
    tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
    for n1 in range(N1):
        s = orc.resolve_scale(sc, D) * tq[0, :, n1] @ tk[0, :, n1 // (N1 // N2)].T
        s = s.masked_fill(~torch.tensor(ok), float("-inf"))
        np.testing.assert_allclose(y[0, :, n1], (torch.softmax(s, 1) @ tv[0, :, n1 // (N1 // N2)]).numpy(),
                                   rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[0, n1], torch.logsumexp(s, 1).numpy(), rtol=1e-13)


# ---------------------------------------------------------------------------------------------
# exact sympy golden
# ---------------------------------------------------------------------------------------------


def golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    S1, S2, N1, N2, D, Dv = (g[x] for x in ("S1", "S2", "N1", "N2", "D", "Dv"))
    from fractions import Fraction
    arr = lambda key, shp: np.array([float(Fraction(x)) if "/" in x or x.lstrip("-").isdigit() else float(x)
                                      for x in g[key]]).reshape(shp)
    return g, dict(
        q=arr("q", (1, S1, N1, D)), k=arr("k", (1, S2, N2, D)), v=arr("v", (1, S2, N2, Dv)),
        dout=arr("dout", (1, S1, N1, Dv)), y=arr("attn_out", (1, S1, N1, Dv)),
        lse=arr("softmax_lse", (1, N1, S1)), dq=arr("dq", (1, S1, N1, D)), dk=arr("dk", (1, S2, N2, D)),
        dv=arr("dv", (1, S2, N2, Dv)))


def test_exact_golden():
    g, a = golden()
    kw = dict(softmax_scale=g["softmax_scale"], mask_mode=g["mask_mode"])
    y, lse = orc.forward(a["q"], a["k"], a["v"], **kw)
    np.testing.assert_allclose(y, a["y"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, a["lse"], rtol=1e-13, atol=1e-14)
    dq, dk, dv, _ = orc.backward(a["q"], a["k"], a["v"], a["dout"], y, lse, **kw)
    np.testing.assert_allclose(dq, a["dq"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, a["dk"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, a["dv"], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------------------------


def test_single_key_closed_form():
    # one key: P == 1, Y = v, dS = 0, so dq = dk = 0 and dv = Σ_i dY_i
    q, k, v, dy = make("BSND", 1, 5, 1, 3, 1, 4, 3, 31)
    y, lse = orc.forward(q, k, v)
    np.testing.assert_allclose(y, np.broadcast_to(v[:, :, :1, :].reshape(1, 1, 1, 3), y.shape), atol=1e-15)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    np.testing.assert_allclose(dv[0, 0, 0], dy[0].sum(axis=(0, 1)), rtol=1e-13)


def test_zero_query_closed_form():
    # q = 0, no mask: P uniform 1/S2, Y_i = mean_j v_j, dv_j = (1/S2) Σ_i dY_i, dk = 0,
    # dq_i = scale · (1/S2) Σ_j (dY_i·(v_j − v̄)) k_j   (a covariance over keys)
    S1, S2, D, Dv = 4, 6, 3, 2
    _, k, v, dy = make("BSND", 1, S1, S2, 1, 1, D, Dv, 41)
    q = np.zeros((1, S1, 1, D))
    y, lse = orc.forward(q, k, v)
    vbar = v[0, :, 0].mean(axis=0)
    np.testing.assert_allclose(y[0, :, 0], np.tile(vbar, (S1, 1)), rtol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.full(S1, math.log(S2)), rtol=1e-14)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse)
    np.testing.assert_allclose(dv[0, :, 0], np.tile(dy[0, :, 0].sum(0) / S2, (S2, 1)), rtol=1e-13)
    assert np.abs(dk).max() < 1e-15
    sc = 1 / math.sqrt(D)
    for i in range(S1):
        w = (v[0, :, 0] - vbar) @ dy[0, i, 0]
        np.testing.assert_allclose(dq[0, i, 0], sc * (w[:, None] * k[0, :, 0]).sum(0) / S2, rtol=1e-12, atol=1e-14)


def test_two_key_logistic_closed_form():
    # two keys: P_0 = σ(a), a = scale q·(k0 − k1); dL/da = P0 (1 − P0) dY·(v0 − v1)
    D, Dv = 3, 2
    q, k, v, dy = make("BSND", 1, 1, 2, 1, 1, D, Dv, 51)
    sc = 0.7
    y, lse = orc.forward(q, k, v, softmax_scale=sc)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, softmax_scale=sc)
    qq, k0, k1, v0, v1, g = q[0, 0, 0], k[0, 0, 0], k[0, 1, 0], v[0, 0, 0], v[0, 1, 0], dy[0, 0, 0]
    a = sc * qq @ (k0 - k1)
    p0 = 1 / (1 + math.exp(-a))
    dLda = p0 * (1 - p0) * g @ (v0 - v1)
    np.testing.assert_allclose(dq[0, 0, 0], sc * dLda * (k0 - k1), rtol=1e-12)
    np.testing.assert_allclose(dk[0, 0, 0], sc * dLda * qq, rtol=1e-12)
    np.testing.assert_allclose(dk[0, 1, 0], -sc * dLda * qq, rtol=1e-12)
    np.testing.assert_allclose(dv[0, 0, 0], p0 * g, rtol=1e-12)
    np.testing.assert_allclose(dv[0, 1, 0], (1 - p0) * g, rtol=1e-12)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rowsum_ds_invariants(case):
    # Σ_j dS_ij = 0 for the exact Y, hence Σ_j dK_j = 0 and Σ_j dV_j = Σ_{i with a key} dY_i
    q, k, v, dy, kw = case_inputs(case, seed=61)
    y, lse = orc.forward(q, k, v, **kw)
    dq, dk, dv, sfmg = orc.backward(q, k, v, dy, y, lse, **kw)
    layout = kw["layout"]
    seq = orc._seq_list(layout, q, k, kw.get("cu_seqlens_q"), kw.get("cu_seqlens_kv"))
    N1 = q.shape[1] if layout == "BNSD" else q.shape[-2]
    N2 = k.shape[1] if layout == "BNSD" else k.shape[-2]
    G = N1 // N2
    mk = dict(mask_mode=kw.get("mask_mode", 0), win_left=kw.get("win_left", -1), win_right=kw.get("win_right", -1))
    for b, rq, rk in seq:
        ok = orc.visible(rq.stop - rq.start, rk.stop - rk.start, **mk)
        has = ok.any(axis=1)
        for n2 in range(N2):
            gk = orc._View(layout, dk).get(b, rk, n2).sum(0)
            assert np.abs(gk).max() < 1e-12
            want = sum(orc._View(layout, dy).get(b, rq, n1)[has].sum(0) for n1 in range(n2 * G, n2 * G + G))
            np.testing.assert_allclose(orc._View(layout, dv).get(b, rk, n2).sum(0), want, rtol=1e-12, atol=1e-12)


def test_empty_rows_and_cols_are_zero():
    # S1 > S2 causal: the first S1 - S2 rows see no key -> lse = +inf, Y = 0, dq = 0
    q, k, v, dy = make("BSND", 1, 6, 4, 2, 2, 3, 3, 71)
    y, lse = orc.forward(q, k, v, mask_mode=1)
    assert np.isinf(lse[0, :, :2]).all() and (y[0, :2] == 0).all()
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, mask_mode=1)
    assert (dq[0, :2] == 0).all()
    # band whose window leaves the last key unseen by every row -> dk = dv = 0 there
    q, k, v, dy = make("BSND", 1, 4, 6, 1, 1, 3, 3, 72)
    y, lse = orc.forward(q, k, v, mask_mode=2, win_left=0, win_right=-1)
    ok = orc.visible(4, 6, 2, 0, -1)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, mask_mode=2, win_left=0, win_right=-1)
    unseen = ~ok.any(axis=0)
    assert unseen.any()
    assert (dk[0, unseen] == 0).all() and (dv[0, unseen] == 0).all()


def test_gqa_equals_repeated_kv():
    S, N1, N2, D, Dv = 7, 6, 2, 4, 3
    G = N1 // N2
    q, k, v, dy = make("BSND", 2, S, S, N1, N2, D, Dv, 81)
    for mk in (dict(), dict(mask_mode=1), dict(mask_mode=2, win_left=2, win_right=1)):
        y, lse = orc.forward(q, k, v, **mk)
        dq, dk, dv, sf = orc.backward(q, k, v, dy, y, lse, **mk)
        kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
        y2, lse2 = orc.forward(q, kr, vr, **mk)
        np.testing.assert_allclose(y2, y, rtol=1e-14, atol=1e-15)
        dq2, dk2, dv2, sf2 = orc.backward(q, kr, vr, dy, y, lse, **mk)
        np.testing.assert_allclose(dq2, dq, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(dk2.reshape(2, S, N2, G, D).sum(3), dk, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(dv2.reshape(2, S, N2, G, Dv).sum(3), dv, rtol=1e-13, atol=1e-14)


def test_tnd_equals_per_sequence_bsnd():
    cu_q, cu_kv = np.array([0, 3, 8, 8, 12]), np.array([0, 5, 9, 11, 15])
    N1, N2, D, Dv = 4, 2, 3, 2
    q, k, v, dy = make("TND", 4, 0, 0, N1, N2, D, Dv, 91, cu_q, cu_kv)
    mk = dict(mask_mode=1, win_left=3, win_right=0)
    y, lse = orc.forward(q, k, v, layout="TND", cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, **mk)
    dq, dk, dv, sf = orc.backward(q, k, v, dy, y, lse, layout="TND", cu_seqlens_q=cu_q,
                                  cu_seqlens_kv=cu_kv, **mk)
    for s in range(4):
        rq, rk = slice(cu_q[s], cu_q[s + 1]), slice(cu_kv[s], cu_kv[s + 1])
        yb, lb = orc.forward(q[None, rq], k[None, rk], v[None, rk], **mk)
        np.testing.assert_allclose(yb[0], y[rq], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lb[0], lse[:, rq], rtol=1e-14)
        gq, gk, gv, gs = orc.backward(q[None, rq], k[None, rk], v[None, rk], dy[None, rq], yb, lb, **mk)
        np.testing.assert_allclose(gq[0], dq[rq], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(gk[0], dk[rk], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(gv[0], dv[rk], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(gs[0], sf[:, rq], rtol=1e-13, atol=1e-14)


def test_sfmg_equals_p_weighted_dp():
    # sfmg_i = dY_i·Y_i = Σ_j P_ij dP_ij when Y = PV (the identity behind rowsum(dS) = 0)
    q, k, v, dy = make("BSND", 1, 6, 6, 2, 2, 3, 4, 101)
    y, lse = orc.forward(q, k, v, mask_mode=1)
    _, _, _, sf = orc.backward(q, k, v, dy, y, lse, mask_mode=1)
    for n in range(2):
        s = torch.tensor(q[0, :, n]) @ torch.tensor(k[0, :, n]).T / math.sqrt(3)
        s = s.masked_fill(~torch.tensor(orc.visible(6, 6, 1, -1, -1)), float("-inf"))
        p = torch.softmax(s, 1).numpy()
        want = (p * (dy[0, :, n] @ v[0, :, n].T)).sum(1)
        np.testing.assert_allclose(sf[0, n], want, rtol=1e-12)


def test_sampled_matches_full():
    cu = np.array([0, 70, 131])
    q, k, v, dy = make("TND", 2, 0, 0, 4, 2, 8, 6, 111, cu, cu)
    mk = dict(layout="TND", cu_seqlens_q=cu, cu_seqlens_kv=cu, mask_mode=1, win_left=20, win_right=0)
    y, lse = orc.forward(q, k, v, **mk)
    lse32 = lse.astype(np.float32)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse32, **mk)
    qr = [(0, 1, 0), (0, 3, 69), (1, 0, 17), (1, 2, 60)]
    kr = [(0, 0, 0), (0, 1, 55), (1, 1, 60), (1, 0, 3)]
    gq, gk, gv = orc.backward_sampled(q, k, v, dy, y, lse32, q_rows=qr, kv_rows=kr, **mk)
    for (s, n, i), g in zip(qr, gq):
        np.testing.assert_allclose(g, dq[cu[s] + i, n], rtol=1e-12, atol=1e-13)
    for (s, n, j), a, b in zip(kr, gk, gv):
        np.testing.assert_allclose(a, dk[cu[s] + j, n], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(b, dv[cu[s] + j, n], rtol=1e-12, atol=1e-13)


def test_argument_checks():
    q, k, v, dy = make("BSND", 1, 3, 3, 3, 2, 2, 2, 1)
    with pytest.raises(ValueError):
        orc.forward(q, k, v)                       # N1 % N2 != 0
    q, k, v, dy = make("BSND", 1, 3, 3, 2, 2, 2, 2, 1)
    with pytest.raises(ValueError):
        orc.forward(q, k, v, mask_mode=0, win_left=2)
    with pytest.raises(ValueError):
        orc.forward(q, k, v, mask_mode=3)
    with pytest.raises(ValueError):
        orc.forward(q, k, v, cu_seqlens_q=np.array([0, 3]), cu_seqlens_kv=np.array([0, 3]))


# ---------------------------------------------------------------------------------------------
# planted mistakes: every pin family must notice a plausible error in the oracle
# ---------------------------------------------------------------------------------------------


def _all_pins_pass():
    try:
        case = [c for c in CASES if c[0] == "causal_s1_lt_s2_gqa"][0]
        q, k, v, dy, kw = case_inputs(case, seed=5)
        if not fd_check(q, k, v, dy, kw, rtol=1e-6):
            return False
        test_exact_golden()
        test_torch_autograd(*TORCH_CASES[1])
        return True
    except AssertionError:
        return False


MUTANTS = {
    "ds_sign": ("_ds", lambda p, dp, sf: p * (dp + sf[:, None])),
    "sfmg_dropped": ("_sfmg", lambda dy, y: np.zeros(dy.shape[0])),
    "dq_no_scale": ("_dq", lambda ds, k, scale: ds @ k),
    "dk_off_by_1pct": ("_dk", lambda ds, q, scale: scale * (ds.T @ q) * 1.01),
    "dv_transposed_p": ("_dv", lambda p, dy: (p.T @ dy)[::-1]),
    "scores_unscaled": ("_scores", lambda q, k, scale: q @ k.T),
    "probs_ignore_mask": ("_probs", lambda s, lse, ok: np.exp(np.minimum(s - lse[:, None], 50.0))),
    "dp_wrong_operand": ("_dp", lambda dy, v: dy @ v.T * 0.5),
}


def test_pins_pass_unmutated():
    assert _all_pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(orc, attr, fn)
    assert not _all_pins_pass(), f"planted mistake {name} went unnoticed"


def test_planted_mask_alignment_is_caught(monkeypatch):
    # a top-left aligned causal mask (j <= i) instead of bottom-right must fail the golden
    real = orc.visible

    def top_left(S1, S2, mask_mode, win_left, win_right):
        ok = real(S1, S2, mask_mode, win_left, win_right)
        if mask_mode == 1:
            ok = np.tril(np.ones((S1, S2), bool))
        return ok

    monkeypatch.setattr(orc, "visible", top_left)
    with pytest.raises(AssertionError):
        test_exact_golden()


def test_planted_gqa_map_is_caught(monkeypatch):
    # an interleaved head map (n1 % N2) instead of contiguous groups (n1 // G) must fail the
    # GQA == repeated-KV pin (np.repeat builds contiguous groups)
    monkeypatch.setattr(orc, "_kv_head", lambda n1, N1, N2: n1 % N2)
    with pytest.raises(AssertionError):
        test_gqa_equals_repeated_kv()


# ---------------------------------------------------------------------------------------------
# (max, sum) statistics form of the forward (LaserAttentionGrad / FusedFloydAttentionGrad pages)
# ---------------------------------------------------------------------------------------------


def test_stats_give_the_logsumexp_of_the_visible_scores():
    from scipy.special import logsumexp

    rng = np.random.default_rng(11)
    S1, S2, D = 9, 13, 5
    q, k, v = rng.normal(size=(S1, D)), rng.normal(size=(S2, D)), rng.normal(size=(S2, 3))
    ok = orc.visible(S1, S2, 2, 3, 1)
    ok[4, :] = False                                  # a row with no visible key
    m, l = orc.forward_stats_head(q, k, v, 0.37, ok)
    lse = orc.lse_from_stats(m, l)
    s = 0.37 * q @ k.T
    for i in range(S1):
        want = logsumexp(s[i][ok[i]]) if ok[i].any() else np.inf
        assert lse[i] == pytest.approx(want, rel=1e-13, abs=1e-13) if np.isfinite(want) else lse[i] == np.inf
    # and the same lse as the forward itself produces
    _, lse_fwd = orc.forward_head(q, k, v, 0.37, ok)
    np.testing.assert_allclose(lse, lse_fwd, rtol=1e-14)


def test_stats_adapter_does_not_need_the_true_maximum():
    # (c, Σ exp(S − c)) for any shift c describes the same softmax: lse must not depend on c
    rng = np.random.default_rng(12)
    s = rng.normal(size=(6, 10)) * 3
    ref = orc.lse_from_stats(s.max(axis=1), np.exp(s - s.max(axis=1, keepdims=True)).sum(axis=1))
    for c in (0.0, -5.0, 7.5):
        np.testing.assert_allclose(orc.lse_from_stats(np.full(6, c), np.exp(s - c).sum(axis=1)), ref, rtol=1e-13)
    assert orc.lse_from_stats(np.array([-np.inf]), np.array([0.0]))[0] == np.inf


# ---------------------------------------------------------------------------------------------
# seqused_q / seqused_kv and sinks (optional inputs of [FAG] §2.1 / §4.2; readings in the oracle)
# ---------------------------------------------------------------------------------------------

SEQUSED_CASES = [
    # name, layout, B, S1, S2, N1, N2, kw, cu_q, cu_kv, seqused_q, seqused_kv
    ("tnd_causal_used", "TND", 3, 0, 0, 4, 2, dict(mask_mode=1), np.array([0, 4, 9, 12]), np.array([0, 5, 9, 13]),
     np.array([3, 5, 0]), np.array([4, 2, 3])),
    ("tnd_window_q_only", "TND", 2, 0, 0, 2, 1, dict(mask_mode=1, win_left=1, win_right=0), np.array([0, 5, 9]),
     np.array([0, 5, 9]), np.array([4, 2]), None),
    ("bsnd_dense_used", "BSND", 2, 5, 6, 2, 2, dict(), None, None, np.array([5, 2]), np.array([3, 6])),
    ("bnsd_band_kv_only", "BNSD", 2, 5, 5, 2, 1, dict(mask_mode=2, win_left=1, win_right=2), None, None, None,
     np.array([4, 1])),
]


def seqused_inputs(case, seed=13):
    name, layout, B, S1, S2, N1, N2, kw, cu_q, cu_kv, uq, ukv = case
    q, k, v, dy = make(layout, B, S1, S2, N1, N2, 3, 2, seed, cu_q, cu_kv)
    kw = dict(kw, layout=layout, seqused_q=uq, seqused_kv=ukv)
    if layout == "TND":
        kw.update(cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv)
    return q, k, v, dy, kw


@pytest.mark.parametrize("case", SEQUSED_CASES, ids=[c[0] for c in SEQUSED_CASES])
def test_seqused_finite_differences(case):
    # rows past seqused take no part in L, so their derivative (and the oracle's gradient) is 0
    q, k, v, dy, kw = seqused_inputs(case)
    assert fd_check(q, k, v, dy, kw)


def _truncate(x, layout, cu, used, axis_rows):
    """The used rows of every sequence only: TND rows re-packed, BSND/BNSD per batch."""
    if layout == "TND":
        return np.concatenate([x[cu[s]:cu[s] + used[s]] for s in range(len(cu) - 1)])
    return [np.take(x[b:b + 1], np.arange(used[b]), axis=axis_rows) for b in range(x.shape[0])]


@pytest.mark.parametrize("case", SEQUSED_CASES, ids=[c[0] for c in SEQUSED_CASES])
def test_seqused_equals_truncated_sequences(case):
    name, layout, B, S1, S2, N1, N2, mk, cu_q, cu_kv, uq, ukv = case
    q, k, v, dy, kw = seqused_inputs(case, seed=17)
    y, lse = orc.forward(q, k, v, **kw)
    dq, dk, dv, sf = orc.backward(q, k, v, dy, y, lse, **kw)
    nq = len(cu_q) - 1 if layout == "TND" else B
    uq_ = uq if uq is not None else (np.diff(cu_q) if layout == "TND" else np.full(B, S1))
    uk_ = ukv if ukv is not None else (np.diff(cu_kv) if layout == "TND" else np.full(B, S2))
    ax = 1 if layout == "BSND" else 2
    if layout == "TND":
        tq, tdy, ty = (_truncate(x, layout, cu_q, uq_, 0) for x in (q, dy, y))
        tk, tv = (_truncate(x, layout, cu_kv, uk_, 0) for x in (k, v))
        tcq, tck = np.concatenate([[0], np.cumsum(uq_)]), np.concatenate([[0], np.cumsum(uk_)])
        tkw = dict(mk, layout="TND", cu_seqlens_q=tcq, cu_seqlens_kv=tck)
        y2, lse2 = orc.forward(tq, tk, tv, **tkw)
        g = orc.backward(tq, tk, tv, tdy, y2, lse2, **tkw)
        np.testing.assert_allclose(_truncate(y, layout, cu_q, uq_, 0), y2, rtol=1e-14, atol=1e-15)
        for got, want, cu, u in ((dq, g[0], cu_q, uq_), (dk, g[1], cu_kv, uk_), (dv, g[2], cu_kv, uk_)):
            np.testing.assert_allclose(_truncate(got, layout, cu, u, 0), want, rtol=1e-13, atol=1e-14)
        # and the rows past seqused: zero gradients, +inf lse, Y = 0
        for s in range(nq):
            assert (dq[cu_q[s] + uq_[s]:cu_q[s + 1]] == 0).all() and (y[cu_q[s] + uq_[s]:cu_q[s + 1]] == 0).all()
            assert np.isinf(lse[:, cu_q[s] + uq_[s]:cu_q[s + 1]]).all()
            assert (dk[cu_kv[s] + uk_[s]:cu_kv[s + 1]] == 0).all() and (dv[cu_kv[s] + uk_[s]:cu_kv[s + 1]] == 0).all()
    else:
        for b in range(B):
            pick = lambda x, n: np.take(x[b:b + 1], np.arange(n), axis=ax)
            tq, tdy, tk, tv = pick(q, uq_[b]), pick(dy, uq_[b]), pick(k, uk_[b]), pick(v, uk_[b])
            tkw = dict(mk, layout=layout)
            y2, lse2 = orc.forward(tq, tk, tv, **tkw)
            g = orc.backward(tq, tk, tv, tdy, y2, lse2, **tkw)
            np.testing.assert_allclose(pick(y, uq_[b]), y2, rtol=1e-14, atol=1e-15)
            np.testing.assert_allclose(pick(dq, uq_[b]), g[0], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(pick(dk, uk_[b]), g[1], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(pick(dv, uk_[b]), g[2], rtol=1e-13, atol=1e-14)
            rest_q = lambda x: np.take(x[b:b + 1], np.arange(uq_[b], S1), axis=ax)
            rest_k = lambda x: np.take(x[b:b + 1], np.arange(uk_[b], S2), axis=ax)
            assert (rest_q(dq) == 0).all() and (rest_k(dk) == 0).all() and (rest_k(dv) == 0).all()


def test_seqused_rows_are_never_read():
    # anything in the rows past seqused (here NaN) leaves the used rows' results unchanged
    case = SEQUSED_CASES[0]
    q, k, v, dy, kw = seqused_inputs(case, seed=19)
    y, lse = orc.forward(q, k, v, **kw)
    ref = orc.backward(q, k, v, dy, y, lse, **kw)
    cu_q, cu_kv, uq, ukv = case[8], case[9], case[10], case[11]
    for s in range(len(cu_q) - 1):
        for x in (q, dy, y):
            x[cu_q[s] + uq[s]:cu_q[s + 1]] = np.nan
        for x in (k, v):
            x[cu_kv[s] + ukv[s]:cu_kv[s + 1]] = np.nan
    got = orc.backward(q, k, v, dy, y, lse, **kw)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)


def test_seqused_bounds_are_checked():
    q, k, v, dy, kw = seqused_inputs(SEQUSED_CASES[0])
    with pytest.raises(ValueError):
        orc.forward(q, k, v, **dict(kw, seqused_q=np.array([5, 5, 0])))   # 5 > span 4 of sequence 0
    with pytest.raises(ValueError):
        orc.forward(q, k, v, **dict(kw, seqused_kv=np.array([1, 1])))     # one entry per sequence


def test_planted_seqused_alignment_is_caught(monkeypatch):
    # a mask aligned to the stored span instead of the used lengths must fail the truncation pin
    real = orc._seq_list

    def span_aligned(layout, q, k, cu_q, cu_kv, seqused_q=None, seqused_kv=None):
        return real(layout, q, k, cu_q, cu_kv, None, None) if seqused_q is not None or seqused_kv is not None \
            else real(layout, q, k, cu_q, cu_kv)

    monkeypatch.setattr(orc, "_seq_list", span_aligned)
    with pytest.raises(AssertionError):
        test_seqused_equals_truncated_sequences(SEQUSED_CASES[0])


SINK_CASES = [
    ("dense", "BSND", 1, 5, 5, 2, 2, 3, 2, dict(), None, None),
    ("causal_gqa_empty_rows", "BSND", 1, 6, 4, 4, 2, 3, 2, dict(mask_mode=1), None, None),
    ("tnd_window", "TND", 2, 0, 0, 2, 2, 2, 3, dict(mask_mode=1, win_left=1, win_right=0),
     np.array([0, 5, 8]), np.array([0, 5, 8])),
]


def _sinks(N1, seed):
    return np.random.default_rng(seed).standard_normal(N1) * 1.5


@pytest.mark.parametrize("case", SINK_CASES, ids=[c[0] for c in SINK_CASES])
def test_sinks_finite_differences(case):
    # L = Σ dY ⊙ Y(q, k, v) of the forward with sink logits; the backward from that forward's lse
    # must be its derivative (the sink only enters through lse)
    q, k, v, dy, kw = case_inputs(case, seed=23)
    N1 = case[5]
    sk = _sinks(N1, 3)
    y, lse = orc.forward(q, k, v, sinks=sk, **kw)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, **kw)
    f = lambda: float((dy * orc.forward(q, k, v, sinks=sk, **kw)[0]).sum())
    for got, x in ((dq, q), (dk, k), (dv, v)):
        ref = fd_grad(x, f)
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6 * max(1.0, np.abs(ref).max()))


def test_sinks_closed_forms():
    # one query, one key: lse = ln(e^s + e^sink), Y = v·σ(s − sink); a row with no key: lse = sink
    rng = np.random.default_rng(29)
    q, k, v = rng.normal(size=(1, 1, 1, 3)), rng.normal(size=(1, 1, 1, 3)), rng.normal(size=(1, 1, 1, 2))
    sink = np.array([0.4])
    y, lse = orc.forward(q, k, v, softmax_scale=0.5, sinks=sink)
    s = 0.5 * float(q[0, 0, 0] @ k[0, 0, 0])
    assert lse[0, 0, 0] == pytest.approx(math.log(math.exp(s) + math.exp(0.4)), rel=1e-14)
    np.testing.assert_allclose(y[0, 0, 0], v[0, 0, 0] / (1 + math.exp(0.4 - s)), rtol=1e-14)
    q, k, v, dy = make("BSND", 1, 6, 4, 2, 2, 3, 3, 33)
    y, lse = orc.forward(q, k, v, mask_mode=1, sinks=np.array([0.25, -1.0]))
    assert (lse[0, 0, :2] == 0.25).all() and (lse[0, 1, :2] == -1.0).all() and (y[0, :2] == 0).all()


def test_sinks_take_the_missing_row_mass_and_vanish_at_minus_infinity():
    q, k, v, dy = make("BSND", 1, 7, 7, 2, 1, 3, 2, 37)
    sk = np.array([0.3, 2.0])
    y, lse = orc.forward(q, k, v, mask_mode=1, sinks=sk)
    ok = orc.visible(7, 7, 1, -1, -1)
    for n in range(2):
        p = orc._probs(orc._scores(q[0, :, n], k[0, :, 0], 1 / math.sqrt(3)), lse[0, n], ok)
        np.testing.assert_allclose(p.sum(1), 1 - np.exp(sk[n] - lse[0, n]), rtol=1e-13)
    y0, lse0 = orc.forward(q, k, v, mask_mode=1)
    y1, lse1 = orc.forward(q, k, v, mask_mode=1, sinks=np.array([-np.inf, -np.inf]))
    np.testing.assert_array_equal(lse1, lse0)
    np.testing.assert_array_equal(y1, y0)


def test_sinks_against_torch_autograd():
    # softmax over [S, sink] with the sink column dropped from P·V, differentiated by torch
    q, k, v, dy = make("BSND", 1, 6, 8, 2, 1, 4, 3, 41)
    sk = np.array([0.7, -0.2])
    ok = orc.visible(6, 8, 1, -1, -1)
    y, lse = orc.forward(q, k, v, mask_mode=1, sinks=sk)
    dq, dk, dv, _ = orc.backward(q, k, v, dy, y, lse, mask_mode=1)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    tot = 0
    for n in range(2):
        s = tq[0, :, n] @ tk[0, :, 0].T / math.sqrt(4)
        s = s.masked_fill(~torch.tensor(ok), float("-inf"))
        full = torch.cat([s, torch.full((6, 1), float(sk[n]), dtype=s.dtype)], dim=1)
        p = torch.softmax(full, dim=1)[:, :-1]
        tot = tot + (torch.tensor(dy[0, :, n]) * (p @ tv[0, :, 0])).sum()
    tot.backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_planted_sink_dropped_from_lse_is_caught(monkeypatch):
    real = orc.forward_head
    monkeypatch.setattr(orc, "forward_head", lambda q, k, v, scale, ok, sink=None: real(q, k, v, scale, ok, None)
                        if sink is None else (real(q, k, v, scale, ok, sink)[0], real(q, k, v, scale, ok, None)[1]))
    with pytest.raises(AssertionError):
        test_sinks_finite_differences(SINK_CASES[1])
