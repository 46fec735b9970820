"""Pins of the fp64 oracle against things other than itself.

Each test ties one part of the oracle to an independent fact: a closed form
worked out by hand, a library routine (PyTorch scaled-dot-product attention in
float64), finite differences of the forward, an invariant that holds by the
mathematics (rows of P sum to one, documents attend independently, ...), or the
scalar triple-loop restatement on tiny shapes.
"""

import math

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from oracle.brute_force import _live, brute_attention

CAPS = [("none", 0.0, 0.0, 0.0), ("tanh", 5.0, 0.0, 0.0), ("soft_sign", 3.0, 0.0, 0.0),
        ("alsc", 4.0, 2.0, 0.5)]


def _rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def _inputs(rng, B, L, Hq, Hkv, D, temp=True, seg=False, bounds=False, scale=1.0):
    q = _rand((B, L, Hq, D), rng, scale)
    k = _rand((B, L, Hkv, D), rng, scale)
    v = _rand((B, L, Hkv, D), rng)
    do = _rand((B, L, Hq, D), rng)
    t = rng.uniform(0.5, 1.5, size=(B, L)) if temp else None
    sg = None
    if seg:
        sg = np.zeros((B, L), np.int32)
        for b in range(B):
            cuts = np.sort(rng.choice(np.arange(1, L), size=min(3, L - 1), replace=False))
            for c in cuts:
                sg[b, c:] += 1
    bd = None
    if bounds:
        bd = np.zeros((B, 4), np.int32)
        for b in range(B):
            hu = int(rng.integers(1, L - 1))
            cu = int(min(L, hu + rng.integers(1, 4)))
            bd[b] = (0, hu, hu, cu)
    return q, k, v, do, t, sg, bd


# ---------------------------------------------------------------------------
# Closed forms of the cap functions (worked out by hand, not by the oracle).
# ALSC forward cap*(sigma(alpha(s/cap+beta)) - sigma(ab)) / (sigma(ab)(1-sigma(ab)) + 1e-12):
#   * at s = 0 the numerator vanishes exactly;
#   * slope at 0 = alpha * sigma(1-sigma)/(sigma(1-sigma)+1e-12), i.e. alpha up to 1e-11;
#   * s -> +inf: cap (1 - sigma)/(sigma(1-sigma)) = cap/sigma = cap (1 + e^{-ab});
#   * s -> -inf: -cap sigma/(sigma(1-sigma)) = -cap/(1-sigma) = -cap (1 + e^{ab}).
# With cap = 30, alpha = 2, beta = 0.5: +41.0363832351, -111.5484548537.
# ---------------------------------------------------------------------------

def test_alsc_closed_forms():
    cfg = orc.OracleConfig(sm_scale=1.0, cap_method="alsc", cap=30.0, alpha=2.0, beta=0.5)
    assert orc.cap_forward(np.array([0.0]), cfg)[0] == 0.0
    h = 1e-5
    slope = (orc.cap_forward(np.array([h]), cfg)[0] - orc.cap_forward(np.array([-h]), cfg)[0]) / (2 * h)
    assert abs(slope - 2.0) < 1e-8
    assert abs(orc.cap_derivative(np.array([0.0]), cfg)[0] - 2.0) < 1e-9
    assert abs(orc.cap_forward(np.array([1e6]), cfg)[0] - 41.0363832351) < 1e-6
    assert abs(orc.cap_forward(np.array([-1e6]), cfg)[0] + 111.5484548537) < 1e-6
    # The printed gradient (alpha/cap) s(1-s)/denom is this slope divided by cap:
    # 2/30 = 0.0666667 at alpha = 2; 4/30 = 0.1333333 at alpha = 4 (module docstring reading).
    cfg4 = orc.OracleConfig(sm_scale=1.0, cap_method="alsc", cap=30.0, alpha=4.0, beta=0.5)
    slope4 = (orc.cap_forward(np.array([h]), cfg4)[0] - orc.cap_forward(np.array([-h]), cfg4)[0]) / (2 * h)
    assert abs(slope4 - 4.0) < 1e-7
    assert abs(slope / 30.0 - 0.0666667) < 1e-6 and abs(slope4 / 30.0 - 0.1333333) < 1e-6


def test_tanh_and_soft_sign_closed_forms():
    tcfg = orc.OracleConfig(sm_scale=1.0, cap_method="tanh", cap=50.0)
    assert orc.cap_derivative(np.array([0.0]), tcfg)[0] == 1.0
    assert abs(orc.cap_forward(np.array([1e4]), tcfg)[0] - 50.0) < 1e-12
    # tanh(1) = 0.7615941559557649
    assert abs(orc.cap_forward(np.array([50.0]), tcfg)[0] - 50 * 0.7615941559557649) < 1e-12
    scfg = orc.OracleConfig(sm_scale=1.0, cap_method="soft_sign", cap=20.0)
    assert abs(orc.cap_forward(np.array([1e12]), scfg)[0] - 20.0) < 1e-9
    assert abs(orc.cap_forward(np.array([-1e12]), scfg)[0] + 20.0) < 1e-9
    assert orc.cap_forward(np.array([20.0]), scfg)[0] == 10.0  # 20 / (1 + 1)
    assert orc.cap_derivative(np.array([20.0]), scfg)[0] == 0.25  # 1 / (1 + 1)^2
    # cap <= 0 behaves as no cap
    zcfg = orc.OracleConfig(sm_scale=1.0, cap_method="tanh", cap=0.0)
    x = np.linspace(-5, 5, 11)
    assert np.array_equal(orc.cap_forward(x, zcfg), x)


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
def test_cap_derivative_matches_finite_differences(method, cap, alpha, beta):
    cfg = orc.OracleConfig(sm_scale=1.0, cap_method=method, cap=cap, alpha=alpha, beta=beta)
    s = np.linspace(-12.0, 12.0, 97) + 0.0123
    h = 1e-6
    fd = (orc.cap_forward(s + h, cfg) - orc.cap_forward(s - h, cfg)) / (2 * h)
    np.testing.assert_allclose(orc.cap_derivative(s, cfg), fd, rtol=1e-7, atol=1e-8)


# ---------------------------------------------------------------------------
# Library special case: no cap, temperature 1 is scaled-dot-product attention.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("G", [1, 2])
def test_matches_torch_sdpa(causal, G):
    rng = np.random.default_rng(3)
    B, L, Hkv, D = 2, 37, 2, 16
    Hq = Hkv * G
    q, k, v, do, _, _, _ = _inputs(rng, B, L, Hq, Hkv, D, temp=False)
    cfg = orc.OracleConfig(sm_scale=0.3, causal=causal)
    O, LSE, _, _ = orc.forward(q, k, v, None, None, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, None, None, None, O, LSE, do, cfg)

    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_(True)
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_(True)
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_(True)
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, is_causal=causal, scale=0.3)
    (out * torch.tensor(do).permute(0, 2, 1, 3)).sum().backward()
    np.testing.assert_allclose(O, out.detach().permute(0, 2, 1, 3).numpy(), atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    # LSE against torch.logsumexp of the library's own causal mask
    s = 0.3 * torch.einsum("bhid,bhjd->bhij", tq.detach(), kk.detach())
    if causal:
        s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(LSE, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


# ---------------------------------------------------------------------------
# Finite differences of L = sum(O * dO) + (z/2) sum LSE^2 pin the backward.
# ---------------------------------------------------------------------------

MASKS = [dict(causal=False, window_len=0, seg=False, bounds=False),
         dict(causal=True, window_len=3, seg=False, bounds=False),
         dict(causal=True, window_len=0, seg=True, bounds=False),
         dict(causal=False, window_len=0, seg=False, bounds=True)]


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("mask", range(len(MASKS)))
@pytest.mark.parametrize("z", [0.0, 0.05])
def test_gradients_match_finite_differences(method, cap, alpha, beta, mask, z):
    mk = MASKS[mask]
    rng = np.random.default_rng(11 + mask)
    B, L, Hq, Hkv, D = 1, 7, 2, 1, 3
    q, k, v, do, t, sg, bd = _inputs(rng, B, L, Hq, Hkv, D, temp=True, seg=mk["seg"],
                                     bounds=mk["bounds"], scale=1.5)
    cfg = orc.OracleConfig(sm_scale=0.7, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=z)
    O, LSE, _, _ = orc.forward(q, k, v, t, sg, bd, cfg)
    grads = orc.backward(q, k, v, t, sg, bd, O, LSE, do, cfg)[:3]
    h = 1e-6
    for x, gx in zip((q, k, v), grads):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + h
            lp = orc.loss(q, k, v, t, sg, bd, do, cfg)
            x[idx] = x0 - h
            lm = orc.loss(q, k, v, t, sg, bd, do, cfg)
            x[idx] = x0
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(gx - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, err


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("mask", [1, 3])
def test_lse_gradient_matches_finite_differences(method, cap, alpha, beta, mask):
    # an upstream gradient of the returned LSE: L = sum O dO + sum LSE dLSE (+ z-loss)
    mk = MASKS[mask]
    rng = np.random.default_rng(23 + mask)
    B, L, Hq, Hkv, D = 1, 7, 2, 1, 3
    q, k, v, do, t, sg, bd = _inputs(rng, B, L, Hq, Hkv, D, seg=mk["seg"], bounds=mk["bounds"],
                                     scale=1.5)
    dlse = rng.standard_normal((B, Hq, L))
    cfg = orc.OracleConfig(sm_scale=0.7, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.05)
    O, LSE, _, _ = orc.forward(q, k, v, t, sg, bd, cfg)
    grads = orc.backward(q, k, v, t, sg, bd, O, LSE, do, cfg, dLSE=dlse)[:3]
    dtemp = orc.backward_dtemp(q, k, v, t, sg, bd, O, LSE, do, cfg, dLSE=dlse)
    h = 1e-6
    for x, gx in zip((q, k, v, t), (*grads, dtemp)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + h
            lp = orc.loss(q, k, v, t, sg, bd, do, cfg, dLSE=dlse)
            x[idx] = x0 - h
            lm = orc.loss(q, k, v, t, sg, bd, do, cfg, dLSE=dlse)
            x[idx] = x0
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(gx - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, err


@pytest.mark.parametrize("causal", [False, True])
def test_lse_gradient_matches_torch_logsumexp(causal):
    # no cap, temperature 1: LSE = logsumexp of the scaled scores; float64 autograd
    rng = np.random.default_rng(29)
    B, L, H, D = 1, 19, 2, 8
    q, k, v, do, _, _, _ = _inputs(rng, B, L, H, H, D, temp=False)
    dlse = rng.standard_normal((B, H, L))
    cfg = orc.OracleConfig(sm_scale=0.4, causal=causal)
    O, LSE, _, _ = orc.forward(q, k, v, None, None, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, None, None, None, O, LSE, do, cfg, dLSE=dlse)
    tq, tk, tv = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
    sc = 0.4 * tq @ tk.transpose(-1, -2)
    if causal:
        sc = sc.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(sc, dim=-1)
    out = torch.softmax(sc, dim=-1) @ tv
    ((out * torch.tensor(do).permute(0, 2, 1, 3)).sum() + (lse * torch.tensor(dlse)).sum()).backward()
    np.testing.assert_allclose(dQ, tq.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
def test_gradients_match_finite_differences_nonpositive_temperature(method, cap, alpha, beta):
    rng = np.random.default_rng(17)
    B, L, Hq, Hkv, D = 1, 7, 2, 1, 3
    q, k, v, do, _, _, _ = _inputs(rng, B, L, Hq, Hkv, D, scale=1.5)
    t = np.array([[-1.1, 0.0, 0.6, -0.3, 0.0, 1.2, -0.7]])
    cfg = orc.OracleConfig(sm_scale=0.7, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=True, window_len=4, z_loss_weight=0.05)
    O, LSE, _, _ = orc.forward(q, k, v, t, None, None, cfg)
    grads = orc.backward(q, k, v, t, None, None, O, LSE, do, cfg)[:3]
    h = 1e-6
    for x, gx in zip((q, k, v), grads):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + h
            lp = orc.loss(q, k, v, t, None, None, do, cfg)
            x[idx] = x0 - h
            lm = orc.loss(q, k, v, t, None, None, do, cfg)
            x[idx] = x0
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(gx - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, err


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("mask", range(len(MASKS)))
@pytest.mark.parametrize("z", [0.0, 0.05])
def test_dtemp_matches_finite_differences(method, cap, alpha, beta, mask, z):
    # dL/dtemp (shared by both query heads of a row) against central differences
    mk = MASKS[mask]
    rng = np.random.default_rng(211 + mask)
    B, L, Hq, Hkv, D = 2, 7, 2, 1, 3
    q, k, v, do, t, sg, bd = _inputs(rng, B, L, Hq, Hkv, D, temp=True, seg=mk["seg"],
                                     bounds=mk["bounds"], scale=1.5)
    cfg = orc.OracleConfig(sm_scale=0.7, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=z)
    O, LSE, _, _ = orc.forward(q, k, v, t, sg, bd, cfg)
    dtemp = orc.backward_dtemp(q, k, v, t, sg, bd, O, LSE, do, cfg)
    h = 1e-6
    fd = np.zeros_like(t, dtype=np.float64)
    for b in range(B):
        for i in range(L):
            t0 = t[b, i]
            t[b, i] = t0 + h
            lp = orc.loss(q, k, v, t, sg, bd, do, cfg)
            t[b, i] = t0 - h
            lm = orc.loss(q, k, v, t, sg, bd, do, cfg)
            t[b, i] = t0
            fd[b, i] = (lp - lm) / (2 * h)
    err = np.linalg.norm(dtemp - fd) / max(np.linalg.norm(fd), 1e-30)
    assert err < 1e-6, err
    # fully masked rows contribute nothing
    dead = ~np.isfinite(LSE).any(axis=1)
    assert np.all(dtemp[dead] == 0.0)


# ---------------------------------------------------------------------------
# Brute force on tiny shapes: catches indexing / blocking / head-mapping bugs.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("mask", range(len(MASKS)))
def test_dense_matches_brute_force(method, cap, alpha, beta, mask, monkeypatch):
    monkeypatch.setattr(orc, "ROW_BLOCK", 5)  # exercise several row blocks and a ragged one
    mk = MASKS[mask]
    rng = np.random.default_rng(100 + mask)
    B, L, Hq, Hkv, D = 2, 13, 4, 2, 5
    q, k, v, do, t, sg, bd = _inputs(rng, B, L, Hq, Hkv, D, seg=mk["seg"], bounds=mk["bounds"])
    cfg = orc.OracleConfig(sm_scale=0.45, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.03)
    O, LSE, Mx, Lx = orc.forward(q, k, v, t, sg, bd, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, sg, bd, O, LSE, do, cfg)
    p = dict(sm_scale=0.45, cap_method=method, cap=cap, alpha=alpha, beta=beta,
             causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.03)
    ref = brute_attention(q.tolist(), k.tolist(), v.tolist(), do.tolist(),
                          None if t is None else t.tolist(), None if sg is None else sg.tolist(),
                          None if bd is None else bd.tolist(), p)
    _compare_with_brute(O, LSE, Mx, Lx, dQ, dK, dV, ref)


def _compare_with_brute(O, LSE, Mx, Lx, dQ, dK, dV, ref):
    np.testing.assert_allclose(O, np.array(ref["O"]), rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.isinf(LSE), np.isinf(np.array(ref["LSE"])))
    fin = np.isfinite(LSE)
    np.testing.assert_allclose(LSE[fin], np.array(ref["LSE"])[fin], rtol=1e-12, atol=1e-12)
    # the softmax residuals: m is the largest LIVE tempered logit, l = sum exp(t - m)
    # over live keys; a row with no live key has m = -inf, l = 0
    rm, rl = np.array(ref["m"]), np.array(ref["l"])
    assert np.array_equal(np.isneginf(Mx), np.isneginf(rm)) and np.array_equal(fin, np.isfinite(rm))
    np.testing.assert_allclose(Mx[fin], rm[fin], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Lx, rl, rtol=1e-12, atol=1e-12)
    assert np.all(Lx[~fin] == 0.0)
    for a, r in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
        np.testing.assert_allclose(a, np.array(ref[r]), rtol=1e-10, atol=1e-11)


# Temperatures that are negative on some rows and exactly zero on others (the
# forward then takes the row's minimum capped score as its largest logit, or
# a uniform softmax over the live keys).
@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("mask", [0, 1, 3])
def test_dense_matches_brute_force_nonpositive_temperature(method, cap, alpha, beta, mask,
                                                           monkeypatch):
    monkeypatch.setattr(orc, "ROW_BLOCK", 4)
    mk = MASKS[mask]
    rng = np.random.default_rng(300 + mask)
    B, L, Hq, Hkv, D = 2, 11, 4, 2, 5
    q, k, v, do, _, sg, bd = _inputs(rng, B, L, Hq, Hkv, D, seg=mk["seg"], bounds=mk["bounds"])
    t = rng.choice([-1.3, -0.4, 0.0, 0.8], size=(B, L))
    cfg = orc.OracleConfig(sm_scale=0.45, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.03)
    O, LSE, Mx, Lx = orc.forward(q, k, v, t, sg, bd, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, sg, bd, O, LSE, do, cfg)
    p = dict(sm_scale=0.45, cap_method=method, cap=cap, alpha=alpha, beta=beta,
             causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.03)
    ref = brute_attention(q.tolist(), k.tolist(), v.tolist(), do.tolist(), t.tolist(),
                          None if sg is None else sg.tolist(), None if bd is None else bd.tolist(), p)
    _compare_with_brute(O, LSE, Mx, Lx, dQ, dK, dV, ref)


def test_residuals_of_a_hand_worked_row():
    """One query against three keys with scores worked out by hand.

    D = 1, q = 1, k = (2, 5, -1), sm_scale = 1, no cap, temperature 0.5, and a
    ranker mask that hides key 1 (history [0, 1), candidates [2, 3), query 2 is
    a candidate: it sees history key 0 and itself, key 2).  Tempered logits:
    t = (1, 2.5, -0.5); key 1 has the largest logit but is masked, so
    m = 1 (not 2.5), l = 1 + e^-1.5, LSE = 1 + ln(1 + e^-1.5), and
    O = (v0 + e^-1.5 v2) / (1 + e^-1.5).
    """
    q = np.zeros((1, 3, 1, 1))
    q[0, 2, 0, 0] = 1.0
    k = np.array([2.0, 5.0, -1.0]).reshape(1, 3, 1, 1)
    v = np.array([3.0, -7.0, 11.0]).reshape(1, 3, 1, 1)
    temp = np.full((1, 3), 0.5)
    bounds = np.array([[0, 1, 2, 3]], np.int32)
    cfg = orc.OracleConfig(sm_scale=1.0)
    O, LSE, Mx, Lx = orc.forward(q, k, v, temp, None, bounds, cfg)
    e = math.exp(-1.5)
    assert Mx[0, 0, 2] == 1.0
    assert abs(Lx[0, 0, 2] - (1.0 + e)) < 1e-15
    assert abs(LSE[0, 0, 2] - (1.0 + math.log1p(e))) < 1e-15
    assert abs(O[0, 2, 0, 0] - (3.0 + 11.0 * e) / (1.0 + e)) < 1e-14
    # query 1 is outside history and candidates: fully masked
    assert Mx[0, 0, 1] == -math.inf and Lx[0, 0, 1] == 0.0 and LSE[0, 0, 1] == -math.inf
    # query 0 (history) sees key 0 only: m = t = 0 (q_0 = 0), l = 1
    assert Mx[0, 0, 0] == 0.0 and Lx[0, 0, 0] == 1.0 and O[0, 0, 0, 0] == 3.0
    # a negative temperature flips which key wins: temp = -0.5 gives t = (-1, ., 0.5)
    temp[0, 2] = -0.5
    O, LSE, Mx, Lx = orc.forward(q, k, v, temp, None, bounds, cfg)
    assert Mx[0, 0, 2] == 0.5 and abs(Lx[0, 0, 2] - (1.0 + e)) < 1e-15
    assert abs(O[0, 2, 0, 0] - (11.0 + 3.0 * e) / (1.0 + e)) < 1e-14


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
def test_zero_temperature_is_a_uniform_softmax(method, cap, alpha, beta):
    """temp_i = 0 makes every live logit 0: P is uniform over the live keys, so
    O is their mean value, m = 0, l = the live count and LSE = ln(count)."""
    rng = np.random.default_rng(41)
    B, L, H, D = 1, 9, 2, 4
    q, k, v, do, _, _, _ = _inputs(rng, B, L, H, H, D)
    t = np.zeros((B, L))
    cfg = orc.OracleConfig(sm_scale=0.7, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=True)
    O, LSE, Mx, Lx = orc.forward(q, k, v, t, None, None, cfg)
    for h in range(H):
        for i in range(L):
            n = i + 1
            np.testing.assert_allclose(O[0, i, h], v[0, :n, h].mean(axis=0), rtol=1e-13, atol=1e-14)
            assert Mx[0, h, i] == 0.0 and Lx[0, h, i] == n
            assert abs(LSE[0, h, i] - math.log(n)) < 1e-14


# ---------------------------------------------------------------------------
# Invariants.
# ---------------------------------------------------------------------------

def test_probabilities_sum_to_one_and_masked_entries_are_zero():
    rng = np.random.default_rng(5)
    L, D = 40, 8
    q, k, v = rng.standard_normal((L, D)), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    bounds = (0, 17, 17, 23)
    cfg = orc.OracleConfig(sm_scale=0.5, cap_method="alsc", cap=30.0, alpha=2.0, beta=0.5)
    M = orc.mask_matrix(L, cfg, None, bounds)
    O, lse, m, l, P, s = orc._forward_block(q, k, v, np.ones(L), M, cfg)
    live = M.any(axis=1)
    np.testing.assert_allclose(P[live].sum(axis=1), 1.0, atol=1e-14)
    assert np.all(P[~M] == 0.0)
    assert np.all(np.isneginf(lse[~live])) and np.all(l[~live] == 0) and np.all(O[~live] == 0)
    do = rng.standard_normal((L, D))
    delta = np.einsum("id,id->i", O, do)
    dq, dk, dv = orc._backward_block(q, k, v, do, np.ones(L), M, lse, delta, cfg)
    assert np.all(dq[~live] == 0.0)
    # rows 23.. are outside history and candidates: no gradient flows through them
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def test_large_tanh_cap_is_uncapped():
    rng = np.random.default_rng(6)
    q, k, v, do, t, _, _ = _inputs(rng, 1, 30, 2, 2, 8)
    a = orc.OracleConfig(sm_scale=0.4, cap_method="tanh", cap=1e6, causal=True)
    b = orc.OracleConfig(sm_scale=0.4, causal=True)
    Oa, La, _, _ = orc.forward(q, k, v, t, None, None, a)
    Ob, Lb, _, _ = orc.forward(q, k, v, t, None, None, b)
    assert np.max(np.abs(Oa - Ob)) < 1e-9 and np.max(np.abs(La - Lb)) < 1e-9


def test_constant_temperature_equals_rescaled_sm_scale():
    rng = np.random.default_rng(7)
    q, k, v, do, _, _, _ = _inputs(rng, 1, 25, 2, 1, 8, temp=False)
    tau = 0.37
    a = orc.OracleConfig(sm_scale=0.5)
    b = orc.OracleConfig(sm_scale=0.5 * tau)
    Oa, La, _, _ = orc.forward(q, k, v, np.full((1, 25), tau), None, None, a)
    Ob, Lb, _, _ = orc.forward(q, k, v, None, None, None, b)
    np.testing.assert_allclose(Oa, Ob, atol=1e-13)
    np.testing.assert_allclose(La, Lb, atol=1e-13)


def test_window_at_least_L_is_plain_causal():
    rng = np.random.default_rng(8)
    q, k, v, do, t, _, _ = _inputs(rng, 1, 31, 2, 2, 8)
    a = orc.OracleConfig(sm_scale=0.4, causal=True, window_len=31)
    b = orc.OracleConfig(sm_scale=0.4, causal=True)
    Oa, La, _, _ = orc.forward(q, k, v, t, None, None, a)
    Ob, Lb, _, _ = orc.forward(q, k, v, t, None, None, b)
    assert np.array_equal(Oa, Ob) and np.array_equal(La, Lb)


def test_window_row_equals_attention_over_its_key_slice():
    rng = np.random.default_rng(12)
    L, W = 29, 6
    q, k, v, do, t, _, _ = _inputs(rng, 1, L, 1, 1, 8)
    cfg = orc.OracleConfig(sm_scale=0.4, causal=True, window_len=W, cap_method="tanh", cap=3.0)
    O, LSE, _, _ = orc.forward(q, k, v, t, None, None, cfg)
    for i in range(L):
        j0 = max(0, i - W + 1)
        sl = slice(j0, i + 1)
        # attention of row i over keys j0..i only, computed without any mask
        ss = 0.4 * q[0, i, 0] @ k[0, sl, 0].T
        tt = t[0, i] * 3.0 * np.tanh(ss / 3.0)
        w = np.exp(tt - tt.max())
        np.testing.assert_allclose(O[0, i, 0], (w / w.sum()) @ v[0, sl, 0], atol=1e-13)
        np.testing.assert_allclose(LSE[0, 0, i], tt.max() + np.log(w.sum()), atol=1e-13)


def test_packed_segments_equal_separate_documents():
    rng = np.random.default_rng(9)
    L = 40
    q, k, v, do, t, _, _ = _inputs(rng, 1, L, 2, 1, 8)
    seg = np.array([[0] * 9 + [1] * 14 + [2] * 17], np.int32)
    cfg = orc.OracleConfig(sm_scale=0.4, causal=True, cap_method="soft_sign", cap=2.0, z_loss_weight=0.1)
    O, LSE, _, _ = orc.forward(q, k, v, t, seg, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, seg, None, O, LSE, do, cfg)
    for a, b in ((0, 9), (9, 23), (23, 40)):
        sl = slice(a, b)
        o, lse, _, _ = orc.forward(q[:, sl], k[:, sl], v[:, sl], t[:, sl], None, None, cfg)
        dq, dk, dv, _ = orc.backward(q[:, sl], k[:, sl], v[:, sl], t[:, sl], None, None, o, lse,
                                     do[:, sl], cfg)
        np.testing.assert_allclose(O[:, sl], o, atol=1e-14)
        np.testing.assert_allclose(LSE[:, :, sl], lse, atol=1e-14)
        np.testing.assert_allclose(dQ[:, sl], dq, atol=1e-13)
        np.testing.assert_allclose(dK[:, sl], dk, atol=1e-13)
        np.testing.assert_allclose(dV[:, sl], dv, atol=1e-13)


def test_ranker_rows_attend_to_history_and_self():
    rng = np.random.default_rng(10)
    L, hu, cu = 30, 12, 19
    q, k, v, do, t, _, _ = _inputs(rng, 1, L, 1, 1, 8, temp=False)
    bounds = np.array([[0, hu, hu, cu]], np.int32)
    cfg = orc.OracleConfig(sm_scale=0.4, cap_method="alsc", cap=30.0, alpha=2.0, beta=0.5)
    O, LSE, _, _ = orc.forward(q, k, v, None, None, bounds, cfg)
    plain = cfg
    for i in range(L):
        if i < hu:
            keys = list(range(hu))
        elif i < cu:
            keys = list(range(hu)) + [i]
        else:
            assert np.all(O[0, i, 0] == 0) and np.isneginf(LSE[0, 0, i])
            continue
        ss = 0.4 * q[0, i, 0] @ k[0, keys, 0].T
        tt = orc.cap_forward(ss, plain)
        w = np.exp(tt - tt.max())
        np.testing.assert_allclose(O[0, i, 0], (w / w.sum()) @ v[0, keys, 0], atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(13)
    G = 3
    q, k, v, do, t, _, _ = _inputs(rng, 2, 21, 6, 2, 8)
    cfg = orc.OracleConfig(sm_scale=0.3, causal=True, cap_method="alsc", cap=10.0, alpha=2.0,
                           beta=0.5, z_loss_weight=0.01)
    O, LSE, _, _ = orc.forward(q, k, v, t, None, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, None, None, O, LSE, do, cfg)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    O2, LSE2, _, _ = orc.forward(q, kr, vr, t, None, None, cfg)
    dQ2, dK2, dV2, _ = orc.backward(q, kr, vr, t, None, None, O2, LSE2, do, cfg)
    np.testing.assert_allclose(O, O2, atol=1e-14)
    np.testing.assert_allclose(dQ, dQ2, atol=1e-13)
    np.testing.assert_allclose(dK, dK2.reshape(2, 21, 2, G, 8).sum(axis=3), atol=1e-13)
    np.testing.assert_allclose(dV, dV2.reshape(2, 21, 2, G, 8).sum(axis=3), atol=1e-13)


def test_backward_kv_head_matches_full_backward():
    rng = np.random.default_rng(14)
    q, k, v, do, t, sg, _ = _inputs(rng, 2, 23, 4, 2, 8, seg=True)
    cfg = orc.OracleConfig(sm_scale=0.3, causal=True, cap_method="tanh", cap=4.0, z_loss_weight=0.02)
    O, LSE, _, _ = orc.forward(q, k, v, t, sg, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, sg, None, O, LSE, do, cfg)
    dq, dk, dv, o, lse = orc.backward_kv_head(q, k, v, t, sg, None, do, cfg, 1, 1)
    np.testing.assert_allclose(dq, dQ[1, :, 2:4], atol=1e-13)
    np.testing.assert_allclose(dk, dK[1, :, 1], atol=1e-13)
    np.testing.assert_allclose(dv, dV[1, :, 1], atol=1e-13)
    np.testing.assert_allclose(o, O[1, :, 2:4], atol=1e-14)


def test_visit_matrix_matches_tile_scan():
    rng = np.random.default_rng(15)
    L = 77
    seg = np.repeat(np.arange(6), [10, 20, 5, 30, 2, 10]).astype(np.int32)
    for cfg, sg, bd in ((orc.OracleConfig(sm_scale=1, causal=True, window_len=9), None, None),
                        (orc.OracleConfig(sm_scale=1, causal=True), seg, None),
                        (orc.OracleConfig(sm_scale=1), None, (0, 30, 30, 41))):
        M = orc.mask_matrix(L, cfg, sg, bd)
        for bq, bk in ((8, 8), (16, 8), (8, 32)):
            V = orc.visit_matrix(L, bq, bk, cfg, sg, bd)
            nq, nk = -(-L // bq), -(-L // bk)
            Mp = np.zeros((nq * bq, nk * bk), bool)
            Mp[:L, :L] = M
            ref = Mp.reshape(nq, bq, nk, bk).any(axis=(1, 3))
            assert np.array_equal(V, ref)



def test_visit_matrix_a_lone_live_key_at_a_tile_edge():
    # History = key 7 alone, the last column of the first 8-wide KV tile;
    # candidates 8..19 see that key and themselves.  Live pairs, worked out by
    # hand: (7, 7), (i, 7) and (i, i) for i in 8..19.
    cfg = orc.OracleConfig(sm_scale=1)
    V = orc.visit_matrix(24, 8, 8, cfg, None, (7, 8, 8, 20))
    assert V.astype(int).tolist() == [[1, 0, 0], [1, 1, 0], [1, 0, 1]]
    # the same pairs through 4-row query tiles and 16-wide KV tiles: rows 0..3
    # and 20..23 hold no live pair, only rows 16..19 reach the second KV tile
    V = orc.visit_matrix(24, 4, 16, cfg, None, (7, 8, 8, 20))
    assert V.astype(int).tolist() == [[0, 0], [1, 0], [1, 0], [1, 0], [1, 1], [0, 0]]


def test_visit_matrix_matches_scalar_liveness():
    """Tile (qt, kt) is visited iff some pair in it is live by the scalar
    restatement of the masks (triple loop over tiles, rows and keys)."""
    rng = np.random.default_rng(31)
    for _ in range(40):
        L = int(rng.integers(1, 40))
        causal = bool(rng.integers(0, 2))
        window = int(rng.choice([0, 1, 2, 5, 50]))
        sg = np.cumsum(rng.random(L) < 0.2).astype(np.int32) if rng.integers(0, 2) else None
        bd = None
        if rng.integers(0, 2):
            hl = int(rng.integers(0, L + 1))
            hu = int(rng.integers(hl, L + 1))
            cl = int(rng.integers(0, L + 1))
            bd = (hl, hu, cl, int(rng.integers(cl, L + 1)))
        bq, bk = int(rng.choice([1, 3, 4, 8])), int(rng.choice([1, 2, 4, 8]))
        cfg = orc.OracleConfig(sm_scale=1, causal=causal, window_len=window)
        V = orc.visit_matrix(L, bq, bk, cfg, sg, bd)
        nq, nk = -(-L // bq), -(-L // bk)
        assert V.shape == (nq, nk)
        for qt in range(nq):
            for kt in range(nk):
                live = any(_live(i, j, causal, window, sg, bd)
                           for i in range(qt * bq, min(L, (qt + 1) * bq))
                           for j in range(kt * bk, min(L, (kt + 1) * bk)))
                assert V[qt, kt] == live, (L, bq, bk, qt, kt)


def test_pair_counts_closed_forms():
    # causal L=2048: L(L+1)/2 per head; causal + window 1024 at L=4096:
    # sum_{i<1023}(i+1) + (4096-1023)*1024 = 523776 + 3146752
    c2 = orc.OracleConfig(sm_scale=1, causal=True)
    assert orc.pair_count(2048, c2) == 2048 * 2049 // 2
    c3 = orc.OracleConfig(sm_scale=1, causal=True, window_len=1024)
    assert orc.pair_count(4096, c3) == 523776 + 3146752
    # ranker: history rows see hu keys, candidate rows hu + 1, others none
    c5 = orc.OracleConfig(sm_scale=1)
    assert orc.pair_count(300, c5, bounds=np.array([[0, 100, 100, 140]])) == 100 * 100 + 40 * 101


def test_stored_pair_counts_match_oracle():
    import json
    import os
    from soft_capped_attention_gb300.workloads import WORKLOADS, make_aux
    with open(os.path.join(os.path.dirname(__file__), "golden", "pair_counts.json")) as f:
        stored = json.load(f)
    for idx, w in WORKLOADS.items():
        aux = make_aux(w, seed=idx)
        n = orc.pair_count(w.L, orc.config_from_workload(w), aux["seg"], aux["bounds"], B=w.B,
                           Lk=w.key_len)
        assert stored[str(idx)]["pairs"] == n * w.Hq
    # the unmasked cross-attention workload: every (query, key) pair
    w6 = WORKLOADS[6]
    assert stored["6"]["pairs"] == w6.B * w6.Hq * w6.L * w6.key_len



# ---------------------------------------------------------------------------
# Ranker bounds from history / candidate segment ids.
# ---------------------------------------------------------------------------

def test_ranker_bounds_from_ids_layouts():
    H, C = 7, 9
    # the pages' test layout: first half history, second half candidates
    seg = np.zeros((1, 128), np.int32)
    seg[:, :64] = H
    seg[:, 64:] = C
    b, ok = orc.ranker_bounds_from_ids(seg, H, C)
    assert b.tolist() == [[0, 64, 64, 128]] and ok.all()
    # padding before and after, candidates absent, history absent, a gap
    rows = np.full((4, 20), 3, np.int32)
    rows[0, 2:10] = H
    rows[0, 10:15] = C
    rows[1, 5:9] = H
    rows[2, 4:6] = C
    rows[3, 1:4] = H
    rows[3, 6:8] = H
    b, ok = orc.ranker_bounds_from_ids(rows, H, C)
    assert b.tolist() == [[2, 10, 10, 15], [5, 9, 0, 0], [0, 0, 4, 6], [1, 8, 0, 0]]
    assert ok.tolist() == [True, True, True, False]


def test_ranker_bounds_from_ids_equal_explicit_bounds():
    # attention with bounds derived from ids equals attention with the same
    # bounds given explicitly (and with the dense ranker mask of those ranges)
    rng = np.random.default_rng(5)
    B, L, Hq, Hkv, D = 2, 24, 2, 1, 4
    q, k, v, do, t, _, _ = _inputs(rng, B, L, Hq, Hkv, D, temp=True)
    seg = np.full((B, L), -1, np.int32)
    seg[0, :15] = 1
    seg[0, 15:20] = 2
    seg[1, 3:11] = 1
    seg[1, 11:24] = 2
    bd, ok = orc.ranker_bounds_from_ids(seg, 1, 2)
    assert ok.all() and bd.tolist() == [[0, 15, 15, 20], [3, 11, 11, 24]]
    cfg = orc.OracleConfig(sm_scale=0.5, cap_method="alsc", cap=30.0, alpha=2.0, beta=0.5,
                           causal=False, window_len=0, z_loss_weight=0.0)
    O1, L1, _, _ = orc.forward(q, k, v, t, None, bd, cfg)
    O2, L2, _, _ = orc.forward(q, k, v, t, None, np.array([[0, 15, 15, 20], [3, 11, 11, 24]]), cfg)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


# ---------------------------------------------------------------------------
# Unequal query and key lengths (q [B, Lq, Hq, D], k / v [B, Lk, Hkv, D];
# positions compared directly, as the pages' masks compare them).
# ---------------------------------------------------------------------------

def _cross_inputs(rng, B, Lq, Lk, Hq, Hkv, D, temp=True, scale=1.0):
    q = _rand((B, Lq, Hq, D), rng, scale)
    k = _rand((B, Lk, Hkv, D), rng, scale)
    v = _rand((B, Lk, Hkv, D), rng)
    do = _rand((B, Lq, Hq, D), rng)
    t = rng.uniform(0.5, 1.5, size=(B, Lq)) if temp else None
    return q, k, v, do, t


CROSS_SHAPES = [(23, 41), (41, 23), (5, 64)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("Lq,Lk", CROSS_SHAPES)
def test_cross_lengths_match_torch_sdpa(causal, G, Lq, Lk):
    # PyTorch's is_causal with unequal lengths keeps key j for query i iff j <= i
    # (its reference mask is ones(Lq, Lk).tril()), the same position comparison
    rng = np.random.default_rng(31)
    B, Hkv, D = 2, 2, 16
    Hq = Hkv * G
    q, k, v, do, _ = _cross_inputs(rng, B, Lq, Lk, Hq, Hkv, D, temp=False)
    cfg = orc.OracleConfig(sm_scale=0.3, causal=causal)
    O, LSE, _, _ = orc.forward(q, k, v, None, None, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, None, None, None, O, LSE, do, cfg)
    assert O.shape == (B, Lq, Hq, D) and dK.shape == (B, Lk, Hkv, D) and LSE.shape == (B, Hq, Lq)

    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_(True)
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_(True)
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_(True)
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, is_causal=causal, scale=0.3)
    (out * torch.tensor(do).permute(0, 2, 1, 3)).sum().backward()
    np.testing.assert_allclose(O, out.detach().permute(0, 2, 1, 3).numpy(), atol=1e-12)
    np.testing.assert_allclose(dQ, tq.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    s = 0.3 * torch.einsum("bhid,bhjd->bhij", tq.detach(), kk.detach())
    if causal:
        s = s.masked_fill(torch.ones(Lq, Lk, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(LSE, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


CROSS_MASKS = [dict(causal=False, window_len=0), dict(causal=True, window_len=0),
               dict(causal=True, window_len=4), dict(causal=False, window_len=3)]


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("mask", range(len(CROSS_MASKS)))
@pytest.mark.parametrize("Lq,Lk", [(9, 14), (14, 9)])
def test_cross_lengths_dense_matches_brute_force(method, cap, alpha, beta, mask, Lq, Lk, monkeypatch):
    monkeypatch.setattr(orc, "ROW_BLOCK", 4)
    mk = CROSS_MASKS[mask]
    rng = np.random.default_rng(400 + mask)
    B, Hq, Hkv, D = 2, 4, 2, 5
    q, k, v, do, t = _cross_inputs(rng, B, Lq, Lk, Hq, Hkv, D)
    cfg = orc.OracleConfig(sm_scale=0.45, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.03)
    O, LSE, _, _ = orc.forward(q, k, v, t, None, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, None, None, O, LSE, do, cfg)
    p = dict(sm_scale=0.45, cap_method=method, cap=cap, alpha=alpha, beta=beta,
             causal=mk["causal"], window_len=mk["window_len"], z_loss_weight=0.03)
    ref = brute_attention(q.tolist(), k.tolist(), v.tolist(), do.tolist(), t.tolist(), None, None, p)
    np.testing.assert_allclose(O, np.array(ref["O"]), rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.isinf(LSE), np.isinf(np.array(ref["LSE"])))
    fin = np.isfinite(LSE)
    np.testing.assert_allclose(LSE[fin], np.array(ref["LSE"])[fin], rtol=1e-12, atol=1e-12)
    for a, r in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
        np.testing.assert_allclose(a, np.array(ref[r]), rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("method,cap,alpha,beta", CAPS)
@pytest.mark.parametrize("Lq,Lk,causal,window", [(4, 7, True, 0), (7, 4, True, 3), (5, 3, False, 0)])
def test_cross_lengths_gradients_match_finite_differences(method, cap, alpha, beta, Lq, Lk, causal,
                                                          window):
    rng = np.random.default_rng(77 + Lq)
    q, k, v, do, t = _cross_inputs(rng, 1, Lq, Lk, 2, 1, 3, scale=1.5)
    cfg = orc.OracleConfig(sm_scale=0.7, cap_method=method, cap=cap, alpha=alpha, beta=beta,
                           causal=causal, window_len=window, z_loss_weight=0.05)
    O, LSE, _, _ = orc.forward(q, k, v, t, None, None, cfg)
    grads = orc.backward(q, k, v, t, None, None, O, LSE, do, cfg)[:3]
    h = 1e-6
    for x, gx in zip((q, k, v), grads):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + h
            lp = orc.loss(q, k, v, t, None, None, do, cfg)
            x[idx] = x0 - h
            lm = orc.loss(q, k, v, t, None, None, do, cfg)
            x[idx] = x0
            fd[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(gx - fd) / max(np.linalg.norm(fd), 1e-30)
        assert err < 1e-6, err


def test_causal_keys_past_the_last_query_are_never_seen():
    # with Lk > Lq, causal query i sees keys 0..i < Lq: the same as attention over
    # the first Lq keys, and the later keys get exactly zero gradient
    rng = np.random.default_rng(8)
    Lq, Lk = 11, 19
    q, k, v, do, t = _cross_inputs(rng, 2, Lq, Lk, 2, 2, 4)
    cfg = orc.OracleConfig(sm_scale=0.5, cap_method="tanh", cap=5.0, causal=True, window_len=6)
    O, LSE, _, _ = orc.forward(q, k, v, t, None, None, cfg)
    dQ, dK, dV, _ = orc.backward(q, k, v, t, None, None, O, LSE, do, cfg)
    O2, LSE2, _, _ = orc.forward(q, k[:, :Lq], v[:, :Lq], t, None, None, cfg)
    dQ2, dK2, dV2, _ = orc.backward(q, k[:, :Lq], v[:, :Lq], t, None, None, O2, LSE2, do, cfg)
    # (equal up to the rounding of sums over more, exactly-zero, terms)
    np.testing.assert_allclose(O, O2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(LSE, LSE2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dQ, dQ2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dK[:, :Lq], dK2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dV[:, :Lq], dV2, rtol=0, atol=1e-13)
    assert np.all(dK[:, Lq:] == 0.0) and np.all(dV[:, Lq:] == 0.0)


@pytest.mark.parametrize("Lq,Lk", [(300, 700), (700, 300), (129, 129)])
def test_cross_lengths_pair_count_closed_forms(Lq, Lk):
    none = orc.OracleConfig(sm_scale=1.0)
    assert orc.pair_count(Lq, none, Lk=Lk) == Lq * Lk
    causal = orc.OracleConfig(sm_scale=1.0, causal=True)
    assert orc.pair_count(Lq, causal, Lk=Lk) == sum(min(i + 1, Lk) for i in range(Lq))
    W = 50
    win = orc.OracleConfig(sm_scale=1.0, causal=True, window_len=W)
    assert orc.pair_count(Lq, win, Lk=Lk) == sum(max(0, min(i, Lk - 1) - max(0, i - W + 1) + 1)
                                               for i in range(Lq))


def test_cross_lengths_reject_segments_and_ranker_bounds():
    rng = np.random.default_rng(2)
    q, k, v, do, t = _cross_inputs(rng, 1, 6, 9, 2, 2, 4)
    cfg = orc.OracleConfig(sm_scale=0.5)
    with pytest.raises(ValueError):
        orc.forward(q, k, v, t, np.zeros((1, 6), np.int32), None, cfg)
    with pytest.raises(ValueError):
        orc.forward(q, k, v, t, None, np.array([[0, 2, 2, 4]]), cfg)
