"""Scalar triple-loop restatement of soft-capped attention for tiny shapes.

TEST INFRASTRUCTURE ONLY (see capattn_oracle.py).  Pure Python and the
``math`` module, one (b, h, i, j) pair at a time, with no vectorisation, no
blocking and no shared helpers, so that indexing mistakes in the dense oracle
(a transposed operand, a wrong head mapping, a row block boundary) show up as a
mismatch.  The formulas are the same definition as the dense oracle (pages
"triton_kernels.py" and "mosaic_backward.py", unified attention with cap,
temperature, segment / causal / window masks and the ranker mask).
"""

from __future__ import annotations

import math


def _cap(s, method, cap, alpha, beta):
    if method == "none" or cap <= 0:
        return s, 1.0
    if method == "tanh":
        th = math.tanh(s / cap)
        return cap * th, 1.0 - th * th
    if method == "soft_sign":
        r = 1.0 / (1.0 + abs(s) / cap)
        return s * r, r * r
    if method == "alsc":
        sb = 1.0 / (1.0 + math.exp(-alpha * beta))
        den = sb * (1.0 - sb) + 1e-12
        z = alpha * (s / cap + beta)
        sz = 1.0 / (1.0 + math.exp(-z)) if z > -700 else 0.0
        return cap * (sz - sb) / den, alpha * sz * (1.0 - sz) / den
    raise ValueError(method)


def _live(i, j, causal, window_len, seg, bnd):
    if seg is not None and seg[i] != seg[j]:
        return False
    if causal and j > i:
        return False
    if window_len > 0 and not (j > i - window_len):
        return False
    if bnd is not None:
        hl, hu, cl, cu = bnd
        ih = hl <= i < hu
        ic = cl <= i < cu
        jh = hl <= j < hu
        jc = cl <= j < cu
        if not ((jh and (ih or ic)) or (ic and jc and i == j)):
            return False
    return True


def brute_attention(q, k, v, do, temp, seg, bounds, p):
    """q, do: nested lists [B][L][Hq][D]; k, v: [B][Lk][Hkv][D] (Lk may differ
    from L; query i and key j positions are compared directly); p: dict with
    sm_scale, cap_method, cap, alpha, beta, causal, window_len, z_loss_weight.

    Returns dict of O, LSE, m, l, dQ, dK, dV as nested lists; m [B][Hq][L] is
    the largest live tempered logit of a row and l the sum of exp(t - m) over its
    live keys (-inf and 0 for a row with no live key)."""
    B, L, Hq, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Lk, Hkv = len(k[0]), len(k[0][0])
    G = Hq // Hkv
    O = [[[[0.0] * D for _ in range(Hq)] for _ in range(L)] for _ in range(B)]
    LSE = [[[0.0] * L for _ in range(Hq)] for _ in range(B)]
    Mx = [[[-math.inf] * L for _ in range(Hq)] for _ in range(B)]
    Ls = [[[0.0] * L for _ in range(Hq)] for _ in range(B)]
    dQ = [[[[0.0] * D for _ in range(Hq)] for _ in range(L)] for _ in range(B)]
    dK = [[[[0.0] * D for _ in range(Hkv)] for _ in range(Lk)] for _ in range(B)]
    dV = [[[[0.0] * D for _ in range(Hkv)] for _ in range(Lk)] for _ in range(B)]
    z = p["z_loss_weight"]
    for b in range(B):
        sg = None if seg is None else list(seg[b])
        bd = None if bounds is None else tuple(int(x) for x in bounds[b])
        for h in range(Hq):
            g = h // G
            for i in range(L):
                ti = 1.0 if temp is None else float(temp[b][i])
                svals, tvals, dcap, live = [], [], [], []
                for j in range(Lk):
                    x = 0.0
                    for d in range(D):
                        x += q[b][i][h][d] * k[b][j][g][d]
                    s = p["sm_scale"] * x
                    c, dc = _cap(s, p["cap_method"], p["cap"], p["alpha"], p["beta"])
                    svals.append(s)
                    tvals.append(ti * c)
                    dcap.append(dc)
                    live.append(_live(i, j, p["causal"], p["window_len"], sg, bd))
                lt = [tvals[j] for j in range(Lk) if live[j]]
                if not lt:
                    LSE[b][h][i] = -math.inf
                    continue
                mx = max(lt)
                lsum = sum(math.exp(t - mx) for t in lt)
                lse = mx + math.log(lsum)
                LSE[b][h][i] = lse
                Mx[b][h][i] = mx
                Ls[b][h][i] = lsum
                P = [math.exp(tvals[j] - lse) if live[j] else 0.0 for j in range(Lk)]
                for d in range(D):
                    O[b][i][h][d] = sum(P[j] * v[b][j][g][d] for j in range(Lk))
                delta = sum(O[b][i][h][d] * do[b][i][h][d] for d in range(D))
                for j in range(Lk):
                    if not live[j]:
                        continue
                    dp = sum(do[b][i][h][d] * v[b][j][g][d] for d in range(D))
                    dt = P[j] * (dp - delta) + z * P[j] * lse
                    dx = p["sm_scale"] * dcap[j] * ti * dt
                    for d in range(D):
                        dQ[b][i][h][d] += dx * k[b][j][g][d]
                        dK[b][j][g][d] += dx * q[b][i][h][d]
                        dV[b][j][g][d] += P[j] * do[b][i][h][d]
    return {"O": O, "LSE": LSE, "m": Mx, "l": Ls, "dQ": dQ, "dK": dK, "dV": dV}
