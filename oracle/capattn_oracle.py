"""fp64 CPU oracle for soft-capped unified attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg
use it.  It shares no code with the CUDA library (no kernels, helpers, tables
or constants); both sides only take their inputs from the seeded generators.

It is the plain dense definition of what the fused kernels compute, evaluated
per (batch, query head) in float64, in blocks of at most 512 query rows to bound
memory.  The sources are two pages:

* "triton_kernels.py" (xrex_unified Pallas-Triton unified attention): the
  forward kernel (scores scaled by sm_scale, segment / causal / window masks,
  online softmax with the l and m residuals) and the dQ and dK/dV kernels
  (cap, then temperature, then mask; dS scaled by temp, cap' and sm_scale).
* "mosaic_backward.py" (xrex_unified Mosaic GPU backward): the cap helpers
  ``_apply_cap_mosaic`` / ``_apply_cap_grad_mosaic``, the ranker
  history/candidate mask ``ranker_mask_mosaic_kv_q``, the GQA head mapping,
  P recomputed from the stored log-sum-exp, the z-loss term and the delta
  pre-pass.

Readings taken where the pages are silent or disagree (each is repeated in the
design notes):

* cap -> temperature -> mask, with masked probabilities exactly 0 (both
  backward kernels use this order; the Triton forward masks before the cap,
  which would let tanh/ALSC leak masked keys).
* ALSC forward exactly as printed; its gradient is the analytic derivative of
  that forward, alpha * s_z (1 - s_z) / denom.  The printed gradient carries an
  extra 1/cap factor, which would make the gradients disagree with finite
  differences of the forward.
* z-loss gradient z * P * LSE (the Mosaic form), the exact gradient of
  (z/2) * sum(LSE^2) over rows that are not fully masked.
* delta = rowsum(O * dO) with the normalised O and the unscaled dO.
* A fully masked row gives m = LSE = -inf, l = 0, O = 0, delta = 0 and no
  gradient contribution.
* Window: key j is kept when j > i - window_len (one-sided, as printed).
* Natural-log LSE.  GQA: kv_head = q_head // (Hq // Hkv).
* Query and key lengths may differ (mosaic_backward.py's orchestration reads
  q as (B, Q, H, D) and k as (B, KV, H_kv, D)): query position i < Lq and key
  position j < Lk are compared directly, as the pages' masks compare positions
  (causal keeps j <= i, the window j > i - window_len).  Segment ids and
  ranker bounds are per-position arrays of one sequence, so they are used only
  when Lq == Lk.

parity unpinned: the ALSC gradient reading, the 1/2 in the z-loss loss and the
fully-masked-row convention are readings, not facts fixed by the pages; the
tests pin each against the mathematics of the reading chosen.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

ROW_BLOCK = 512


@dataclass(frozen=True)
class OracleConfig:
    sm_scale: float
    cap_method: str = "none"  # none | tanh | soft_sign | alsc
    cap: float = 0.0
    alpha: float = 0.0
    beta: float = 0.0
    causal: bool = False
    window_len: int = 0
    z_loss_weight: float = 0.0


def config_from_workload(w) -> OracleConfig:
    return OracleConfig(sm_scale=float(w.sm_scale), cap_method=w.cap_method,
                        cap=float(w.cap), alpha=float(w.alpha), beta=float(w.beta),
                        causal=bool(w.causal), window_len=int(w.window_len),
                        z_loss_weight=float(w.z_loss_weight))


# ---------------------------------------------------------------------------
# Cap functions: mosaic_backward.py, _apply_cap_mosaic (forward) and the
# derivative of each branch (see the ALSC reading in the module docstring).
# ---------------------------------------------------------------------------

def _sigmoid(x):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def alsc_constants(alpha: float, beta: float):
    """sigma(alpha*beta) and denom = sigma(1 - sigma) + 1e-12 (ALSC branch)."""
    sb = 1.0 / (1.0 + math.exp(-alpha * beta))
    return sb, sb * (1.0 - sb) + 1e-12


def cap_is_active(cfg: OracleConfig) -> bool:
    # mosaic_backward.py, _apply_cap_mosaic: method "none" or cap <= 0 leaves s unchanged.
    return cfg.cap_method != "none" and cfg.cap > 0


def cap_forward(s, cfg: OracleConfig):
    s = np.asarray(s, dtype=np.float64)
    if not cap_is_active(cfg):
        return s
    c = cfg.cap
    if cfg.cap_method == "tanh":
        return c * np.tanh(s / c)
    if cfg.cap_method == "soft_sign":
        return s / (1.0 + np.abs(s) / c)
    if cfg.cap_method == "alsc":
        sb, denom = alsc_constants(cfg.alpha, cfg.beta)
        z = cfg.alpha * (s / c + cfg.beta)
        return c * (_sigmoid(z) - sb) / denom
    raise ValueError(f"unknown cap method {cfg.cap_method!r}")


def cap_derivative(s, cfg: OracleConfig):
    """d cap(s) / d s for each method."""
    s = np.asarray(s, dtype=np.float64)
    if not cap_is_active(cfg):
        return np.ones_like(s)
    c = cfg.cap
    if cfg.cap_method == "tanh":
        t = np.tanh(s / c)
        return 1.0 - t * t
    if cfg.cap_method == "soft_sign":
        r = 1.0 / (1.0 + np.abs(s) / c)
        return r * r
    if cfg.cap_method == "alsc":
        sb, denom = alsc_constants(cfg.alpha, cfg.beta)
        sz = _sigmoid(cfg.alpha * (s / c + cfg.beta))
        return cfg.alpha * sz * (1.0 - sz) / denom
    raise ValueError(f"unknown cap method {cfg.cap_method!r}")


# ---------------------------------------------------------------------------
# Masks: triton_kernels.py forward kernel (segment equality, causal i >= j,
# window j > i - window_len) and mosaic_backward.py ranker_mask_mosaic_kv_q
# (history keys visible to history and candidate queries; a candidate query
# also sees itself), written here in query x key orientation.
# ---------------------------------------------------------------------------

def mask_rows(rows, Lk: int, cfg: OracleConfig, seg_row=None, bounds_row=None) -> np.ndarray:
    """Boolean mask M[len(rows), Lk] for query positions ``rows`` of one batch
    row against key positions 0 .. Lk - 1."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(Lk, dtype=np.int64)[None, :]
    M = np.ones((i.shape[0], Lk), dtype=bool)
    if seg_row is not None:
        seg_row = np.asarray(seg_row)
        M &= seg_row[i] == seg_row[j]
    if cfg.causal:
        M &= i >= j
    if cfg.window_len > 0:
        M &= j > i - cfg.window_len
    if bounds_row is not None:
        hl, hu, cl, cu = (int(x) for x in bounds_row)
        q_hist = (i >= hl) & (i < hu)
        q_cand = (i >= cl) & (i < cu)
        k_hist = (j >= hl) & (j < hu)
        k_cand = (j >= cl) & (j < cu)
        M &= (k_hist & (q_hist | q_cand)) | (q_cand & k_cand & (i == j))
    return M


def mask_matrix(L: int, cfg: OracleConfig, seg_row=None, bounds_row=None, Lk: int | None = None) -> np.ndarray:
    return mask_rows(np.arange(L), L if Lk is None else Lk, cfg, seg_row, bounds_row)


def _check_lengths(Lq: int, Lk: int, seg, bounds):
    # segment ids and ranker bounds describe one sequence (reading in the module docstring)
    if Lq != Lk and (seg is not None or bounds is not None):
        raise ValueError("segment ids and ranker bounds need equal query and key lengths")


def _row_inputs(temp, seg, bounds, b, L):
    t = np.ones(L) if temp is None else np.asarray(temp[b], dtype=np.float64)
    s = None if seg is None else np.asarray(seg[b])
    bd = None if bounds is None else np.asarray(bounds[b])
    return t, s, bd


# ---------------------------------------------------------------------------
# Forward for a block of query rows of one head.
# ---------------------------------------------------------------------------

def _forward_block(q_rows, k, v, temp_rows, M, cfg: OracleConfig):
    """Returns (O, LSE, m, l, P, s) for the given rows, all float64.

    s = sm_scale * Q K^T; c = cap(s); t = temp_i * c; masked entries drop out;
    m = max over live t, l = sum exp(t - m), LSE = m + ln l,
    P = exp(t - LSE) on live entries (0 elsewhere), O = P V.
    """
    s = cfg.sm_scale * (q_rows @ k.T)
    t = temp_rows[:, None] * cap_forward(s, cfg)
    t_live = np.where(M, t, -np.inf)
    m = t_live.max(axis=1)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    e = np.where(M, np.exp(np.where(M, t, 0.0) - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    lse = np.where(live, m_safe + np.log(np.where(live, l, 1.0)), -np.inf)
    lse_safe = np.where(live, lse, 0.0)
    P = np.where(M, np.exp(np.where(M, t, 0.0) - lse_safe[:, None]), 0.0)
    O = P @ v
    return O, lse, m, l, P, s


def forward(q, k, v, temp, seg, bounds, cfg: OracleConfig):
    """q [B,L,Hq,D], k/v [B,Lk,Hkv,D] (any float dtype; used as float64).

    Returns O [B,L,Hq,D], LSE [B,Hq,L], m [B,Hq,L], l [B,Hq,L], all float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, L, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _check_lengths(L, Lk, seg, bounds)
    G = Hq // Hkv
    O = np.zeros((B, L, Hq, D))
    LSE = np.empty((B, Hq, L))
    Mx = np.empty((B, Hq, L))
    Lx = np.empty((B, Hq, L))
    for b in range(B):
        t_row, s_row, b_row = _row_inputs(temp, seg, bounds, b, L)
        for r0 in range(0, L, ROW_BLOCK):
            rows = np.arange(r0, min(L, r0 + ROW_BLOCK))
            M = mask_rows(rows, Lk, cfg, s_row, b_row)
            for h in range(Hq):
                g = h // G
                o, lse, m, l, _, _ = _forward_block(q[b, rows, h], k[b, :, g], v[b, :, g],
                                                    t_row[rows], M, cfg)
                O[b, rows, h] = o
                LSE[b, h, rows] = lse
                Mx[b, h, rows] = m
                Lx[b, h, rows] = l
    return O, LSE, Mx, Lx


# ---------------------------------------------------------------------------
# Backward: mosaic_backward.py dQ / dK-dV kernels and the delta pre-pass,
# triton_kernels.py dQ / dK-dV kernels for where temperature enters.
# ---------------------------------------------------------------------------

def _backward_block(q_rows, k, v, do_rows, temp_rows, M, lse_rows, delta_rows, cfg,
                    dlse_rows=None):
    """dQ rows plus this block's contributions to dK and dV of its KV head."""
    s = cfg.sm_scale * (q_rows @ k.T)
    t = temp_rows[:, None] * cap_forward(s, cfg)
    live = np.isfinite(lse_rows)
    lse_safe = np.where(live, lse_rows, 0.0)
    P = np.where(M, np.exp(np.where(M, t, 0.0) - lse_safe[:, None]), 0.0)
    dP = do_rows @ v.T
    dT = P * (dP - delta_rows[:, None]) + cfg.z_loss_weight * P * lse_safe[:, None]
    if dlse_rows is not None:
        # d LSE_i / d t_ij = P_ij: an upstream gradient of the LSE adds dLSE_i P_ij
        dT = dT + P * np.where(live, dlse_rows, 0.0)[:, None]
    dX = cfg.sm_scale * cap_derivative(s, cfg) * temp_rows[:, None] * dT
    return dX @ k, dX.T @ q_rows, P.T @ do_rows


def backward(q, k, v, temp, seg, bounds, O, LSE, dO, cfg: OracleConfig, dLSE=None):
    """Returns dQ [B,L,Hq,D], dK and dV [B,Lk,Hkv,D] and delta [B,Hq,L] (float64).

    delta_i = sum_d O_id dO_id; dP = dO V^T; dT = P (dP - delta) + z P LSE;
    dX = sm_scale * cap'(s) * temp_i * dT; dQ = dX K; dK_g = sum over the
    group's query heads of dX^T Q; dV_g likewise of P^T dO.  dLSE [B,Hq,L]
    (optional) is an upstream gradient of the returned LSE; it adds
    dLSE_i P_ij to dT (ignored on fully masked rows).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    O = np.asarray(O, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, L, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _check_lengths(L, Lk, seg, bounds)
    G = Hq // Hkv
    delta = np.einsum("blhd,blhd->bhl", O, dO)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for b in range(B):
        t_row, s_row, b_row = _row_inputs(temp, seg, bounds, b, L)
        for r0 in range(0, L, ROW_BLOCK):
            rows = np.arange(r0, min(L, r0 + ROW_BLOCK))
            M = mask_rows(rows, Lk, cfg, s_row, b_row)
            for h in range(Hq):
                g = h // G
                dq, dk, dv = _backward_block(q[b, rows, h], k[b, :, g], v[b, :, g], dO[b, rows, h],
                                             t_row[rows], M, LSE[b, h, rows], delta[b, h, rows], cfg,
                                             None if dLSE is None else dLSE[b, h, rows])
                dQ[b, rows, h] = dq
                dK[b, :, g] += dk
                dV[b, :, g] += dv
    return dQ, dK, dV, delta


def backward_kv_head(q, k, v, temp, seg, bounds, dO, cfg: OracleConfig, b: int, g: int):
    """Full recomputation for one (batch, KV head): returns (dQ [L,G,D] for the
    group's query heads, dK [Lk,D], dV [Lk,D], O [L,G,D], LSE [G,L])."""
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    L, D, Lk = q.shape[1], q.shape[3], k.shape[1]
    _check_lengths(L, Lk, seg, bounds)
    t_row, s_row, b_row = _row_inputs(temp, seg, bounds, b, L)
    kk = np.asarray(k[b, :, g], np.float64)
    vv = np.asarray(v[b, :, g], np.float64)
    dQ = np.zeros((L, G, D))
    O = np.zeros((L, G, D))
    LSE = np.zeros((G, L))
    dK = np.zeros((Lk, D))
    dV = np.zeros((Lk, D))
    for r0 in range(0, L, ROW_BLOCK):
        rows = np.arange(r0, min(L, r0 + ROW_BLOCK))
        M = mask_rows(rows, Lk, cfg, s_row, b_row)
        for hh in range(G):
            h = g * G + hh
            qr = np.asarray(q[b, rows, h], np.float64)
            dor = np.asarray(dO[b, rows, h], np.float64)
            o, lse, _, _, _, _ = _forward_block(qr, kk, vv, t_row[rows], M, cfg)
            delta = np.einsum("id,id->i", o, dor)
            dq, dk, dv = _backward_block(qr, kk, vv, dor, t_row[rows], M, lse, delta, cfg)
            dQ[rows, hh] = dq
            O[rows, hh] = o
            LSE[hh, rows] = lse
            dK += dk
            dV += dv
    return dQ, dK, dV, O, LSE


def backward_dtemp(q, k, v, temp, seg, bounds, O, LSE, dO, cfg: OracleConfig, dLSE=None):
    """Gradient with respect to the per-query temperature, [B, L] (float64).

    The temperature multiplies the capped score, t = temp_i * c with
    c = cap(sm_scale * Q K^T) (triton_kernels.py forward; the pages' backward
    returns zeros for it).  With dT = dL/dt = P (dP - delta) + z P LSE as in
    the backward above, dL/dtemp_i = sum over query heads h and keys j of
    dT[h, i, j] * c[h, i, j] (the temperature is shared by all heads of a
    row; masked pairs have P = 0 and add nothing).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    O = np.asarray(O, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, L, Hq, D = q.shape
    Lk = k.shape[1]
    _check_lengths(L, Lk, seg, bounds)
    G = Hq // k.shape[2]
    delta = np.einsum("blhd,blhd->bhl", O, dO)
    dtemp = np.zeros((B, L))
    for b in range(B):
        t_row, s_row, b_row = _row_inputs(temp, seg, bounds, b, L)
        for r0 in range(0, L, ROW_BLOCK):
            rows = np.arange(r0, min(L, r0 + ROW_BLOCK))
            M = mask_rows(rows, Lk, cfg, s_row, b_row)
            for h in range(Hq):
                g = h // G
                s = cfg.sm_scale * (q[b, rows, h] @ k[b, :, g].T)
                c = cap_forward(s, cfg)
                lse = LSE[b, h, rows]
                live = np.isfinite(lse)
                lse_safe = np.where(live, lse, 0.0)
                P = np.where(M, np.exp(np.where(M, t_row[rows][:, None] * c, 0.0) - lse_safe[:, None]), 0.0)
                dP = dO[b, rows, h] @ v[b, :, g].T
                dT = P * (dP - delta[b, h, rows][:, None]) + cfg.z_loss_weight * P * lse_safe[:, None]
                if dLSE is not None:
                    dT = dT + P * np.where(live, dLSE[b, h, rows], 0.0)[:, None]
                dtemp[b, rows] += np.sum(dT * c, axis=1)
    return dtemp


def loss(q, k, v, temp, seg, bounds, dO, cfg: OracleConfig, dLSE=None) -> float:
    """L = sum(O * dO) + (z/2) * sum of LSE^2 over rows that are not fully masked
    (+ sum of LSE * dLSE over those rows when dLSE is given).

    The backward above is the gradient of this scalar with respect to Q, K, V.
    """
    O, LSE, _, _ = forward(q, k, v, temp, seg, bounds, cfg)
    live = np.isfinite(LSE)
    lse = np.where(live, LSE, 0.0)
    extra = 0.0 if dLSE is None else float(np.sum(lse * np.asarray(dLSE, np.float64)))
    return float(np.sum(O * np.asarray(dO, np.float64))
                 + 0.5 * cfg.z_loss_weight * np.sum(lse ** 2)) + extra


# ---------------------------------------------------------------------------
# Ranker bounds from history / candidate segment ids.
# ---------------------------------------------------------------------------

def ranker_bounds_from_ids(seg, history_id: int, candidate_id: int):
    """Per batch row, (hl, hu, cl, cu) and whether both id runs are contiguous.

    mosaic_backward.py's test marks the history positions of a row with
    HISTORY_SEGMENT_ID and the candidate positions with CANDIDATE_SEGMENT_ID;
    the mapping to bounds sits in a module the pages do not show.  Reading: the
    history range is [first, last + 1) of the positions carrying history_id,
    the candidate range likewise for candidate_id; an absent id gives the
    empty range (0, 0); a run with gaps is not a range (flagged, its bounds
    are still the hull).
    """
    seg = np.asarray(seg)
    B, L = seg.shape
    bounds = np.zeros((B, 4), np.int32)
    contiguous = np.ones(B, bool)
    for b in range(B):
        for slot, ident in ((0, history_id), (2, candidate_id)):
            pos = np.nonzero(seg[b] == ident)[0]
            if pos.size:
                lo, hi = int(pos[0]), int(pos[-1]) + 1
                bounds[b, slot:slot + 2] = (lo, hi)
                if hi - lo != pos.size:
                    contiguous[b] = False
    return bounds, contiguous


# ---------------------------------------------------------------------------
# Block visit sets and pair counts, by brute force over the mask.
# ---------------------------------------------------------------------------

def visit_matrix(L: int, block_q: int, block_kv: int, cfg: OracleConfig, seg_row=None,
                 bounds_row=None, Lk: int | None = None) -> np.ndarray:
    """V[qt, kt] = True iff the (block_q x block_kv) tile (qt, kt) holds at least
    one unmasked pair (L query rows, Lk keys, Lk = L by default).  The forward
    and dQ kernels visit row qt of V; the dK/dV kernel visits column kt."""
    Lk = L if Lk is None else Lk
    nq = -(-L // block_q)
    nk = -(-Lk // block_kv)
    V = np.zeros((nq, nk), dtype=bool)
    for r0 in range(0, L, ROW_BLOCK):
        rows = np.arange(r0, min(L, r0 + ROW_BLOCK))
        M = mask_rows(rows, Lk, cfg, seg_row, bounds_row)
        qt = rows // block_q
        for kt in range(nk):
            any_live = M[:, kt * block_kv:(kt + 1) * block_kv].any(axis=1)
            np.logical_or.at(V[:, kt], qt, any_live)
    return V


def pair_count(L: int, cfg: OracleConfig, seg=None, bounds=None, B: int = 1,
               Lk: int | None = None) -> int:
    """Number of unmasked (query, key) pairs summed over the batch (one head;
    L query rows, Lk keys, Lk = L by default)."""
    Lk = L if Lk is None else Lk
    total = 0
    for b in range(B):
        s_row = None if seg is None else seg[b]
        b_row = None if bounds is None else bounds[b]
        for r0 in range(0, L, ROW_BLOCK):
            rows = np.arange(r0, min(L, r0 + ROW_BLOCK))
            total += int(mask_rows(rows, Lk, cfg, s_row, b_row).sum())
    return total
