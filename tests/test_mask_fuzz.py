"""Randomised CPU sweep of the host mask exports against the oracle.

The fixed cases in test_boundary.py cover each mask kind at a few lengths.
This sweep draws lengths, windows, segment layouts and ranker bounds from
edge-heavy distributions: windows of 1 and windows longer than the sequence,
a single segment and every position its own segment, empty history or
candidate ranges, ranges that overlap or touch the sequence ends, lengths one
off a tile boundary, and query lengths apart from key lengths.  Each draw
compares the live-pair bits of every batch row and both visit maps (at the
bf16 and fp32 tile sizes) with the oracle's brute-force mask, bit for bit."""

import os

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca

N_DRAWS = 48


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ca.LIB_PATH):
        from soft_capped_attention_gb300 import build
        build.build()
    return ca.lib()


def _length(rng):
    kind = rng.integers(0, 4)
    if kind == 0:
        return int(rng.integers(1, 9))
    if kind == 1:  # one off a 64- or 128-row tile boundary
        return int(rng.choice([64, 128, 256, 384])) + int(rng.choice([-1, 0, 1]))
    return int(rng.integers(9, 700))


def _window(rng, L):
    kind = rng.integers(0, 5)
    if kind == 0:
        return 0
    if kind == 1:
        return 1
    if kind == 2:
        return L + int(rng.integers(0, 50))  # covers the whole sequence
    return int(rng.integers(1, max(2, L)))


def _segments(rng, B, L):
    seg = np.zeros((B, L), np.int32)
    for b in range(B):
        kind = rng.integers(0, 4)
        if kind == 0 or L == 1:
            continue  # one segment
        if kind == 1:
            seg[b] = np.arange(L)  # every position its own segment
            continue
        n_cuts = int(rng.integers(1, min(L - 1, 24) + 1))
        cuts = np.sort(rng.choice(np.arange(1, L), size=n_cuts, replace=False))
        for c in cuts:
            seg[b, c:] += 1
        seg[b] += int(rng.integers(-3, 4))  # ids need not start at 0
    return seg


def _range(rng, L):
    kind = rng.integers(0, 4)
    if kind == 0:
        x = int(rng.integers(0, L + 1))
        return x, x  # empty
    if kind == 1:
        return 0, int(rng.integers(0, L + 1))
    if kind == 2:
        return int(rng.integers(0, L + 1)), L
    lo = int(rng.integers(0, L + 1))
    return lo, int(rng.integers(lo, L + 1))


def _bounds(rng, B, L):
    bounds = np.zeros((B, 4), np.int32)
    for b in range(B):
        hl, hu = _range(rng, L)
        if rng.integers(0, 2):  # candidates after the history, as a ranker lays them out
            cl = int(rng.integers(hu, L + 1))
            cu = int(rng.integers(cl, L + 1))
        else:  # anywhere, overlapping the history or not
            cl, cu = _range(rng, L)
        bounds[b] = (hl, hu, cl, cu)
    return bounds


def _draw(seed):
    rng = np.random.default_rng(1000003 + seed)
    B = int(rng.integers(1, 4))
    L = _length(rng)
    causal = bool(rng.integers(0, 2))
    window = _window(rng, L)
    seg = _segments(rng, B, L) if rng.integers(0, 2) else None
    bounds = _bounds(rng, B, L) if rng.integers(0, 3) == 0 else None
    return B, L, causal, window, seg, bounds


def _pack(V):
    nr, nc = V.shape
    words = -(-nc // 32)
    out = np.zeros((nr, words), np.uint32)
    for c in range(nc):
        out[:, c // 32] |= V[:, c].astype(np.uint32) << np.uint32(c % 32)
    return out


@pytest.mark.parametrize("seed", range(N_DRAWS))
def test_random_masks_match_oracle(lib, seed):
    B, L, causal, window, seg, bounds = _draw(seed)
    ap = ca.AttnParams(sm_scale=0.1, cap_method="tanh", cap=5.0, causal=causal, window_len=window)
    ocfg = orc.OracleConfig(sm_scale=1.0, causal=causal, window_len=window)
    rows = lambda a, b: None if a is None else a[b]

    c = ca.make_config(ap, B, L, 2, 2, 128, torch.bfloat16)
    for b in range(B):
        bits = ca.capattn_mask_bits_host(c, b, seg, bounds)
        assert np.array_equal(bits, orc.mask_matrix(L, ocfg, rows(seg, b), rows(bounds, b))), b

    for D, dtype in ((128, torch.bfloat16), (64, torch.float32)):
        c = ca.make_config(ap, B, L, 2, 2, D, dtype)
        bq, bk = ca.capattn_tile_sizes(c)
        Vs = [orc.visit_matrix(L, bq, bk, ocfg, rows(seg, b), rows(bounds, b)) for b in range(B)]
        for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
            got = ca.capattn_visit_map_host(c, seg, bounds, which)
            ref = np.concatenate([_pack(V if which == ca.VISIT_Q_TILES else V.T) for V in Vs],
                                 axis=0).reshape(-1)
            assert np.array_equal(got, ref), (dtype, which)


@pytest.mark.parametrize("seed", range(N_DRAWS // 2))
def test_random_unequal_lengths_match_oracle(lib, seed):
    """Query and key lengths drawn apart (segment ids and ranker bounds need
    equal lengths, so only the causal and window masks apply)."""
    rng = np.random.default_rng(2000003 + seed)
    L, Lk = _length(rng), _length(rng)
    causal = bool(rng.integers(0, 2))
    window = _window(rng, max(L, Lk))
    ap = ca.AttnParams(sm_scale=0.1, cap_method="tanh", cap=5.0, causal=causal, window_len=window)
    ocfg = orc.OracleConfig(sm_scale=1.0, causal=causal, window_len=window)
    c = ca.make_config(ap, 1, L, 2, 2, 128, torch.bfloat16, Lk=Lk)
    bits = ca.capattn_mask_bits_host(c, 0)
    assert bits.shape == (L, Lk) and np.array_equal(bits, orc.mask_matrix(L, ocfg, Lk=Lk))
    for D, dtype in ((128, torch.bfloat16), (64, torch.float32)):
        c = ca.make_config(ap, 2, L, 2, 2, D, dtype, Lk=Lk)
        bq, bk = ca.capattn_tile_sizes(c)
        V = orc.visit_matrix(L, bq, bk, ocfg, Lk=Lk)
        for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
            got = ca.capattn_visit_map_host(c, None, None, which)
            ref = np.concatenate([_pack(V if which == ca.VISIT_Q_TILES else V.T)] * 2,
                                 axis=0).reshape(-1)
            assert np.array_equal(got, ref), (dtype, which)


def test_draws_reach_the_edge_cases():
    """The sweep's distributions do produce the cases it is there for."""
    draws = [_draw(s) for s in range(N_DRAWS)]
    assert any(w == 1 for _, _, _, w, _, _ in draws)
    assert any(w >= L for _, L, _, w, _, _ in draws)
    assert any(L % 64 in (1, 63) for _, L, _, _, _, _ in draws)
    assert any(L <= 8 for _, L, _, _, _, _ in draws)
    assert any(s is not None and (s[:, 1:] != s[:, :-1]).all() for _, L, _, _, s, _ in draws if L > 1)
    assert any(bd is not None and (bd[:, 0] == bd[:, 1]).any() for *_, bd in draws)
    assert any(bd is not None and (bd[:, 2] == bd[:, 3]).any() for *_, bd in draws)
    assert any(bd is not None and ((bd[:, 2] < bd[:, 1]) & (bd[:, 3] > bd[:, 2])).any() for *_, bd in draws)
