"""CPU tests of the C-ABI boundary: the library loads, exports what the header
declares, validates arguments on the host, and its host-side mask bits and
visit maps are bit-exact against the oracle's brute force."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca
from soft_capped_attention_gb300.workloads import WORKLOADS, make_aux

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ca.LIB_PATH):
        from soft_capped_attention_gb300 import build
        build.build()
    return ca.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "capattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(capattn_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ca.EXPORTED_SYMBOLS)


def _cfg(**kw):
    base = dict(B=2, L=300, Hq=4, Hkv=2, D=128, dtype=torch.bfloat16)
    base.update(kw)
    ap = ca.AttnParams(sm_scale=0.1, cap_method=base.pop("cap_method", "tanh"),
                       cap=base.pop("cap", 5.0), causal=base.pop("causal", True),
                       window_len=base.pop("window_len", 0))
    Lk = base.pop("Lk", 0)
    return ca.make_config(ap, **base, Lk=Lk)


def test_validation_codes(lib):
    v = lambda c: lib.capattn_validate_config(ctypes.byref(c))
    assert v(_cfg()) == 0
    assert v(_cfg(Hq=3)) == 1                 # Hq not a multiple of Hkv
    assert v(_cfg(L=0)) == 1
    assert v(_cfg(D=64)) == 0                 # bf16: D = 64 or 128
    assert v(_cfg(D=96)) == 2
    assert v(_cfg(D=64, dtype=torch.float32)) == 0
    assert v(_cfg(D=96, dtype=torch.float32)) == 2
    c = _cfg()
    c.struct_size = 4
    assert v(c) == 1
    c = _cfg()
    c.cap_method = 7
    assert v(c) == 1
    c = _cfg()
    c.z_loss_weight = -1.0
    assert v(c) == 1
    c = _cfg()
    c.window_len = -3
    assert v(c) == 1
    assert lib.capattn_workspace_bytes(ctypes.byref(_cfg(Hq=3)), 0) == 0
    assert lib.capattn_workspace_bytes(ctypes.byref(_cfg()), 0) > 0
    assert lib.capattn_status_string(4) == b"a kernel gave up on a bounded wait"


def test_compute_calls_reject_bad_arguments_before_launch(lib):
    c = _cfg()
    ws = (ctypes.c_uint8 * 4096)()
    # null q: rejected on the host, nothing is launched
    st = lib.capattn_fwd(ctypes.byref(c), None, ctypes.c_void_p(16), ctypes.c_void_p(16), None,
                         None, None, ctypes.c_void_p(16), ctypes.c_void_p(16), None, None,
                         ctypes.c_void_p(256), 1 << 20, None)
    assert st == 1
    # misaligned pointer
    st = lib.capattn_fwd(ctypes.byref(c), ctypes.c_void_p(18), ctypes.c_void_p(16),
                         ctypes.c_void_p(16), None, None, None, ctypes.c_void_p(16),
                         ctypes.c_void_p(16), None, None, ctypes.c_void_p(256), 1 << 20, None)
    assert st == 1
    # workspace too small
    st = lib.capattn_fwd(ctypes.byref(c), ctypes.c_void_p(16), ctypes.c_void_p(16),
                         ctypes.c_void_p(16), None, None, None, ctypes.c_void_p(16),
                         ctypes.c_void_p(16), None, None, ctypes.c_void_p(256), 8, None)
    assert st == 5
    st = lib.capattn_bwd(ctypes.byref(c), *([ctypes.c_void_p(16)] * 3), None, None, None,
                         *([ctypes.c_void_p(16)] * 3), None, *([ctypes.c_void_p(16)] * 3),
                         ctypes.c_void_p(256), 1 << 20, None)
    assert st == 1  # null dq


def test_backward_workspace_holds_the_temperature_partials(lib):
    c = _cfg(B=3, L=300, Hq=4, Hkv=2)
    fwd = lib.capattn_workspace_bytes(ctypes.byref(c), 0)
    no_pool = lib.capattn_workspace_bytes(ctypes.byref(c), 2)
    extra = 8 * 3 * 4 * 300  # two float partial sums per (b, query head, row)
    assert no_pool == fwd + ((extra + 255) // 256) * 256
    # a forward-sized workspace is refused by the backward before any launch
    p16 = ctypes.c_void_p(16)
    st = lib.capattn_bwd(ctypes.byref(c), p16, p16, p16, None, None, None, *([p16] * 7),
                         ctypes.c_void_p(256), fwd, None)
    assert st == 5
    assert lib.capattn_workspace_bytes(ctypes.byref(c), 3) == 0


def _band_width(L, Lk, causal, window, tile=128):
    """Widest set of key tiles that some (query, key) pair of a query tile may
    see under the causal / window masks alone, by brute force over positions."""
    nq, nk = -(-L // tile), -(-Lk // tile)
    widest = 0
    for qt in range(nq):
        i = np.arange(qt * tile, min(L, qt * tile + tile))[:, None]
        seen = 0
        for kt in range(nk):
            j = np.arange(kt * tile, min(Lk, kt * tile + tile))[None, :]
            ok = np.ones((i.size, j.size), bool)
            if causal:
                ok &= j <= i
            if window:
                ok &= j > i - window
            seen += bool(ok.any())
        widest = max(widest, seen)
    return widest


@pytest.mark.parametrize("L,Lk,causal,window", [
    (300, 0, True, 0), (1000, 0, True, 300), (1000, 0, False, 300), (1000, 0, True, 129),
    (700, 0, True, 1), (300, 1000, False, 0), (2048, 0, True, 0), (640, 0, False, 0)])
def test_dx_pool_size_is_the_band_of_the_masks(lib, L, Lk, causal, window):
    B, Hq = 2, 4
    c = _cfg(B=B, L=L, Lk=Lk, Hq=Hq, Hkv=2, causal=causal, window_len=window)
    no_pool = lib.capattn_workspace_bytes(ctypes.byref(c), 2)
    bwd = lib.capattn_workspace_bytes(ctypes.byref(c), 1)
    nq = -(-L // 128)
    pool = B * Hq * nq * _band_width(L, Lk or L, causal, window) * 128 * 128 * 2
    assert bwd == ((no_pool + 1023) // 1024) * 1024 + pool


def test_dx_pool_is_left_out_for_fp32_and_above_16_gib(lib):
    c = _cfg(dtype=torch.float32, D=64)
    assert lib.capattn_workspace_bytes(ctypes.byref(c), 1) == lib.capattn_workspace_bytes(ctypes.byref(c), 2)
    # full attention, 128 x 128 tiles: 64 * 128 * 128 tiles of 32 KB = 32 GiB
    c = _cfg(B=64, L=16384, Hq=1, Hkv=1, causal=False)
    assert lib.capattn_workspace_bytes(ctypes.byref(c), 1) == lib.capattn_workspace_bytes(ctypes.byref(c), 2)
    # at the cap: 16 GiB exactly is kept
    c = _cfg(B=32, L=16384, Hq=1, Hkv=1, causal=False)
    pool = 32 * 128 * 128 * 32768
    assert pool == 16 << 30
    no_pool = lib.capattn_workspace_bytes(ctypes.byref(c), 2)
    assert lib.capattn_workspace_bytes(ctypes.byref(c), 1) == ((no_pool + 1023) // 1024) * 1024 + pool


def test_backward_flags_are_checked_on_the_host(lib):
    c = _cfg()
    p16 = ctypes.c_void_p(16)
    bwd = lib.capattn_workspace_bytes(ctypes.byref(c), 1)
    # unknown flag bits: rejected before any launch (the pointers are never touched)
    for flags in (2, 0x80000000, 3):
        st = lib.capattn_bwd_ex(ctypes.byref(c), p16, p16, p16, None, None, None, *([p16] * 3),
                                None, *([p16] * 4), None, flags, ctypes.c_void_p(256), bwd, None)
        assert st == 1, flags
    assert ca.BWD_REUSE_FWD_MAPS == 1


def test_bounded_wait_check_rejects_bad_arguments(lib):
    # checked on the host before any CUDA call
    assert lib.capattn_check_bounded_wait(None, 1000, None) == 5
    assert lib.capattn_check_bounded_wait(ctypes.c_void_p(128), 1000, None) == 5
    assert lib.capattn_check_bounded_wait(ctypes.c_void_p(256), 0, None) == 1
    assert lib.capattn_check_bounded_wait(ctypes.c_void_p(256), 100000001, None) == 1


def _oracle_cfg(causal, window_len):
    return orc.OracleConfig(sm_scale=1.0, causal=causal, window_len=window_len)


CASES = [
    dict(causal=False, window_len=0, seg=None, bounds=None),
    dict(causal=True, window_len=0, seg=None, bounds=None),
    dict(causal=True, window_len=37, seg=None, bounds=None),
    dict(causal=False, window_len=50, seg=None, bounds=None),
    dict(causal=True, window_len=0, seg="packed", bounds=None),
    dict(causal=False, window_len=0, seg="packed", bounds=None),
    dict(causal=True, window_len=29, seg="packed", bounds=None),
    dict(causal=False, window_len=0, seg=None, bounds="ranker"),
    dict(causal=True, window_len=0, seg=None, bounds="ranker"),
    dict(causal=True, window_len=40, seg="packed", bounds="ranker"),
]


def _aux(case, B, L, rng):
    seg = bounds = None
    if case["seg"]:
        seg = np.zeros((B, L), np.int32)
        for b in range(B):
            cuts = np.sort(rng.choice(np.arange(1, L), size=5, replace=False))
            for c in cuts:
                seg[b, c:] += 1
    if case["bounds"]:
        bounds = np.zeros((B, 4), np.int32)
        for b in range(B):
            hl = int(rng.integers(0, L // 3))
            hu = int(rng.integers(hl, L))
            cl = int(rng.integers(hu // 2, L))
            cu = int(rng.integers(cl, L + 1))
            bounds[b] = (hl, hu, cl, cu)
    return seg, bounds


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("L", [1, 63, 130, 300])
def test_mask_bits_match_oracle(lib, case, L):
    cs = CASES[case]
    rng = np.random.default_rng(case * 1000 + L)
    B = 2
    seg, bounds = _aux(cs, B, L, rng) if L > 8 else (None, None)
    c = _cfg(B=B, L=L, causal=cs["causal"], window_len=cs["window_len"])
    ocfg = _oracle_cfg(cs["causal"], cs["window_len"])
    for b in range(B):
        bits = ca.capattn_mask_bits_host(c, b, seg, bounds)
        ref = orc.mask_matrix(L, ocfg, None if seg is None else seg[b],
                              None if bounds is None else bounds[b])
        assert np.array_equal(bits, ref)


def _pack(V):
    nr, nc = V.shape
    words = -(-nc // 32)
    out = np.zeros((nr, words), np.uint32)
    for w in range(words):
        blk = V[:, w * 32:(w + 1) * 32]
        for bit in range(blk.shape[1]):
            out[:, w] |= blk[:, bit].astype(np.uint32) << np.uint32(bit)
    return out


def oracle_visit_words(B, L, bq, bk, ocfg, seg, bounds, which):
    rows = []
    for b in range(B):
        V = orc.visit_matrix(L, bq, bk, ocfg, None if seg is None else seg[b],
                             None if bounds is None else bounds[b])
        rows.append(_pack(V if which == ca.VISIT_Q_TILES else V.T))
    return np.concatenate(rows, axis=0).reshape(-1)


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("L,dtype", [(300, torch.bfloat16), (777, torch.bfloat16),
                                     (200, torch.float32), (4100, torch.bfloat16)])
def test_visit_maps_match_oracle(lib, case, L, dtype):
    cs = CASES[case]
    rng = np.random.default_rng(case + 7 * L)
    B = 2
    seg, bounds = _aux(cs, B, L, rng)
    D = 128 if dtype == torch.bfloat16 else 64
    c = _cfg(B=B, L=L, D=D, dtype=dtype, causal=cs["causal"], window_len=cs["window_len"])
    bq, bk = ca.capattn_tile_sizes(c)
    ocfg = _oracle_cfg(cs["causal"], cs["window_len"])
    for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
        got = ca.capattn_visit_map_host(c, seg, bounds, which)
        ref = oracle_visit_words(B, L, bq, bk, ocfg, seg, bounds, which)
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_visit_maps_of_the_five_workloads(lib, idx):
    w = WORKLOADS[idx]
    aux = make_aux(w, seed=idx)
    B = min(w.B, 4)
    seg = None if aux["seg"] is None else np.ascontiguousarray(aux["seg"][:B])
    bounds = None if aux["bounds"] is None else np.ascontiguousarray(aux["bounds"][:B])
    c = ca.make_config(ca.params_from_workload(w), B, w.L, w.Hq, w.Hkv, w.D, torch.bfloat16)
    bq, bk = ca.capattn_tile_sizes(c)
    ocfg = orc.config_from_workload(w)
    for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
        got = ca.capattn_visit_map_host(c, seg, bounds, which)
        ref = oracle_visit_words(B, w.L, bq, bk, ocfg, seg, bounds, which)
        assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Unequal query and key lengths (config field Lk; 0 means Lk = L).
# ---------------------------------------------------------------------------

CROSS = [(300, 700), (700, 300), (129, 1000), (1, 64), (64, 1)]
CROSS_MASKS = [dict(causal=False, window_len=0), dict(causal=True, window_len=0),
               dict(causal=True, window_len=37), dict(causal=False, window_len=50)]


def test_key_length_validation(lib):
    v = lambda c: lib.capattn_validate_config(ctypes.byref(c))
    assert v(_cfg(Lk=0)) == 0 and v(_cfg(Lk=301)) == 0 and v(_cfg(Lk=1)) == 0
    assert v(_cfg(Lk=-1)) == 1
    ws = lambda c: lib.capattn_workspace_bytes(ctypes.byref(c), 1)
    assert ws(_cfg(Lk=0)) == ws(_cfg(Lk=300))
    assert ws(_cfg(Lk=30000)) > ws(_cfg(Lk=300))


def test_unequal_lengths_reject_segments_and_bounds(lib):
    c = _cfg(L=300, Lk=500)
    seg = np.zeros((2, 300), np.int32)
    bounds = np.array([[0, 10, 10, 20], [0, 10, 10, 20]], np.int32)
    for s, bd in ((seg, None), (None, bounds)):
        with pytest.raises(ca.CapattnError):
            ca.capattn_visit_map_host(c, s, bd, ca.VISIT_Q_TILES)
        with pytest.raises(ca.CapattnError):
            ca.capattn_mask_bits_host(c, 0, s, bd)
    # the compute calls reject them on the host, before any launch
    p16 = ctypes.c_void_p(16)
    st = lib.capattn_fwd(ctypes.byref(c), p16, p16, p16, None, p16, None, p16, p16, None, None,
                         ctypes.c_void_p(256), 1 << 24, None)
    assert st == 1
    st = lib.capattn_bwd(ctypes.byref(c), p16, p16, p16, None, None, p16, *([p16] * 7),
                         ctypes.c_void_p(256), 1 << 24, None)
    assert st == 1


@pytest.mark.parametrize("mask", range(len(CROSS_MASKS)))
@pytest.mark.parametrize("L,Lk", CROSS)
def test_unequal_lengths_mask_bits_match_oracle(lib, mask, L, Lk):
    cs = CROSS_MASKS[mask]
    c = _cfg(B=1, L=L, Lk=Lk, causal=cs["causal"], window_len=cs["window_len"])
    bits = ca.capattn_mask_bits_host(c, 0)
    ref = orc.mask_matrix(L, _oracle_cfg(cs["causal"], cs["window_len"]), Lk=Lk)
    assert bits.shape == (L, Lk) and np.array_equal(bits, ref)


@pytest.mark.parametrize("mask", range(len(CROSS_MASKS)))
@pytest.mark.parametrize("L,Lk", CROSS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_unequal_lengths_visit_maps_match_oracle(lib, mask, L, Lk, dtype):
    cs = CROSS_MASKS[mask]
    D = 128 if dtype == torch.bfloat16 else 64
    c = _cfg(B=2, L=L, Lk=Lk, D=D, dtype=dtype, causal=cs["causal"], window_len=cs["window_len"])
    bq, bk = ca.capattn_tile_sizes(c)
    ocfg = _oracle_cfg(cs["causal"], cs["window_len"])
    V = orc.visit_matrix(L, bq, bk, ocfg, Lk=Lk)
    for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
        got = ca.capattn_visit_map_host(c, None, None, which)
        ref = np.concatenate([_pack(V if which == ca.VISIT_Q_TILES else V.T)] * 2, axis=0).reshape(-1)
        assert np.array_equal(got, ref)


# ALSC on the FMA pipe: the host-fitted polynomial the kernels use in place of
# the sigmoid when every raw score of a warp's step lies within xmax.
@pytest.mark.parametrize("cap,alpha,beta,sm_scale", [
    (30.0, 2.0, 0.5, 1.0 / np.sqrt(128.0)),   # the windowed GQA and ranker workloads
    (30.0, 4.0, 0.5, 0.125),                  # mosaic_backward.py's test cap
    (20.0, 1.0, 0.0, 1.0 / np.sqrt(64.0)),
    (50.0, 8.0, -0.25, 1.0 / np.sqrt(128.0)),
    (5.0, 0.5, 3.0, 0.3),
])
def test_alsc_polynomial_matches_the_sigmoid(lib, cap, alpha, beta, sm_scale):
    ap = ca.AttnParams(sm_scale=float(sm_scale), cap_method="alsc", cap=cap, alpha=alpha, beta=beta)
    cfg = ca.make_config(ap, 1, 128, 2, 2, 128, torch.bfloat16)
    coeffs = (ctypes.c_float * 7)()
    xmax = ctypes.c_float(0.0)
    assert lib.capattn_debug_alsc_poly(ctypes.byref(cfg), coeffs, ctypes.byref(xmax)) == 0
    g = np.array(list(coeffs), np.float64)
    u = sm_scale * alpha / cap
    assert abs(xmax.value * u - 0.5) < 1e-6
    x = np.linspace(-xmax.value, xmax.value, 4001)
    sig = lambda z: 1.0 / (1.0 + np.exp(-z))
    exact = sig(u * x + alpha * beta) - sig(alpha * beta)
    poly = x * np.polyval(g[::-1], x)
    # float32 coefficients: a few ulps of the result's scale (|exact| <= 0.25)
    assert np.max(np.abs(poly - exact)) <= 2e-7
    assert abs(poly[2000]) == 0.0  # exactly zero at X = 0


def test_alsc_polynomial_needs_an_alsc_cap(lib):
    ap = ca.AttnParams(sm_scale=0.1, cap_method="tanh", cap=30.0)
    cfg = ca.make_config(ap, 1, 128, 2, 2, 128, torch.bfloat16)
    coeffs = (ctypes.c_float * 7)()
    xmax = ctypes.c_float(0.0)
    assert lib.capattn_debug_alsc_poly(ctypes.byref(cfg), coeffs, ctypes.byref(xmax)) == 1
