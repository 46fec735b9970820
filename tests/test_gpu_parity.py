"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on shapes that span several tiles and a ragged tail."""

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca
from soft_capped_attention_gb300.workloads import WORKLOADS, make_inputs, round_to_bf16

from parity_utils import compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

CAPS = {"none": (0.0, 0.0, 0.0), "tanh": (50.0, 0.0, 0.0), "soft_sign": (20.0, 0.0, 0.0),
        "alsc": (30.0, 2.0, 0.5)}
MASKS = {
    "full": dict(causal=False, window_len=0, seg=False, ranker=False),
    "causal": dict(causal=True, window_len=0, seg=False, ranker=False),
    "window": dict(causal=True, window_len=200, seg=False, ranker=False),
    "window_nc": dict(causal=False, window_len=77, seg=False, ranker=False),
    "packed": dict(causal=True, window_len=0, seg=True, ranker=False),
    "ranker": dict(causal=False, window_len=0, seg=False, ranker=True),
}


def make_case(B, L, Hq, Hkv, D, dtype, mask, temp, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    r = lambda *s: (rng.standard_normal(s) * scale).astype(np.float32)
    inp = {"q": r(B, L, Hq, D), "k": r(B, L, Hkv, D), "v": rng.standard_normal((B, L, Hkv, D)).astype(np.float32),
           "do": rng.standard_normal((B, L, Hq, D)).astype(np.float32)}
    if dtype == torch.bfloat16:
        for n in ("q", "k", "v", "do"):
            inp[n] = round_to_bf16(inp[n])
    inp["temp"] = rng.uniform(0.5, 1.5, size=(B, L)).astype(np.float32) if temp else None
    inp["seg"] = None
    inp["bounds"] = None
    m = MASKS[mask]
    if m["seg"]:
        seg = np.zeros((B, L), np.int32)
        for b in range(B):
            cuts = np.sort(rng.choice(np.arange(1, L), size=min(4, L - 1), replace=False))
            for c in cuts:
                seg[b, c:] += 1
        inp["seg"] = seg
    if m["ranker"]:
        bd = np.zeros((B, 4), np.int32)
        for b in range(B):
            hu = int(rng.integers(L // 4, 3 * L // 4))
            bd[b] = (0, hu, hu, min(L, hu + int(rng.integers(5, 60))))
        inp["bounds"] = bd
    return inp


def params(cap, mask, z):
    c, a, bta = CAPS[cap]
    m = MASKS[mask]
    return ca.AttnParams(sm_scale=float(1.0 / np.sqrt(128.0)), cap_method=cap, cap=c, alpha=a,
                         beta=bta, causal=m["causal"], window_len=m["window_len"], z_loss_weight=z)


BF16_CASES = [
    # (B, L, Hq, Hkv, cap, mask, temp, z)
    (1, 128, 2, 2, "none", "full", False, 0.0),
    (2, 300, 4, 2, "tanh", "causal", False, 0.0),
    (1, 513, 4, 1, "alsc", "window", True, 1e-4),
    (2, 384, 2, 2, "soft_sign", "packed", False, 0.0),
    (2, 400, 4, 2, "alsc", "ranker", False, 0.0),
    (1, 257, 2, 1, "tanh", "window_nc", True, 0.01),
    (1, 1000, 2, 2, "soft_sign", "causal", True, 0.0),
    (2, 640, 8, 2, "none", "packed", True, 0.001),
    (1, 77, 2, 2, "alsc", "full", False, 0.0),
    (1, 1, 2, 1, "tanh", "causal", False, 0.0),
    (1, 130, 2, 2, "none", "ranker", True, 0.05),
]


@pytest.mark.parametrize("pool", [True, False], ids=["stored_dx", "recompute"])
@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: "-".join(map(str, c)))
def test_bf16_matches_oracle(case, pool):
    B, L, Hq, Hkv, cap, mask, temp, z = case
    inp = make_case(B, L, Hq, Hkv, 128, torch.bfloat16, mask, temp, seed=L * 7 + Hq)
    ap = params(cap, mask, z)
    got = run_gpu(inp, ap, torch.bfloat16, pool=pool)
    ref = run_oracle(inp, ap)
    compare(got, ref, torch.bfloat16)


# bf16 with head dim 64 (the tcgen05 kernels' D = 64 instantiation).  The first
# case is the shape mosaic_backward.py's test_mosaic_backward_correctness
# draws: B=1, L=128, H=4, H_kv=2, D=64, ALSC cap 30, alpha 4, beta 0.5, and a
# per-query temperature (there drawn from U[0.8, 1.2], here U[0.5, 1.5]).
D64_CASES = [
    # (B, L, Hq, Hkv, cap, (cap, alpha, beta) or None, mask, temp, z)
    (1, 128, 4, 2, "alsc", (30.0, 4.0, 0.5), "full", True, 0.0),
    (2, 300, 4, 2, "tanh", None, "causal", False, 0.0),
    (1, 513, 4, 1, "alsc", None, "window", True, 1e-4),
    (2, 384, 2, 2, "soft_sign", None, "packed", False, 0.0),
    (2, 400, 4, 2, "alsc", None, "ranker", False, 0.01),
    (1, 257, 2, 1, "none", None, "window_nc", True, 0.0),
    # (L = 1 would leave a single live key per row, where dP - delta cancels
    # exactly and dQ, dK are zero: no relative error is defined there)
    (1, 2, 2, 1, "tanh", None, "causal", False, 0.0),
    (2, 520, 4, 2, "soft_sign", None, "full", False, 0.0),
    (2, 700, 4, 4, "tanh", None, "causal", False, 0.0),
]


@pytest.mark.parametrize("pool", [True, False], ids=["stored_dx", "recompute"])
@pytest.mark.parametrize("case", D64_CASES, ids=lambda c: "-".join(map(str, c)))
def test_bf16_head_dim_64_matches_oracle(case, pool):
    B, L, Hq, Hkv, cap, cparams, mask, temp, z = case
    inp = make_case(B, L, Hq, Hkv, 64, torch.bfloat16, mask, temp, seed=L * 5 + Hq)
    ap = params(cap, mask, z)
    if cparams is not None:
        ap = ca.AttnParams(sm_scale=0.125, cap_method=cap, cap=cparams[0], alpha=cparams[1],
                           beta=cparams[2], causal=ap.causal, window_len=ap.window_len,
                           z_loss_weight=z)
    got = run_gpu(inp, ap, torch.bfloat16, want_ml=(L == 300), pool=pool)
    ref = run_oracle(inp, ap)
    compare(got, ref, torch.bfloat16)
    np.testing.assert_allclose(got["delta"], ref["delta"], atol=5e-2)


def test_bf16_head_dim_64_dtemp_and_lse_gradient():
    from parity_utils import oracle_cfg, rel_fro
    inp = make_case(2, 300, 4, 2, 64, torch.bfloat16, "causal", True, seed=64)
    ap = params("tanh", "causal", 0.01)
    dlse = np.random.default_rng(64).standard_normal((2, 4, 300)).astype(np.float32)
    q, k, v, do = (to_dev(inp[n], torch.bfloat16) for n in ("q", "k", "v", "do"))
    temp = to_dev(inp["temp"])
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp)
    dq, dk, dv, _, dtemp = ca.capattn_bwd_ex(q, k, v, o, lse, do, ap, temp, dlse=to_dev(dlse),
                                             want_dtemp=True)
    oc = oracle_cfg(ap)
    O, LSE, _, _ = orc.forward(inp["q"], inp["k"], inp["v"], inp["temp"], None, None, oc)
    ref = orc.backward(inp["q"], inp["k"], inp["v"], inp["temp"], None, None, O, LSE, inp["do"], oc,
                       dLSE=dlse.astype(np.float64))
    for got, r in zip((dq, dk, dv), ref[:3]):
        assert rel_fro(got.float().cpu().numpy(), r) <= 2e-2
    rdt = orc.backward_dtemp(inp["q"], inp["k"], inp["v"], inp["temp"], None, None, O, LSE, inp["do"],
                             oc, dLSE=dlse.astype(np.float64))
    assert rel_fro(dtemp.cpu().numpy(), rdt) <= 2e-2


FP32_CASES = [
    (1, 128, 2, 2, 64, "none", "full", False, 0.0),
    (2, 200, 4, 2, 64, "tanh", "causal", True, 0.0),
    (1, 131, 2, 1, 128, "alsc", "window", True, 1e-3),
    (2, 190, 2, 2, 64, "soft_sign", "packed", False, 0.0),
    (2, 150, 4, 2, 128, "alsc", "ranker", False, 0.02),
    (1, 65, 2, 2, 64, "none", "window_nc", True, 0.0),
    # rows past the window (the cases above have windows longer than L)
    (1, 300, 2, 1, 64, "tanh", "window", True, 0.0),
    (2, 190, 2, 2, 128, "soft_sign", "window_nc", False, 0.0),
]


@pytest.mark.parametrize("case", FP32_CASES, ids=lambda c: "-".join(map(str, c)))
def test_fp32_matches_oracle(case):
    B, L, Hq, Hkv, D, cap, mask, temp, z = case
    inp = make_case(B, L, Hq, Hkv, D, torch.float32, mask, temp, seed=L * 3 + D)
    ap = params(cap, mask, z)
    got = run_gpu(inp, ap, torch.float32)
    ref = run_oracle(inp, ap)
    compare(got, ref, torch.float32)


def test_workload_1_tiny_fp32_full():
    w = WORKLOADS[1]
    inp = make_inputs(w, seed=1)
    ap = ca.params_from_workload(w)
    got = run_gpu(inp, ap, torch.float32, want_ml=True)
    ref = run_oracle(inp, ap)
    compare(got, ref, torch.float32)
    np.testing.assert_allclose(got["delta"], ref["delta"], atol=1e-4)
    np.testing.assert_allclose(got["m"], ref["m"], atol=1e-4)
    np.testing.assert_allclose(got["l"], ref["l"], rtol=1e-4)


def test_residuals_m_l_and_delta_bf16():
    inp = make_case(2, 300, 4, 2, 128, torch.bfloat16, "ranker", True, seed=5)
    ap = params("tanh", "ranker", 0.0)
    got = run_gpu(inp, ap, torch.bfloat16, want_ml=True)
    ref = run_oracle(inp, ap)
    live = np.isfinite(ref["LSE"])
    assert np.array_equal(np.isneginf(got["m"]), ~live)
    np.testing.assert_allclose(got["m"][live], ref["m"][live], atol=1e-3)
    np.testing.assert_allclose(got["l"][live], ref["l"][live], rtol=5e-3)
    assert np.all(got["l"][~live] == 0)
    # LSE = m + log l
    np.testing.assert_allclose(got["LSE"][live], got["m"][live] + np.log(got["l"][live]), atol=1e-5)
    assert np.max(np.abs(got["delta"] - ref["delta"])) < 5e-2


def test_fully_masked_rows_are_exact():
    # ranker rows at or past cu see nothing: O = 0, LSE = -inf, no gradient
    inp = make_case(1, 256, 2, 2, 128, torch.bfloat16, "ranker", False, seed=9)
    inp["bounds"] = np.array([[0, 100, 100, 120]], np.int32)
    ap = params("alsc", "ranker", 1e-3)
    got = run_gpu(inp, ap, torch.bfloat16)
    assert np.all(got["O"][0, 120:] == 0)
    assert np.all(np.isneginf(got["LSE"][0, :, 120:]))
    assert np.all(got["dQ"][0, 120:] == 0)
    assert np.all(np.isfinite(got["dK"])) and np.all(np.isfinite(got["dV"]))
    # keys past hu that are not a candidate's own position get no gradient
    assert np.all(got["dK"][0, 120:] == 0) and np.all(got["dV"][0, 120:] == 0)


def test_device_status_reports_bad_segments_and_bounds():
    inp = make_case(1, 200, 2, 2, 128, torch.bfloat16, "packed", False, seed=3)
    ap = params("none", "packed", 0.0)
    q, k, v = (to_dev(inp[n], torch.bfloat16) for n in ("q", "k", "v"))
    cfg = ca.make_config(ap, 1, 200, 2, 2, 128, torch.bfloat16)
    ws = ca.new_workspace(cfg, q.device)
    seg = to_dev(np.ascontiguousarray(inp["seg"][:, ::-1]))  # decreasing ids
    ca.capattn_fwd(q, k, v, ap, None, seg, None, workspace=ws)
    st, bits = ca.capattn_device_status(ws)
    assert st == 6 and bits & 2
    assert ca.capattn_device_status(ws)[0] == 0  # cleared
    bounds = to_dev(np.array([[0, 300, 10, 20]], np.int32))
    ca.capattn_fwd(q, k, v, ap, None, None, bounds, workspace=ws)
    st, bits = ca.capattn_device_status(ws)
    assert st == 6 and bits & 4


def test_autograd_function_matches_direct_calls():
    inp = make_case(1, 300, 4, 2, 128, torch.bfloat16, "causal", True, seed=4)
    ap = params("tanh", "causal", 0.0)
    q, k, v, do = (to_dev(inp[n], torch.bfloat16) for n in ("q", "k", "v", "do"))
    temp = to_dev(inp["temp"])
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = ca.attention(qq, kk, vv, ap, temp)
    o.backward(do)
    o2, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp)
    dq, dk, dv, _ = ca.capattn_bwd(q, k, v, o2, lse, do, ap, temp)
    assert torch.equal(o, o2)
    assert torch.equal(qq.grad, dq) and torch.equal(kk.grad, dk) and torch.equal(vv.grad, dv)


def test_fixed_reference_and_running_max_agree_bf16():
    # Capped rows without m / l requested take the fixed reference; asking for
    # m / l switches to the running max.  Both must match the oracle.
    inp = make_case(2, 333, 4, 2, 128, torch.bfloat16, "causal", True, seed=21)
    ap = params("tanh", "causal", 0.0)
    ref = run_oracle(inp, ap)
    a = run_gpu(inp, ap, torch.bfloat16, want_ml=False)
    b = run_gpu(inp, ap, torch.bfloat16, want_ml=True)
    compare(a, ref, torch.bfloat16)
    compare(b, ref, torch.bfloat16)


def test_scores_at_the_bottom_of_the_cap_window():
    # Every score far below -cap: all capped logits sit near the low end of the
    # tanh window, where the fixed reference puts exponents near -120.  The
    # softmax is then nearly uniform and must still match the oracle.
    B, L, H, D = 1, 256, 2, 128
    rng = np.random.default_rng(31)
    base = np.abs(rng.standard_normal((B, L, H, D))).astype(np.float32) + 0.5
    inp = {"q": round_to_bf16(base * 4.0), "k": round_to_bf16(-base * 4.0),
           "v": round_to_bf16(rng.standard_normal((B, L, H, D)).astype(np.float32)),
           "do": round_to_bf16(rng.standard_normal((B, L, H, D)).astype(np.float32)),
           "temp": None, "seg": None, "bounds": None}
    ap = params("tanh", "full", 0.0)
    got, ref = run_gpu(inp, ap, torch.bfloat16), run_oracle(inp, ap)
    # the forward is what the fixed reference changes (the saturated cap leaves
    # the score gradients near zero, where a relative comparison says little)
    assert np.max(np.abs(got["O"] - ref["O"])) <= 2e-2
    assert np.all(np.isfinite(got["LSE"]))
    assert np.max(np.abs(got["LSE"] - ref["LSE"])) <= 1e-3


@pytest.mark.parametrize("sign", [1.0, -1.0], ids=["top", "bottom"])
def test_alsc_window_just_over_the_plain_split(sign):
    # ALSC cap 30, alpha 2, beta 0.5: a logit window of 220.13 (log2 units),
    # just over kSpanLo + kTopMax, where the fixed reference keeps the top
    # exponent at 100 and lets the bottom go a little below -120.  Scores far
    # above (top) or below (bottom) the cap put every logit at that end.
    B, L, H, D = 1, 256, 2, 128
    rng = np.random.default_rng(37)
    base = np.abs(rng.standard_normal((B, L, H, D))).astype(np.float32) + 0.5
    inp = {"q": round_to_bf16(base * 4.0), "k": round_to_bf16(sign * base * 4.0),
           "v": round_to_bf16(rng.standard_normal((B, L, H, D)).astype(np.float32)),
           "do": round_to_bf16(rng.standard_normal((B, L, H, D)).astype(np.float32)),
           "temp": None, "seg": None, "bounds": None}
    ap = params("alsc", "full", 0.0)
    got, ref = run_gpu(inp, ap, torch.bfloat16), run_oracle(inp, ap)
    assert np.max(np.abs(got["O"] - ref["O"])) <= 2e-2
    assert np.all(np.isfinite(got["LSE"]))
    assert np.max(np.abs(got["LSE"] - ref["LSE"])) <= 1e-3


def test_wide_cap_window_uses_running_max():
    # tanh cap 200: the logit window (2 * 200 * log2 e) is wider than the fixed
    # reference allows, so the forward keeps the running max.
    inp = make_case(1, 300, 2, 2, 128, torch.bfloat16, "causal", False, seed=41, scale=3.0)
    ap = ca.AttnParams(sm_scale=float(1.0 / np.sqrt(128.0)), cap_method="tanh", cap=200.0, alpha=0.0,
                       beta=0.0, causal=True, window_len=0, z_loss_weight=0.0)
    compare(run_gpu(inp, ap, torch.bfloat16), run_oracle(inp, ap), torch.bfloat16)


# Temperatures that are negative on some rows and exactly zero on others: a
# negative temperature makes the row's smallest capped score its largest logit
# (the forward's running max then tracks the raw minimum), and temperature 0 is
# a uniform softmax over the live keys.
NONPOS_CASES = [
    # (dtype, D, L, cap, mask, want_ml, z)
    ("bf16", 128, 300, "tanh", "causal", False, 0.0),
    ("bf16", 128, 300, "tanh", "causal", True, 0.0),
    ("bf16", 128, 513, "alsc", "window", False, 1e-3),
    ("bf16", 128, 513, "alsc", "window", True, 1e-3),
    ("bf16", 128, 260, "soft_sign", "packed", False, 0.0),
    ("bf16", 128, 260, "none", "full", True, 0.0),
    ("bf16", 128, 400, "alsc", "ranker", False, 0.0),
    ("fp32", 64, 200, "tanh", "causal", True, 0.0),
    ("fp32", 128, 131, "alsc", "window", True, 1e-3),
    ("fp32", 64, 150, "none", "full", True, 0.0),
]


@pytest.mark.parametrize("case", NONPOS_CASES, ids=lambda c: "-".join(map(str, c)))
def test_nonpositive_temperature_matches_oracle(case):
    dname, D, L, cap, mask, want_ml, z = case
    dtype = torch.bfloat16 if dname == "bf16" else torch.float32
    inp = make_case(2, L, 4, 2, D, dtype, mask, True, seed=L + 13)
    rng = np.random.default_rng(L)
    inp["temp"] = rng.choice(np.array([-1.3, -0.4, 0.0, 0.8], np.float32), size=(2, L))
    ap = params(cap, mask, z)
    got = run_gpu(inp, ap, dtype, want_ml=want_ml)
    ref = run_oracle(inp, ap)
    compare(got, ref, dtype)
    if want_ml:
        live = np.isfinite(ref["LSE"])
        tol = 1e-4 if dtype == torch.float32 else 1e-3
        np.testing.assert_allclose(got["m"][live], ref["m"][live], atol=tol)
        np.testing.assert_allclose(got["l"][live], ref["l"][live], rtol=5e-3)
    # rows with temperature 0: P uniform over live keys, so LSE = ln(#live)
    zero = inp["temp"] == 0.0
    counts = np.stack([orc.mask_matrix(L, oracle_cfg_of(ap), None if inp["seg"] is None else inp["seg"][b],
                                       None if inp["bounds"] is None else inp["bounds"][b]).sum(axis=1)
                       for b in range(2)])
    for h in range(4):
        sel = zero & (counts > 0)
        np.testing.assert_allclose(got["LSE"][:, h][sel], np.log(counts[sel]), atol=1e-3)


def oracle_cfg_of(ap):
    from parity_utils import oracle_cfg
    return oracle_cfg(ap)


def test_dtemp_nonpositive_temperature_bf16():
    from parity_utils import rel_fro
    inp = make_case(2, 300, 4, 2, 128, torch.bfloat16, "causal", True, seed=301)
    inp["temp"] = np.random.default_rng(3).choice(np.array([-1.3, -0.4, 0.0, 0.8], np.float32),
                                                  size=(2, 300))
    ap = params("tanh", "causal", 0.0)
    got = _run_dtemp(inp, ap, torch.bfloat16)
    ref, _ = _oracle_dtemp(inp, ap)
    assert rel_fro(got["dtemp"], ref) <= 2e-2, rel_fro(got["dtemp"], ref)


# ---------------------------------------------------------------------------
# Temperature gradient (capattn_bwd_dtemp) against the oracle's definition.
# ---------------------------------------------------------------------------

def _run_dtemp(inp, ap, dtype):
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("q", "k", "v", "do"))
    temp, seg, bounds = to_dev(inp.get("temp")), to_dev(inp.get("seg")), to_dev(inp.get("bounds"))
    B, L, Hq, D = q.shape
    cfg = ca.make_config(ap, B, L, Hq, k.shape[2], D, dtype)
    ws = ca.new_workspace(cfg, q.device)
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp, seg, bounds, workspace=ws)
    dq, dk, dv, _, dtemp = ca.capattn_bwd_dtemp(q, k, v, o, lse, do, ap, temp, seg, bounds, workspace=ws)
    st, bits = ca.capattn_device_status(ws)
    assert st == 0, f"device status {st} bits {bits}"
    return {"dQ": dq.float().cpu().numpy(), "dtemp": dtemp.cpu().numpy(), "LSE": lse.cpu().numpy()}


def _oracle_dtemp(inp, ap):
    from parity_utils import oracle_cfg
    cfg = oracle_cfg(ap)
    O, LSE, _, _ = orc.forward(inp["q"], inp["k"], inp["v"], inp["temp"], inp.get("seg"),
                               inp.get("bounds"), cfg)
    return orc.backward_dtemp(inp["q"], inp["k"], inp["v"], inp["temp"], inp.get("seg"),
                              inp.get("bounds"), O, LSE, inp["do"], cfg), LSE


DTEMP_CASES = [
    # (B, L, Hq, Hkv, cap, mask, z)
    (2, 300, 4, 2, "tanh", "causal", 0.0),
    (1, 513, 4, 1, "alsc", "window", 1e-4),
    (2, 384, 2, 2, "soft_sign", "packed", 0.0),
    (2, 400, 4, 2, "alsc", "ranker", 0.01),
    (1, 257, 2, 1, "none", "window_nc", 0.0),
]


@pytest.mark.parametrize("case", DTEMP_CASES, ids=lambda c: "-".join(map(str, c)))
def test_dtemp_bf16_matches_oracle(case):
    from parity_utils import rel_fro
    B, L, Hq, Hkv, cap, mask, z = case
    inp = make_case(B, L, Hq, Hkv, 128, torch.bfloat16, mask, True, seed=L + 7)
    ap = params(cap, mask, z)
    got = _run_dtemp(inp, ap, torch.bfloat16)
    ref, LSE = _oracle_dtemp(inp, ap)
    assert rel_fro(got["dtemp"], ref) <= 2e-2, rel_fro(got["dtemp"], ref)
    dead = ~np.isfinite(LSE).any(axis=1)
    assert np.all(got["dtemp"][dead] == 0.0)
    # dQ is the same whether or not dtemp is asked for
    plain = run_gpu(inp, ap, torch.bfloat16)
    assert rel_fro(got["dQ"], plain["dQ"]) < 1e-3


@pytest.mark.parametrize("dname", ["bf16", "fp32"])
def test_dtemp_is_deterministic(dname):
    # per-(head, row) partial sums added in a fixed order: identical bits on
    # every run (and dQ / dK / dV, which use no atomics, too)
    dtype = torch.bfloat16 if dname == "bf16" else torch.float32
    D = 128 if dname == "bf16" else 64
    inp = make_case(2, 700, 8, 2, D, dtype, "causal", True, seed=5)
    ap = params("tanh", "causal", 0.01)
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("q", "k", "v", "do"))
    temp = to_dev(inp["temp"])
    cfg = ca.make_config(ap, 2, 700, 8, 2, D, dtype)
    ws = ca.new_workspace(cfg, q.device)
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp, workspace=ws)
    runs = [ca.capattn_bwd_dtemp(q, k, v, o, lse, do, ap, temp, workspace=ws) for _ in range(4)]
    assert ca.capattn_device_status(ws) == (0, 0)
    for r in runs[1:]:
        for a, b in zip(r, runs[0]):
            assert torch.equal(a, b)


def test_dtemp_fp32_matches_oracle():
    inp = make_case(1, 130, 2, 1, 64, torch.float32, "causal", True, seed=77)
    ap = params("tanh", "causal", 0.02)
    got = _run_dtemp(inp, ap, torch.float32)
    ref, _ = _oracle_dtemp(inp, ap)
    assert np.max(np.abs(got["dtemp"] - ref)) <= 1e-4 * max(1.0, float(np.max(np.abs(ref))))


def test_autograd_temperature_gradient():
    inp = make_case(1, 200, 2, 2, 128, torch.bfloat16, "causal", True, seed=91)
    ap = params("soft_sign", "causal", 0.0)
    q, k, v = (to_dev(inp[n], torch.bfloat16).requires_grad_(True) for n in ("q", "k", "v"))
    temp = to_dev(inp["temp"]).requires_grad_(True)
    o, lse = ca.CapAttnFunction.apply(q, k, v, ap, temp, None, None)
    (o.float() * to_dev(inp["do"], torch.float32)).sum().backward()
    ref, _ = _oracle_dtemp(inp, ap)
    from parity_utils import rel_fro
    assert rel_fro(temp.grad.cpu().numpy(), ref) <= 2e-2


# ---------------------------------------------------------------------------
# Upstream gradient of the returned LSE (capattn_bwd_ex dlse).
# ---------------------------------------------------------------------------

LSE_GRAD_CASES = [
    # (dtype, D, B, L, Hq, Hkv, cap, mask, z, dtemp)
    ("bf16", 128, 2, 300, 4, 2, "tanh", "causal", 0.0, False),
    ("bf16", 128, 1, 513, 4, 1, "alsc", "window", 1e-3, True),
    ("bf16", 128, 2, 400, 4, 2, "soft_sign", "ranker", 0.0, True),
    ("fp32", 64, 2, 200, 4, 2, "tanh", "causal", 0.01, True),
    ("fp32", 128, 1, 131, 2, 1, "none", "packed", 0.0, False),
]


@pytest.mark.parametrize("case", LSE_GRAD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_lse_gradient_matches_oracle(case):
    from parity_utils import oracle_cfg, rel_fro
    dname, D, B, L, Hq, Hkv, cap, mask, z, want_dt = case
    dtype = torch.bfloat16 if dname == "bf16" else torch.float32
    inp = make_case(B, L, Hq, Hkv, D, dtype, mask, True, seed=L + 99)
    dlse = np.random.default_rng(L).standard_normal((B, Hq, L)).astype(np.float32)
    ap = params(cap, mask, z)
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("q", "k", "v", "do"))
    temp, seg, bounds = to_dev(inp["temp"]), to_dev(inp["seg"]), to_dev(inp["bounds"])
    cfg = ca.make_config(ap, B, L, Hq, Hkv, D, dtype)
    ws = ca.new_workspace(cfg, q.device)
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp, seg, bounds, workspace=ws)
    dq, dk, dv, _, dtemp = ca.capattn_bwd_ex(q, k, v, o, lse, do, ap, temp, seg, bounds,
                                             dlse=to_dev(dlse), want_dtemp=want_dt, workspace=ws)
    assert ca.capattn_device_status(ws) == (0, 0)
    oc = oracle_cfg(ap)
    O, LSE, _, _ = orc.forward(inp["q"], inp["k"], inp["v"], inp["temp"], inp["seg"], inp["bounds"], oc)
    ref = orc.backward(inp["q"], inp["k"], inp["v"], inp["temp"], inp["seg"], inp["bounds"], O, LSE,
                       inp["do"], oc, dLSE=dlse.astype(np.float64))
    for got, r in zip((dq, dk, dv), ref[:3]):
        g = got.float().cpu().numpy()
        if dtype == torch.float32:
            assert np.max(np.abs(g - r)) <= 1e-4
        else:
            assert rel_fro(g, r) <= 2e-2, rel_fro(g, r)
    if want_dt:
        rdt = orc.backward_dtemp(inp["q"], inp["k"], inp["v"], inp["temp"], inp["seg"], inp["bounds"],
                                 O, LSE, inp["do"], oc, dLSE=dlse.astype(np.float64))
        assert rel_fro(dtemp.cpu().numpy(), rdt) <= 2e-2


def test_autograd_passes_the_lse_gradient():
    inp = make_case(1, 300, 4, 2, 128, torch.bfloat16, "causal", True, seed=8)
    ap = params("tanh", "causal", 0.0)
    q, k, v, do = (to_dev(inp[n], torch.bfloat16) for n in ("q", "k", "v", "do"))
    temp = to_dev(inp["temp"])
    dlse = torch.randn(1, 4, 300, device="cuda")
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o, lse = ca.CapAttnFunction.apply(qq, kk, vv, ap, temp, None, None)
    ((o.float() * do.float()).sum() + (lse * dlse).sum()).backward()
    o2, lse2, _, _ = ca.capattn_fwd(q, k, v, ap, temp)
    dq, dk, dv, _, _ = ca.capattn_bwd_ex(q, k, v, o2, lse2, do, ap, temp, dlse=dlse)
    assert torch.equal(qq.grad, dq) and torch.equal(kk.grad, dk) and torch.equal(vv.grad, dv)
    # a loss of the lse alone (no gradient reaches o)
    qq.grad = kk.grad = vv.grad = None
    o, lse = ca.CapAttnFunction.apply(qq, kk, vv, ap, temp, None, None)
    (lse * dlse).sum().backward()
    dq0, dk0, dv0, _, _ = ca.capattn_bwd_ex(q, k, v, o2, lse2, torch.zeros_like(do), ap, temp, dlse=dlse)
    assert torch.equal(qq.grad, dq0) and torch.equal(kk.grad, dk0) and torch.equal(vv.grad, dv0)


# ---------------------------------------------------------------------------
# Every mask family with the fixed reference (a cap, no temperature, no m / l
# requested): the persistent forward then takes each row's live keys from the
# pre-pass spans and its key tiles from the visit sets.
# ---------------------------------------------------------------------------

PERSISTENT_MASK_CASES = [
    # (B, L, Hq, Hkv, D, cap, mask)
    (2, 600, 4, 2, 128, "tanh", "window"),
    (1, 333, 2, 2, 128, "soft_sign", "window_nc"),
    (2, 515, 4, 4, 128, "tanh", "packed"),
    (2, 640, 4, 1, 128, "tanh", "ranker"),
    (1, 260, 2, 2, 128, "alsc", "packed"),
    (2, 450, 4, 2, 64, "soft_sign", "ranker"),
    (1, 700, 2, 1, 64, "tanh", "window"),
]


@pytest.mark.parametrize("case", PERSISTENT_MASK_CASES, ids=lambda c: "-".join(map(str, c)))
def test_persistent_forward_with_masks(case):
    B, L, Hq, Hkv, D, cap, mask = case
    inp = make_case(B, L, Hq, Hkv, D, torch.bfloat16, mask, False, seed=L + 13 * Hq + D)
    ap = params(cap, mask, 0.0)
    got = run_gpu(inp, ap, torch.bfloat16)
    ref = run_oracle(inp, ap)
    compare(got, ref, torch.bfloat16)
    dead = np.isneginf(ref["LSE"])
    if dead.any():
        assert np.all(np.transpose(got["O"], (0, 2, 1, 3))[dead] == 0)


# ---------------------------------------------------------------------------
# Ranker bounds that leave whole query tiles without a live key next to live
# ones (the two-tile forward then has an idle tile in a CTA with work): O and
# the gradients of the dead rows must be exactly zero, the rest match.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bounds_row", [(0, 60, 60, 100), (0, 200, 200, 250), (0, 0, 0, 90)])
def test_ranker_with_dead_query_tiles(bounds_row):
    B, L = 2, 700
    inp = make_case(B, L, 4, 2, 128, torch.bfloat16, "ranker", False, seed=sum(bounds_row))
    inp["bounds"] = np.array([bounds_row, (0, 300, 300, 380)], np.int32)
    ap = params("alsc", "ranker", 0.0)
    for _ in range(3):
        got = run_gpu(inp, ap, torch.bfloat16)
        ref = run_oracle(inp, ap)
        compare(got, ref, torch.bfloat16)
        dead = np.isneginf(ref["LSE"])  # [B, Hq, L]
        o = np.transpose(got["O"], (0, 2, 1, 3))[dead]
        assert dead.any() and np.all(o == 0)


# ---------------------------------------------------------------------------
# Backward reusing the forward's spans and visit maps (CAPATTN_BWD_REUSE_FWD_MAPS).
# ---------------------------------------------------------------------------

REUSE_CASES = [
    # (dtype, D, B, L, Hq, Hkv, cap, mask)
    ("bf16", 128, 2, 700, 4, 2, "tanh", "packed"),
    ("bf16", 128, 2, 400, 4, 2, "soft_sign", "ranker"),
    ("bf16", 64, 1, 4200, 2, 1, "alsc", "window"),
    ("bf16", 128, 1, 4200, 2, 2, "tanh", "causal"),
    ("fp32", 64, 2, 300, 4, 2, "tanh", "packed"),
]


@pytest.mark.parametrize("want_dt", [True, False], ids=["dtemp", "no_dtemp"])
@pytest.mark.parametrize("case", REUSE_CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward_reusing_the_forward_maps_is_bit_identical(case, want_dt):
    """The forward runs on a workspace whose bytes were all 0xFF (only the
    status word zeroed), so maps (and, without dtemp on bf16, dX slots) that
    were not written would show; the backward that reuses the forward's maps,
    twice in a row, must give the same bits as a backward that rebuilds them on
    a fresh workspace."""
    dname, D, B, L, Hq, Hkv, cap, mask = case
    dtype = torch.bfloat16 if dname == "bf16" else torch.float32
    inp = make_case(B, L, Hq, Hkv, D, dtype, mask, True, seed=L + 5)
    ap = params(cap, mask, 1e-3)
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("q", "k", "v", "do"))
    temp, seg, bounds = to_dev(inp["temp"]), to_dev(inp["seg"]), to_dev(inp["bounds"])
    cfg = ca.make_config(ap, B, L, Hq, Hkv, D, dtype)
    ws = ca.new_workspace(cfg, q.device)
    ws.fill_(0xFF)
    ws[:4].zero_()
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp, seg, bounds, workspace=ws)
    dlse = torch.randn(B, Hq, L, device="cuda")
    ref = ca.capattn_bwd_ex(q, k, v, o, lse, do, ap, temp, seg, bounds, dlse=dlse, want_dtemp=want_dt)
    for _ in range(2):
        got = ca.capattn_bwd_ex(q, k, v, o, lse, do, ap, temp, seg, bounds, dlse=dlse,
                                want_dtemp=want_dt, workspace=ws, reuse_fwd_maps=True)
        for name, a, b in zip(("dq", "dk", "dv", "delta", "dtemp"), got, ref):
            assert (a is None and b is None) or torch.equal(a, b), name
    assert ca.capattn_device_status(ws) == (0, 0)


def test_reuse_needs_the_forward_workspace():
    inp = make_case(1, 200, 2, 2, 128, torch.bfloat16, "causal", False, seed=3)
    ap = params("tanh", "causal", 0.0)
    q, k, v, do = (to_dev(inp[n], torch.bfloat16) for n in ("q", "k", "v", "do"))
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap)
    with pytest.raises(ValueError):
        ca.capattn_bwd_ex(q, k, v, o, lse, do, ap, reuse_fwd_maps=True)


# ---------------------------------------------------------------------------
# Ranker bounds from history / candidate segment ids (bit-exact).
# ---------------------------------------------------------------------------

def test_ranker_bounds_from_ids_bit_exact():
    rng = np.random.default_rng(123)
    H, C, B, L = 11, 12, 16, 4096
    seg = np.full((B, L), 5, np.int32)
    for b in range(B):
        kind = b % 4
        hl = int(rng.integers(0, 64))
        hu = hl + int(rng.integers(1, 2048))
        cu = min(L, hu + int(rng.integers(16, 128)))
        if kind != 2:                       # kind 2: no history
            seg[b, hl:hu] = H
        if kind != 1:                       # kind 1: no candidates
            seg[b, hu:cu] = C
        if kind == 3:                       # kind 3: a gap in the history run
            seg[b, (hl + hu) // 2] = 5
    ref, contiguous = orc.ranker_bounds_from_ids(seg, H, C)
    cfg = ca.make_config(ca.AttnParams(sm_scale=0.1), B, L, 2, 2, 128, torch.bfloat16)
    ws = ca.new_workspace(cfg, torch.device("cuda"))
    got = ca.ranker_bounds_from_ids(to_dev(seg), H, C, workspace=ws).cpu().numpy()
    assert np.array_equal(got, ref)
    st, bits = ca.capattn_device_status(ws)
    assert (bits & 8) != 0 and not contiguous.all()
    # contiguous rows only: no flag
    ok_rows = np.nonzero(contiguous)[0]
    got2 = ca.ranker_bounds_from_ids(to_dev(seg[ok_rows]), H, C, workspace=ws).cpu().numpy()
    assert np.array_equal(got2, ref[ok_rows])
    assert ca.capattn_device_status(ws) == (0, 0)
