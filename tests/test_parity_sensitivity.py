"""The GPU parity tests would catch plausible kernel mistakes.

Each mistake of test_oracle_mutations.py that changes what the kernels
compute is planted in a copy of the oracle, which then stands in for a
faulty kernel: its outputs on the inputs of one GPU parity case go through
that case's own comparison against the true oracle, which must reject them.
A tolerance loose enough to let such a mistake through would fail here,
without a GPU.  Mistakes in parts the kernels do not compute (ranker bounds
from ids, visit matrices, pair counts, the loss helper) are left to the
bit-exact CPU tests, and a 1e-12 to 1e-6 change of ALSC's epsilon moves
results by ~1e-5, below any tolerance and harmless.
"""

import os
import sys
import types

import numpy as np
import pytest
import torch

from parity_utils import compare, oracle_cfg, rel_fro
from test_oracle_mutations import MUTATIONS
import test_gpu_parity as tp
import test_gpu_tanh_curved as tc
import test_gpu_z_loss as tz

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "capattn_oracle.py")).read()

NOT_KERNEL = {"ranker_bounds_inclusive_end", "ranker_gaps_not_flagged", "visit_rows_by_kv_block",
              "visit_column_short", "pair_count_without_bounds", "loss_without_half", "alsc_epsilon"}

TANH_CAUSAL = ("bf16", tp.BF16_CASES[1])     # (2, 300, 4, 2, tanh, causal)
ALSC_WINDOW = ("bf16", tp.BF16_CASES[2])     # (1, 513, 4, 1, alsc, window, temp, z 1e-4)
SOFTSIGN_PACKED = ("bf16", tp.BF16_CASES[3])
ALSC_RANKER = ("bf16", tp.BF16_CASES[4])
TANH_WINDOW_NC = ("bf16", tp.BF16_CASES[5])
FP32_WINDOW = ("fp32", tp.FP32_CASES[6])     # (1, 300, 2, 1, 64, tanh, window 200)
FP32_WINDOW_NC = ("fp32", tp.FP32_CASES[7])  # (2, 190, 2, 2, 128, soft_sign, window 77, not causal)

# mistake -> the GPU parity case whose comparison has to reject it
CATCHER = {
    "tanh_without_cap_factor": TANH_CAUSAL,
    "soft_sign_without_abs": SOFTSIGN_PACKED,
    "alsc_without_denominator": ALSC_WINDOW,
    "alsc_beta_sign": ALSC_WINDOW,
    "alsc_shift_sign": ALSC_WINDOW,
    "tanh_derivative_unsquared": ("curved", tc.CASES[0]),
    "soft_sign_derivative_unsquared": SOFTSIGN_PACKED,
    "alsc_derivative_without_alpha": ALSC_WINDOW,
    "causal_strict": TANH_CAUSAL,
    "window_inclusive": ALSC_WINDOW,
    "segments_ordered_not_equal": SOFTSIGN_PACKED,
    "ranker_without_self_term": ALSC_RANKER,
    "ranker_candidates_see_candidates": ALSC_RANKER,
    "ranker_history_keys_only_for_history": ALSC_RANKER,
    "temperature_inside_the_cap": ALSC_WINDOW,
    "lse_without_max": TANH_CAUSAL,
    "p_normalised_by_max": TANH_CAUSAL,
    "gqa_heads_interleaved": TANH_CAUSAL,
    "scores_without_scale": TANH_CAUSAL,
    "m_over_masked_keys": ("residuals", None),
    "l_without_max_shift": TANH_CAUSAL,
    "masked_p_leaks": TANH_CAUSAL,
    "window_two_sided": TANH_WINDOW_NC,
    "dead_row_lse_zero": ALSC_RANKER,
    "backward_without_delta": TANH_CAUSAL,
    "z_loss_sign": ("z", tz.CASES[0]),
    "backward_masked_p_leaks": TANH_CAUSAL,
    "dlse_dropped": ("lse_grad", tp.LSE_GRAD_CASES[0]),
    "dx_without_scale": TANH_CAUSAL,
    "dx_without_temperature": ALSC_WINDOW,
    "dv_from_dx": TANH_CAUSAL,
    "dk_from_do": TANH_CAUSAL,
    "delta_from_o_squared": TANH_CAUSAL,
    "dk_not_summed_over_group": TANH_CAUSAL,
    "dtemp_times_score": ("dtemp", tp.DTEMP_CASES[1]),
    "dtemp_without_z_loss": ("dtemp", tp.DTEMP_CASES[3]),
    "dtemp_first_head_only": ("dtemp", tp.DTEMP_CASES[0]),
    "dtemp_without_dlse": ("lse_grad", tp.LSE_GRAD_CASES[1]),
    "row_block_short": ALSC_WINDOW,
}


def _oracle(old="", new="", count=0):
    mod = types.ModuleType("planted_oracle")
    sys.modules[mod.__name__] = mod  # dataclasses look the module up while the class is built
    exec(compile(SRC.replace(old, new, count) if old else SRC, "capattn_oracle.py", "exec"), mod.__dict__)
    return mod


def _cfg(mod, ap):
    oc = oracle_cfg(ap)
    return mod.OracleConfig(sm_scale=oc.sm_scale, cap_method=oc.cap_method, cap=oc.cap, alpha=oc.alpha,
                            beta=oc.beta, causal=oc.causal, window_len=oc.window_len,
                            z_loss_weight=oc.z_loss_weight)


def _outputs(mod, inp, ap, dlse=None, dtemp=False):
    c = _cfg(mod, ap)
    args = (inp["q"], inp["k"], inp["v"], inp["temp"], inp["seg"], inp["bounds"])
    with np.errstate(divide="ignore"):  # some planted mistakes take log(0) on dead rows
        O, LSE, m, l = mod.forward(*args, c)
    dQ, dK, dV, _ = mod.backward(*args, O, LSE, inp["do"], c, dLSE=dlse)
    out = {"O": O, "LSE": LSE, "m": m, "l": l, "dQ": dQ, "dK": dK, "dV": dV}
    if dtemp:
        out["dtemp"] = mod.backward_dtemp(*args, O, LSE, inp["do"], c, dLSE=dlse)
    return out


def _rejected(kind, case, bad, good):
    """Whether the GPU test of this kind rejects `bad`'s outputs (True) or
    would pass them (False); each branch repeats that test's assertions."""
    try:
        if kind == "fp32":  # test_fp32_matches_oracle
            B, L, Hq, Hkv, D, cap, mask, temp, z = case
            inp = tp.make_case(B, L, Hq, Hkv, D, torch.float32, mask, temp, seed=L * 3 + D)
            ap = tp.params(cap, mask, z)
            compare(_outputs(bad, inp, ap), _outputs(good, inp, ap), torch.float32)
        elif kind in ("bf16", "curved", "z"):
            if kind == "bf16":
                B, L, Hq, Hkv, cap, mask, temp, z = case
                inp = tp.make_case(B, L, Hq, Hkv, 128, torch.bfloat16, mask, temp, seed=L * 7 + Hq)
                ap = tp.params(cap, mask, z)
            else:
                inp, ap = (tc if kind == "curved" else tz)._case(case)
            compare(_outputs(bad, inp, ap), _outputs(good, inp, ap), torch.bfloat16)
        elif kind == "residuals":  # test_residuals_m_l_and_delta_bf16
            inp = tp.make_case(2, 300, 4, 2, 128, torch.bfloat16, "ranker", True, seed=5)
            ap = tp.params("tanh", "ranker", 0.0)
            got, ref = _outputs(bad, inp, ap), _outputs(good, inp, ap)
            live = np.isfinite(ref["LSE"])
            np.testing.assert_allclose(got["m"][live], ref["m"][live], atol=1e-3)
            np.testing.assert_allclose(got["l"][live], ref["l"][live], rtol=5e-3)
        elif kind == "dtemp":  # test_dtemp_bf16_matches_oracle
            B, L, Hq, Hkv, cap, mask, z = case
            inp = tp.make_case(B, L, Hq, Hkv, 128, torch.bfloat16, mask, True, seed=L + 7)
            ap = tp.params(cap, mask, z)
            got, ref = _outputs(bad, inp, ap, dtemp=True), _outputs(good, inp, ap, dtemp=True)
            assert rel_fro(got["dtemp"], ref["dtemp"]) <= 2e-2
        elif kind == "lse_grad":  # test_lse_gradient_matches_oracle (bf16 cases)
            dname, D, B, L, Hq, Hkv, cap, mask, z, want_dt = case
            assert dname == "bf16"
            inp = tp.make_case(B, L, Hq, Hkv, D, torch.bfloat16, mask, True, seed=L + 99)
            dlse = np.random.default_rng(L).standard_normal((B, Hq, L)).astype(np.float32).astype(np.float64)
            ap = tp.params(cap, mask, z)
            got = _outputs(bad, inp, ap, dlse=dlse, dtemp=want_dt)
            ref = _outputs(good, inp, ap, dlse=dlse, dtemp=want_dt)
            for n in ("dQ", "dK", "dV") + (("dtemp",) if want_dt else ()):
                assert rel_fro(got[n], ref[n]) <= 2e-2, n
        else:
            raise ValueError(kind)
    except AssertionError:
        return True
    return False


# the fp32 path has kernels of its own: its window cases must catch the window mistakes too
FP32_CATCHER = {"window_inclusive": FP32_WINDOW, "window_two_sided": FP32_WINDOW_NC,
                "causal_strict": FP32_WINDOW}


def test_every_kernel_mistake_has_a_catcher():
    names = {m[0] for m in MUTATIONS}
    assert set(CATCHER) | NOT_KERNEL == names
    assert not set(CATCHER) & NOT_KERNEL


@pytest.mark.parametrize("name,old,new,count", [m for m in MUTATIONS if m[0] in CATCHER],
                         ids=[m[0] for m in MUTATIONS if m[0] in CATCHER])
def test_gpu_comparison_rejects_the_mistake(name, old, new, count):
    kind, case = CATCHER[name]
    assert _rejected(kind, case, _oracle(old, new, count), _oracle()), name


@pytest.mark.parametrize("name", sorted(FP32_CATCHER))
def test_fp32_comparison_rejects_the_window_mistakes(name):
    _, old, new, count = next(m for m in MUTATIONS if m[0] == name)
    kind, case = FP32_CATCHER[name]
    assert _rejected(kind, case, _oracle(old, new, count), _oracle()), name


def test_gpu_comparisons_accept_the_true_oracle():
    # the control: every catcher passes the unmodified oracle's own outputs
    good = _oracle()
    for kind, case in {(k, c) for k, c in list(CATCHER.values()) + list(FP32_CATCHER.values())}:
        assert not _rejected(kind, case, good, good), (kind, case)
