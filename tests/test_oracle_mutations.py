"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's source (a dropped term,
a flipped sign, an off-by-one, a wrong operand or index), loads that copy in a
fresh process in place of the oracle, and runs the pin suite
(test_oracle_pins.py) against it: the suite must fail.  A control run with no
mistake must pass, so a failure is the planted mistake's and not the harness's.
Nothing here touches the CUDA library; the mistakes live on the CPU only.
"""

import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle", "capattn_oracle.py")

# (name, text in the oracle, replacement, how many occurrences to replace)
MUTATIONS = [
    # caps and their derivatives
    ("tanh_without_cap_factor", "return c * np.tanh(s / c)", "return np.tanh(s / c)", 1),
    ("soft_sign_without_abs", "return s / (1.0 + np.abs(s) / c)", "return s / (1.0 + s / c)", 1),
    ("alsc_without_denominator", "return c * (_sigmoid(z) - sb) / denom",
     "return c * (_sigmoid(z) - sb)", 1),
    ("alsc_beta_sign", "z = cfg.alpha * (s / c + cfg.beta)", "z = cfg.alpha * (s / c - cfg.beta)", 1),
    ("alsc_shift_sign", "sb = 1.0 / (1.0 + math.exp(-alpha * beta))",
     "sb = 1.0 / (1.0 + math.exp(alpha * beta))", 1),
    ("alsc_epsilon", "sb * (1.0 - sb) + 1e-12", "sb * (1.0 - sb) + 1e-6", 1),
    ("tanh_derivative_unsquared", "return 1.0 - t * t", "return 1.0 - t", 1),
    ("soft_sign_derivative_unsquared", "return r * r", "return r", 1),
    ("alsc_derivative_without_alpha", "return cfg.alpha * sz * (1.0 - sz) / denom",
     "return sz * (1.0 - sz) / denom", 1),
    # masks
    ("causal_strict", "M &= i >= j", "M &= i > j", 1),
    ("window_inclusive", "M &= j > i - cfg.window_len", "M &= j >= i - cfg.window_len", 1),
    ("segments_ordered_not_equal", "M &= seg_row[i] == seg_row[j]", "M &= seg_row[i] >= seg_row[j]", 1),
    ("ranker_without_self_term", " | (q_cand & k_cand & (i == j))", "", 1),
    ("ranker_candidates_see_candidates", "(q_cand & k_cand & (i == j))", "(q_cand & k_cand)", 1),
    ("ranker_history_keys_only_for_history", "(k_hist & (q_hist | q_cand))", "(k_hist & q_hist)", 1),
    # forward
    ("temperature_inside_the_cap", "t = temp_rows[:, None] * cap_forward(s, cfg)",
     "t = cap_forward(temp_rows[:, None] * s, cfg)", 2),
    ("lse_without_max", "m_safe + np.log(", "np.log(", 1),
    ("p_normalised_by_max", "- lse_safe[:, None]), 0.0)\n    O = P @ v",
     "- m_safe[:, None]), 0.0)\n    O = P @ v", 1),
    ("gqa_heads_interleaved", "g = h // G", "g = h % Hkv", 1),
    ("scores_without_scale", "s = cfg.sm_scale * (q_rows @ k.T)", "s = q_rows @ k.T", 2),
    ("m_over_masked_keys", "m = t_live.max(axis=1)", "m = t.max(axis=1)", 1),
    ("l_without_max_shift", "e = np.where(M, np.exp(np.where(M, t, 0.0) - m_safe[:, None]), 0.0)",
     "e = np.where(M, np.exp(np.where(M, t, 0.0)), 0.0)", 1),
    ("masked_p_leaks", "P = np.where(M, np.exp(np.where(M, t, 0.0) - lse_safe[:, None]), 0.0)\n    O = P @ v",
     "P = np.exp(t - lse_safe[:, None])\n    O = P @ v", 1),
    ("window_two_sided", "M &= j > i - cfg.window_len",
     "M &= (j > i - cfg.window_len) & (j < i + cfg.window_len)", 1),
    ("dead_row_lse_zero", "np.log(np.where(live, l, 1.0)), -np.inf)",
     "np.log(np.where(live, l, 1.0)), 0.0)", 1),
    # backward
    ("backward_without_delta", "dT = P * (dP - delta_rows[:, None])", "dT = P * dP", 1),
    ("z_loss_sign", "+ cfg.z_loss_weight * P * lse_safe[:, None]\n    if dlse_rows",
     "- cfg.z_loss_weight * P * lse_safe[:, None]\n    if dlse_rows", 1),
    ("backward_masked_p_leaks",
     "P = np.where(M, np.exp(np.where(M, t, 0.0) - lse_safe[:, None]), 0.0)\n    dP = do_rows @ v.T",
     "P = np.exp(t - lse_safe[:, None])\n    dP = do_rows @ v.T", 1),
    ("dlse_dropped", "dT = dT + P * np.where(live, dlse_rows, 0.0)[:, None]", "dT = dT", 1),
    ("dx_without_scale", "dX = cfg.sm_scale * cap_derivative(s, cfg)", "dX = cap_derivative(s, cfg)", 1),
    ("dx_without_temperature", "* temp_rows[:, None] * dT", "* dT", 1),
    ("dv_from_dx", "dX.T @ q_rows, P.T @ do_rows", "dX.T @ q_rows, dX.T @ do_rows", 1),
    ("dk_from_do", "return dX @ k, dX.T @ q_rows", "return dX @ k, dX.T @ do_rows", 1),
    ("delta_from_o_squared", 'delta = np.einsum("blhd,blhd->bhl", O, dO)',
     'delta = np.einsum("blhd,blhd->bhl", O, O)', 1),
    ("dk_not_summed_over_group", "dK[b, :, g] += dk", "dK[b, :, g] = dk", 1),
    ("loss_without_half", "0.5 * cfg.z_loss_weight * np.sum(lse ** 2)",
     "cfg.z_loss_weight * np.sum(lse ** 2)", 1),
    # temperature gradient
    ("dtemp_times_score", "dtemp[b, rows] += np.sum(dT * c, axis=1)",
     "dtemp[b, rows] += np.sum(dT * s, axis=1)", 1),
    ("dtemp_without_z_loss", "+ cfg.z_loss_weight * P * lse_safe[:, None]\n                if dLSE",
     "\n                if dLSE", 1),
    ("dtemp_first_head_only", "dtemp[b, rows] += np.sum(dT * c, axis=1)",
     "dtemp[b, rows] += np.sum(dT * c, axis=1) if h == 0 else 0.0", 1),
    ("dtemp_without_dlse", "dT = dT + P * np.where(live, dLSE[b, h, rows], 0.0)[:, None]",
     "dT = dT", 1),
    # ranker bounds, visit matrices, pair counts, row blocks
    ("ranker_bounds_inclusive_end", "int(pos[-1]) + 1", "int(pos[-1])", 1),
    ("ranker_gaps_not_flagged", "if hi - lo != pos.size", "if hi - lo < pos.size", 1),
    ("visit_rows_by_kv_block", "qt = rows // block_q", "qt = rows // block_kv", 1),
    ("visit_column_short", "M[:, kt * block_kv:(kt + 1) * block_kv]",
     "M[:, kt * block_kv:(kt + 1) * block_kv - 1]", 1),
    ("pair_count_without_bounds", "total += int(mask_rows(rows, Lk, cfg, s_row, b_row).sum())",
     "total += int(mask_rows(rows, Lk, cfg, s_row, None).sum())", 1),
    ("row_block_short", "rows = np.arange(r0, min(L, r0 + ROW_BLOCK))\n            M = mask_rows(rows, Lk, cfg, s_row, b_row)\n            for h in range(Hq):\n                g = h // G\n                o,",
     "rows = np.arange(r0, min(L, r0 + ROW_BLOCK - 1))\n            M = mask_rows(rows, Lk, cfg, s_row, b_row)\n            for h in range(Hq):\n                g = h // G\n                o,", 1),
]

DRIVER = r"""
import importlib.util, json, sys
root, old, new, count = sys.argv[1], *json.loads(sys.argv[2])
sys.path.insert(0, root)
import oracle
path = root + "/oracle/capattn_oracle.py"
src = open(path).read()
if old:
    assert src.count(old) >= count, "mutation text not found"
    src = src.replace(old, new, count)
name = "oracle.capattn_oracle"
mod = importlib.util.module_from_spec(importlib.util.spec_from_loader(name, loader=None))
mod.__file__ = path
sys.modules[name] = mod
exec(compile(src, path, "exec"), mod.__dict__)
oracle.capattn_oracle = mod
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", root + "/tests/test_oracle_pins.py"]))
"""


def _run(old, new, count):
    r = subprocess.run([sys.executable, "-c", DRIVER, ROOT, json.dumps([old, new, count])],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    return r.returncode, r.stdout[-3000:] + r.stderr[-3000:]


@pytest.fixture(scope="module")
def runs():
    """Every mutant's pin run, started together on a few host cores."""
    pool = ThreadPoolExecutor(max_workers=max(1, min(8, (os.cpu_count() or 2) // 2)))
    futures = {name: pool.submit(_run, old, new, count) for name, old, new, count in MUTATIONS}
    yield futures
    pool.shutdown(wait=True)


def test_mutation_texts_are_in_the_oracle():
    src = open(ORACLE).read()
    for name, old, _, count in MUTATIONS:
        assert src.count(old) >= count, name


def test_unmutated_oracle_passes_the_pins():
    rc, out = _run("", "", 0)
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_the_planted_mistake(runs, name, old, new, count):
    rc, out = runs[name].result()
    # exit code 1: tests ran and at least one failed (2-4 would be a usage,
    # collection or internal error, which proves nothing)
    assert rc == 1, f"{name}: pin suite exit code {rc}\n{out}"
