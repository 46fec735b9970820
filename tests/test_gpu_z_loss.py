"""GPU parity with a z-loss weight large enough to matter.

The z-loss adds z * P * LSE to dT (mosaic_backward.py's form of the gradient
of (z/2) * sum of LSE^2).  In the other parity cases the weight is 0 or small
(1e-4 .. 0.05), where leaving the term out moves the gradients by at most
~3 %, about the tolerance.  Weights of 0.2 and 0.5 move them by 9-30 %
(checked on the CPU below), so these cases pin the term's sign and size in
both backward paths, for three caps and three mask families.
"""

import dataclasses

import numpy as np
import pytest
import torch

from parity_utils import compare, rel_fro, run_gpu, run_oracle
from test_gpu_parity import make_case, params

CASES = [
    # (B, L, Hq, Hkv, cap, mask, temp, z)
    (2, 300, 4, 2, "tanh", "causal", False, 0.5),
    (2, 384, 2, 2, "soft_sign", "packed", True, 0.2),
    (1, 513, 4, 1, "alsc", "window", True, 0.2),
]


def _case(case):
    B, L, Hq, Hkv, cap, mask, temp, z = case
    return make_case(B, L, Hq, Hkv, 128, torch.bfloat16, mask, temp, seed=L * 13 + Hq), params(cap, mask, z)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_cases_need_the_z_term(case):
    """CPU: without the z-loss term the oracle's dQ and dK move by more than
    three times the gradient tolerance."""
    inp, ap = _case(case)
    ref = run_oracle(inp, ap)
    plain = run_oracle(inp, dataclasses.replace(ap, z_loss_weight=0.0))
    for name in ("dQ", "dK"):
        assert rel_fro(plain[name], ref[name]) > 3 * 2e-2, name
    np.testing.assert_array_equal(plain["dV"], ref["dV"])  # dV does not see dT


@pytest.mark.gpu
@pytest.mark.parametrize("pool", [True, False], ids=["stored_dx", "recompute"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_large_z_loss_matches_oracle(case, pool):
    inp, ap = _case(case)
    compare(run_gpu(inp, ap, torch.bfloat16, pool=pool), run_oracle(inp, ap), torch.bfloat16)
