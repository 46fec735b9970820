"""Failure detection on the GPU without a fault: the kernels' bounded waits.

Every mbarrier wait in the tcgen05 kernels gives up after a time limit,
records the timeout bit in the status word, raises the CTA's abort flag and
lets the CTA free its TMEM and return.  capattn_check_bounded_wait runs that
protocol on every SM with a wait that nothing satisfies and a limit of
microseconds; the test reads the timeout through capattn_device_status and
then shows that the attention kernels still run on every SM and give the same
results as before (a TMEM allocation left behind would stall them, a broken
context would fail them).
"""

import numpy as np
import pytest
import torch

from soft_capped_attention_gb300 import capattn as ca

from parity_utils import compare, run_gpu, run_oracle, to_dev
from test_gpu_parity import make_case, params

pytestmark = pytest.mark.gpu


def _step(inp, ap, ws):
    q, k, v, do = (to_dev(inp[n], torch.bfloat16) for n in ("q", "k", "v", "do"))
    temp = to_dev(inp["temp"])
    o, lse, _, _ = ca.capattn_fwd(q, k, v, ap, temp, workspace=ws)
    dq, dk, dv, _ = ca.capattn_bwd(q, k, v, o, lse, do, ap, temp, workspace=ws)
    return [t.clone() for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("limit_ns", [2_000, 50_000])
def test_wait_timeout_is_reported_and_kernels_recover(limit_ns):
    dev = torch.device("cuda")
    # a grid larger than the SM count in every kernel (B=2, H=16, L=2048)
    big = make_case(2, 2048, 16, 16, 128, torch.bfloat16, "causal", True, seed=58)
    ap = params("tanh", "causal", 0.0)
    cfg = ca.make_config(ap, 2, 2048, 16, 16, 128, torch.bfloat16)
    ws = ca.new_workspace(cfg, dev)
    before = _step(big, ap, ws)
    assert ca.capattn_device_status(ws) == (0, 0)

    ca.capattn_check_bounded_wait(ws, limit_ns)
    st, bits = ca.capattn_device_status(ws)
    assert st == 4 and bits == 1, (st, bits)
    assert ca.capattn_device_status(ws) == (0, 0)  # read and cleared

    after = _step(big, ap, ws)
    assert ca.capattn_device_status(ws) == (0, 0)
    for a, b in zip(before, after):
        assert torch.equal(a, b)
    # and a small case against the oracle
    inp = make_case(2, 700, 4, 2, 128, torch.bfloat16, "causal", True, seed=57)
    compare(run_gpu(inp, ap, torch.bfloat16), run_oracle(inp, ap), torch.bfloat16)
