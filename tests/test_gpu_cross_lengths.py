"""GPU parity with unequal query and key lengths (q [B, Lq, Hq, D], k / v
[B, Lk, Hkv, D]; positions compared directly), through the C ABI, against the
fp64 oracle on the same rounded inputs."""

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca
from soft_capped_attention_gb300.workloads import round_to_bf16

from parity_utils import compare, oracle_cfg, rel_fro, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

CAPS = {"none": (0.0, 0.0, 0.0), "tanh": (50.0, 0.0, 0.0), "soft_sign": (20.0, 0.0, 0.0),
        "alsc": (30.0, 2.0, 0.5)}
MASKS = {"full": (False, 0), "causal": (True, 0), "window": (True, 200), "window_nc": (False, 77)}


def make_case(B, Lq, Lk, Hq, Hkv, D, dtype, seed, temp=True):
    rng = np.random.default_rng(seed)
    r = lambda *s: rng.standard_normal(s).astype(np.float32)
    inp = {"q": r(B, Lq, Hq, D), "k": r(B, Lk, Hkv, D), "v": r(B, Lk, Hkv, D), "do": r(B, Lq, Hq, D)}
    if dtype == torch.bfloat16:
        for n in ("q", "k", "v", "do"):
            inp[n] = round_to_bf16(inp[n])
    inp["temp"] = rng.uniform(0.5, 1.5, size=(B, Lq)).astype(np.float32) if temp else None
    inp["seg"] = None
    inp["bounds"] = None
    return inp


def params(cap, mask, z=0.0, D=128):
    c, a, b = CAPS[cap]
    causal, window = MASKS[mask]
    return ca.AttnParams(sm_scale=float(1.0 / np.sqrt(D)), cap_method=cap, cap=c, alpha=a, beta=b,
                         causal=causal, window_len=window, z_loss_weight=z)


SHAPES = [(300, 700), (700, 300), (129, 1000), (1000, 129)]
BF16_CASES = [(s, m, cap) for i, s in enumerate(SHAPES) for j, m in enumerate(MASKS)
              for cap in [list(CAPS)[(i + j) % 4]]]


@pytest.mark.parametrize("shape,mask,cap", BF16_CASES)
def test_cross_lengths_bf16_match_oracle(shape, mask, cap):
    Lq, Lk = shape
    inp = make_case(2, Lq, Lk, 4, 2, 128, torch.bfloat16, seed=Lq * 7 + Lk)
    ap = params(cap, mask, z=0.01)
    got = run_gpu(inp, ap, torch.bfloat16)
    ref = run_oracle(inp, ap)
    assert got["O"].shape == (2, Lq, 4, 128) and got["dK"].shape == (2, Lk, 2, 128)
    compare(got, ref, torch.bfloat16)


@pytest.mark.parametrize("shape,mask,cap", [((200, 333), "causal", "tanh"), ((333, 200), "window", "alsc"),
                                            ((65, 129), "full", "soft_sign")])
def test_cross_lengths_fp32_match_oracle(shape, mask, cap):
    Lq, Lk = shape
    inp = make_case(2, Lq, Lk, 4, 2, 64, torch.float32, seed=Lq + Lk)
    ap = params(cap, mask, D=64)
    compare(run_gpu(inp, ap, torch.float32), run_oracle(inp, ap), torch.float32)


def test_cross_lengths_dtemp_and_autograd():
    Lq, Lk = 257, 520
    inp = make_case(1, Lq, Lk, 2, 1, 128, torch.bfloat16, seed=5)
    ap = params("tanh", "causal")
    q, k, v, do = (to_dev(inp[n], torch.bfloat16).requires_grad_(n != "do") for n in ("q", "k", "v", "do"))
    temp = to_dev(inp["temp"]).requires_grad_(True)
    o = ca.attention(q, k, v, ap, temp)
    (o.float() * do.float()).sum().backward()
    cfg = oracle_cfg(ap)
    O, LSE, _, _ = orc.forward(inp["q"], inp["k"], inp["v"], inp["temp"], None, None, cfg)
    dQ, dK, dV, _ = orc.backward(inp["q"], inp["k"], inp["v"], inp["temp"], None, None, O, LSE, inp["do"], cfg)
    dT = orc.backward_dtemp(inp["q"], inp["k"], inp["v"], inp["temp"], None, None, O, LSE, inp["do"], cfg)
    assert float(np.max(np.abs(o.detach().float().cpu().numpy() - O))) <= 2e-2
    for g, r in ((q.grad, dQ), (k.grad, dK), (v.grad, dV), (temp.grad, dT)):
        assert rel_fro(g.float().cpu().numpy(), r) <= 2e-2


@pytest.mark.parametrize("shape,mask", [((300, 700), "causal"), ((1000, 129), "window"),
                                        ((129, 1000), "window_nc")])
def test_cross_lengths_device_visit_maps_match_host(shape, mask):
    Lq, Lk = shape
    ap = params("tanh", mask)
    cfg = ca.make_config(ap, 2, Lq, 4, 2, 128, torch.bfloat16, Lk=Lk)
    for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
        host = ca.capattn_visit_map_host(cfg, None, None, which)
        dev = ca.capattn_visit_map_device(cfg, None, None, which)
        assert np.array_equal(host, dev)
