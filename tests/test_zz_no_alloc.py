"""GPU test of capattn_fwd_noalloc, the forward for callers that cannot
allocate device memory (plugins in frameworks that own all memory, services
with a fixed memory budget).  It must give the same results as capattn_fwd,
which takes a caller-provided workspace, and keep doing so on consecutive
calls that share its fixed scratch array.  Collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from soft_capped_attention_gb300 import capattn as ca

pytestmark = pytest.mark.gpu

TOL_O = 2e-2     # bf16 output, max-abs
TOL_LSE = 1e-3   # max-abs on live rows, -inf identical


def _noalloc():
    fn = ca.lib().capattn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ca.CapattnConfig)] + [ctypes.c_void_p] * 10 + [ctypes.c_void_p]
    return fn


def _inputs(seed, B, L, Hq, Hkv):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, Hq, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, L, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, L, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    temp = (0.5 + torch.rand(B, L, generator=g)).cuda()
    seg = torch.cumsum((torch.rand(B, L, generator=g) < 0.01).to(torch.int32), dim=1).to(torch.int32).cuda()
    return q, k, v, temp, seg


def _check_same(o, lse, o_ref, lse_ref):
    assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O
    assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
    fin = torch.isfinite(lse_ref)
    assert (lse[fin] - lse_ref[fin]).abs().max().item() <= TOL_LSE


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    fn = _noalloc()
    ap = ca.AttnParams(sm_scale=1 / np.sqrt(128), cap_method="alsc", cap=30.0, alpha=2.0,
                       beta=0.5, causal=True, window_len=300)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, (seed, B, L, Hq, Hkv) in enumerate(((1, 2, 700, 4, 2), (2, 1, 1000, 2, 2))):
        q, k, v, temp, seg = _inputs(seed, B, L, Hq, Hkv)
        cfg = ca.make_config(ap, B, L, Hq, Hkv, 128, torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, L, dtype=torch.float32, device="cuda")
        st = fn(ctypes.byref(cfg), *(ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, temp, seg)),
                None, ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), None, None,
                stream)
        assert st == 0, f"call {call}: status {st}"
        o_ref, lse_ref, _, _ = ca.capattn_fwd(q, k, v, ap, temp, seg, None)
        torch.cuda.synchronize()
        _check_same(o, lse, o_ref, lse_ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _noalloc()
    ap = ca.AttnParams(sm_scale=0.1)
    cfg = ca.make_config(ap, 64, 16384, 1, 1, 128, torch.bfloat16)  # 16 MiB of row spans
    dummy = ctypes.c_void_p(256)
    st = fn(ctypes.byref(cfg), dummy, dummy, dummy, None, None, None, dummy, dummy, None, None,
            None)
    assert st == 7
    assert ca.lib().capattn_status_string(7) == b"problem exceeds the fixed scratch of capattn_fwd_noalloc"
