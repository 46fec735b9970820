"""GPU test of capattn_fwd_noalloc, the forward for callers that cannot
allocate device memory (plugins in frameworks that own all memory, services
with a fixed memory budget).  It must give the same results as capattn_fwd,
which takes a caller-provided workspace, and keep doing so on consecutive
calls that share its fixed scratch array: a small problem, then one whose
scratch is close to the array's 8 MiB, so that the second call's spans and
visit maps sit over the first call's.  The calls after the first must leave
the device's free memory unchanged, and capattn_noalloc_status must report
the device-side status bits of the last call.  Collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

from soft_capped_attention_gb300 import capattn as ca

pytestmark = pytest.mark.gpu

TOL_O = 2e-2     # bf16 output, max-abs
TOL_LSE = 1e-3   # max-abs on live rows, -inf identical
SCRATCH = 8 << 20


def _noalloc():
    fn = ca.lib().capattn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ca.CapattnConfig)] + [ctypes.c_void_p] * 10 + [ctypes.c_void_p]
    return fn


def _status():
    fn = ca.lib().capattn_noalloc_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    bits = ctypes.c_uint32(0)
    st = fn(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def _inputs(seed, B, L, Hq, Hkv):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, L, Hq, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, L, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, L, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    temp = (0.5 + torch.rand(B, L, generator=g)).cuda()
    seg = torch.cumsum((torch.rand(B, L, generator=g) < 0.01).to(torch.int32), dim=1).to(torch.int32).cuda()
    return q, k, v, temp, seg


def _check_same(got, ref):
    o, lse, m, l = got
    o_ref, lse_ref, m_ref, l_ref = ref
    assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O
    assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
    fin = torch.isfinite(lse_ref)
    assert (lse[fin] - lse_ref[fin]).abs().max().item() <= TOL_LSE
    assert torch.equal(torch.isneginf(m), torch.isneginf(m_ref))
    assert (m[fin] - m_ref[fin]).abs().max().item() <= TOL_LSE
    assert ((l[fin] - l_ref[fin]).abs() / l_ref[fin]).max().item() <= TOL_LSE
    assert torch.all(l[~fin] == 0)


def _call(fn, cfg, q, k, v, temp, seg, out):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return fn(ctypes.byref(cfg), p(q), p(k), p(v), p(temp), p(seg), None, *(p(t) for t in out), stream)


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    fn = _noalloc()
    ap = ca.AttnParams(sm_scale=1 / np.sqrt(128), cap_method="alsc", cap=30.0, alpha=2.0,
                       beta=0.5, causal=True, window_len=300)
    # small first, then a problem whose forward scratch nearly fills the array
    shapes = ((1, 2, 700, 4, 2), (2, 3, 150_000, 2, 1))
    cfg_big = ca.make_config(ap, *shapes[1][1:], 128, torch.bfloat16)
    need = ca.workspace_bytes(cfg_big, ca.PASS_FWD)
    assert 0.9 * SCRATCH < need <= SCRATCH, need
    for call, (seed, B, L, Hq, Hkv) in enumerate(shapes):
        q, k, v, temp, seg = _inputs(seed, B, L, Hq, Hkv)
        cfg = ca.make_config(ap, B, L, Hq, Hkv, 128, torch.bfloat16)
        out = (torch.empty_like(q), torch.empty(B, Hq, L, dtype=torch.float32, device="cuda"),
               torch.empty(B, Hq, L, dtype=torch.float32, device="cuda"),
               torch.empty(B, Hq, L, dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        st = _call(fn, cfg, q, k, v, temp, seg, out)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert st == 0, f"call {call}: status {st}"
        if call > 0:  # the first call may load the library's module on this device
            assert free1 == free0, (free0, free1)
        assert _status() == (0, 0)
        ref = ca.capattn_fwd(q, k, v, ap, temp, seg, None, want_ml=True)
        torch.cuda.synchronize()
        _check_same(out, ref)
        del q, k, v, out, ref


def test_noalloc_status_reports_bad_segment_ids():
    fn = _noalloc()
    ap = ca.AttnParams(sm_scale=1 / np.sqrt(128), causal=True)
    q, k, v, _, seg = _inputs(5, 1, 300, 2, 2)
    cfg = ca.make_config(ap, 1, 300, 2, 2, 128, torch.bfloat16)
    out = (torch.empty_like(q), torch.empty(1, 2, 300, dtype=torch.float32, device="cuda"), None, None)
    bad = torch.flip(seg, dims=[1]).contiguous()  # decreasing ids: bit 2
    assert _call(fn, cfg, q, k, v, None, bad, out) == 0
    assert _status() == (6, 2)
    assert _status() == (0, 0)  # read and cleared
    assert _call(fn, cfg, q, k, v, None, seg, out) == 0
    assert _status() == (0, 0)


def test_noalloc_rejects_problems_beyond_its_scratch():
    fn = _noalloc()
    ap = ca.AttnParams(sm_scale=0.1)
    cfg = ca.make_config(ap, 64, 16384, 1, 1, 128, torch.bfloat16)  # 16 MiB of row spans
    dummy = ctypes.c_void_p(256)
    st = fn(ctypes.byref(cfg), dummy, dummy, dummy, None, None, None, dummy, dummy, None, None,
            None)
    assert st == 7
    assert ca.lib().capattn_status_string(7) == b"problem exceeds the fixed scratch of capattn_fwd_noalloc"
