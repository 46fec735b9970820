"""Python binding of libcapattn.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; PyTorch only
provides device memory and the current stream.  The names mirror the C ABI in
include/capattn.h: ``capattn_fwd`` / ``capattn_bwd`` (device tensors),
``capattn_workspace_bytes``, ``capattn_device_status`` and the visit-map /
mask-bit debug exports.  ``CapAttnFunction`` wraps the pair as a
``torch.autograd.Function``.

There is no fallback: if the shared library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcapattn.so")

CAP_METHODS = {"none": 0, "tanh": 1, "soft_sign": 2, "alsc": 3}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}
PASS_FWD, PASS_BWD, PASS_BWD_NO_POOL = 0, 1, 2
VISIT_Q_TILES, VISIT_KV_TILES = 0, 1
BWD_REUSE_FWD_MAPS = 1
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
                4: "device wait timeout", 5: "workspace missing, misaligned or too small",
                6: "invalid device data (segment ids or ranker bounds)",
                7: "problem exceeds the fixed scratch of capattn_fwd_noalloc"}


class CapattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} (status {status})")


class CapattnConfig(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("cap_method", ctypes.c_int32),
                ("cap", ctypes.c_float), ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("sm_scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("window_len", ctypes.c_int32), ("z_loss_weight", ctypes.c_float),
                ("q_heads_per_kv_head", ctypes.c_int32), ("B", ctypes.c_int32),
                ("L", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("dtype", ctypes.c_int32), ("Lk", ctypes.c_int32)]


_lib_handle = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m soft_capped_attention_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
        cfgp = ctypes.POINTER(CapattnConfig)
        h.capattn_status_string.restype = ctypes.c_char_p
        h.capattn_status_string.argtypes = [ctypes.c_int]
        h.capattn_validate_config.restype = ctypes.c_int
        h.capattn_validate_config.argtypes = [cfgp]
        h.capattn_workspace_bytes.restype = sz
        h.capattn_workspace_bytes.argtypes = [cfgp, ctypes.c_int]
        h.capattn_tile_sizes.restype = ctypes.c_int
        h.capattn_tile_sizes.argtypes = [cfgp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        h.capattn_fwd.restype = ctypes.c_int
        h.capattn_fwd.argtypes = [cfgp] + [vp] * 10 + [vp, sz, vp]
        h.capattn_bwd.restype = ctypes.c_int
        h.capattn_bwd.argtypes = [cfgp] + [vp] * 13 + [vp, sz, vp]
        h.capattn_bwd_dtemp.restype = ctypes.c_int
        h.capattn_bwd_dtemp.argtypes = [cfgp] + [vp] * 14 + [vp, sz, vp]
        h.capattn_bwd_ex.restype = ctypes.c_int
        h.capattn_bwd_ex.argtypes = [cfgp] + [vp] * 15 + [ctypes.c_uint32, vp, sz, vp]
        h.capattn_ranker_bounds_from_ids.restype = ctypes.c_int
        h.capattn_ranker_bounds_from_ids.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_int32, vp, vp, vp]
        h.capattn_device_status.restype = ctypes.c_int
        h.capattn_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        h.capattn_check_bounded_wait.restype = ctypes.c_int
        h.capattn_check_bounded_wait.argtypes = [vp, ctypes.c_uint64, vp]
        h.capattn_visit_map_host.restype = ctypes.c_int
        h.capattn_visit_map_host.argtypes = [cfgp, vp, vp, ctypes.c_int, vp, sz,
                                             ctypes.POINTER(sz)]
        h.capattn_visit_map_device.restype = ctypes.c_int
        h.capattn_visit_map_device.argtypes = [cfgp, vp, vp, ctypes.c_int, vp, sz, vp, sz, vp]
        h.capattn_mask_bits_host.restype = ctypes.c_int
        h.capattn_mask_bits_host.argtypes = [cfgp, vp, vp, i32, vp, sz]
        h.capattn_profile_enable.restype = ctypes.c_int
        h.capattn_profile_enable.argtypes = [ctypes.c_int]
        h.capattn_profile_select.restype = ctypes.c_int
        h.capattn_profile_select.argtypes = [ctypes.c_uint]
        h.capattn_profile_read.restype = ctypes.c_int
        h.capattn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int]
        h.capattn_kernel_name.restype = ctypes.c_char_p
        h.capattn_kernel_name.argtypes = [ctypes.c_int]
        _lib_handle = h
    return _lib_handle


EXPORTED_SYMBOLS = ("capattn_status_string", "capattn_validate_config", "capattn_workspace_bytes",
                    "capattn_tile_sizes", "capattn_fwd", "capattn_bwd", "capattn_bwd_dtemp", "capattn_bwd_ex",
                    "capattn_device_status", "capattn_ranker_bounds_from_ids",
                    "capattn_visit_map_host", "capattn_visit_map_device", "capattn_mask_bits_host",
                    "capattn_profile_enable", "capattn_profile_select", "capattn_profile_read", "capattn_kernel_name",
                    "capattn_fwd_noalloc", "capattn_noalloc_status", "capattn_check_bounded_wait",
                    "capattn_debug_alsc_poly")
KERNEL_KINDS = ("prepass", "fwd", "delta", "dkv", "dq")


@dataclass(frozen=True)
class AttnParams:
    """The method's parameters (the pages' KernelConfig fields)."""
    sm_scale: float
    cap_method: str = "none"
    cap: float = 0.0
    alpha: float = 0.0
    beta: float = 0.0
    causal: bool = False
    window_len: int = 0
    z_loss_weight: float = 0.0


def params_from_workload(w) -> AttnParams:
    return AttnParams(sm_scale=float(w.sm_scale), cap_method=w.cap_method, cap=float(w.cap),
                      alpha=float(w.alpha), beta=float(w.beta), causal=bool(w.causal),
                      window_len=int(w.window_len), z_loss_weight=float(w.z_loss_weight))


def make_config(ap: AttnParams, B: int, L: int, Hq: int, Hkv: int, D: int,
                dtype: torch.dtype, Lk: int = 0) -> CapattnConfig:
    """Lk: key / value length (0: equal to the query length L)."""
    if dtype not in DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    if ap.cap_method not in CAP_METHODS:
        raise ValueError(f"unknown cap method {ap.cap_method!r}")
    c = CapattnConfig()
    c.struct_size = ctypes.sizeof(CapattnConfig)
    c.cap_method = CAP_METHODS[ap.cap_method]
    c.cap, c.alpha, c.beta = ap.cap, ap.alpha, ap.beta
    c.sm_scale = ap.sm_scale
    c.causal = 1 if ap.causal else 0
    c.window_len = ap.window_len
    c.z_loss_weight = ap.z_loss_weight
    c.q_heads_per_kv_head = Hq // Hkv if Hkv > 0 else 0
    c.B, c.L, c.Hq, c.Hkv, c.D = B, L, Hq, Hkv, D
    c.dtype = DTYPES[dtype]
    c.Lk = Lk
    return c


def key_len(cfg: CapattnConfig) -> int:
    return cfg.Lk if cfg.Lk > 0 else cfg.L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise CapattnError(status, where)


def workspace_bytes(cfg: CapattnConfig, pass_: int) -> int:
    return int(lib().capattn_workspace_bytes(ctypes.byref(cfg), pass_))


def new_workspace(cfg: CapattnConfig, device) -> torch.Tensor:
    n = max(workspace_bytes(cfg, PASS_FWD), workspace_bytes(cfg, PASS_BWD))
    if n == 0:
        _check(lib().capattn_validate_config(ctypes.byref(cfg)), "capattn_workspace_bytes")
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _config(q, k, ap: AttnParams) -> CapattnConfig:
    """Config for q [B, L, Hq, D] and k [B, Lk, Hkv, D]."""
    B, L, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    return make_config(ap, B, L, Hq, Hkv, D, q.dtype, Lk=Lk)


def capattn_fwd(q, k, v, ap: AttnParams, temp=None, seg=None, bounds=None, workspace=None,
                want_ml=False, stream=None, out=None):
    """Forward.  q [B,L,Hq,D], k/v [B,Lk,Hkv,D] (bf16 or fp32, contiguous, on the GPU).
    Returns (o, lse, m, l); m and l are None unless want_ml.  out: optional
    preallocated (o, lse, m, l) to write into (m, l may be None)."""
    cfg = _config(q, k, ap)
    B, L, Hq = cfg.B, cfg.L, cfg.Hq
    if workspace is None:
        workspace = new_workspace(cfg, q.device)
    if out is not None:
        o, lse, m, l = out
    else:
        o = torch.empty_like(q)
        lse = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
        m = torch.empty_like(lse) if want_ml else None
        l = torch.empty_like(lse) if want_ml else None
    st = lib().capattn_fwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(temp), _ptr(seg),
                           _ptr(bounds), _ptr(o), _ptr(lse), _ptr(m), _ptr(l), _ptr(workspace),
                           workspace.numel(), _stream(stream))
    _check(st, "capattn_fwd")
    return o, lse, m, l


def capattn_bwd(q, k, v, o, lse, do, ap: AttnParams, temp=None, seg=None, bounds=None,
                workspace=None, stream=None, out=None):
    """Backward.  Returns (dq, dk, dv, delta).  out: optional preallocated
    (dq, dk, dv, delta) to write into."""
    cfg = _config(q, k, ap)
    B, L, Hq = cfg.B, cfg.L, cfg.Hq
    if workspace is None:
        workspace = new_workspace(cfg, q.device)
    if out is not None:
        dq, dk, dv, delta = out
    else:
        dq = torch.empty_like(q)
        dk = torch.empty_like(k)
        dv = torch.empty_like(v)
        delta = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
    st = lib().capattn_bwd(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(temp), _ptr(seg),
                           _ptr(bounds), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(delta), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check(st, "capattn_bwd")
    return dq, dk, dv, delta


def capattn_bwd_dtemp(q, k, v, o, lse, do, ap: AttnParams, temp, seg=None, bounds=None,
                      workspace=None, stream=None):
    """Backward with the temperature gradient.  Returns (dq, dk, dv, delta, dtemp [B,L])."""
    if temp is None:
        raise ValueError("capattn_bwd_dtemp needs the temperature tensor")
    cfg = _config(q, k, ap)
    B, L, Hq = cfg.B, cfg.L, cfg.Hq
    if workspace is None:
        workspace = new_workspace(cfg, q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    delta = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
    dtemp = torch.empty(B, L, dtype=torch.float32, device=q.device)
    st = lib().capattn_bwd_dtemp(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(temp), _ptr(seg),
                                 _ptr(bounds), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(delta), _ptr(dtemp), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(st, "capattn_bwd_dtemp")
    return dq, dk, dv, delta, dtemp


def capattn_bwd_ex(q, k, v, o, lse, do, ap: AttnParams, temp=None, seg=None, bounds=None, dlse=None,
                   want_dtemp=False, workspace=None, stream=None, reuse_fwd_maps=False):
    """Backward with an optional upstream LSE gradient dlse [B,Hq,L] (fp32) and,
    with want_dtemp, the temperature gradient.  Returns (dq, dk, dv, delta, dtemp).
    reuse_fwd_maps: use the spans and visit maps that capattn_fwd left in
    `workspace` for the same inputs instead of rebuilding them."""
    if want_dtemp and temp is None:
        raise ValueError("the temperature gradient needs the temperature tensor")
    if reuse_fwd_maps and workspace is None:
        raise ValueError("reusing the forward's maps needs the forward's workspace")
    cfg = _config(q, k, ap)
    B, L, Hq = cfg.B, cfg.L, cfg.Hq
    if workspace is None:
        workspace = new_workspace(cfg, q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    delta = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
    dtemp = torch.empty(B, L, dtype=torch.float32, device=q.device) if want_dtemp else None
    st = lib().capattn_bwd_ex(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(temp), _ptr(seg),
                              _ptr(bounds), _ptr(o), _ptr(lse), _ptr(do), _ptr(dlse), _ptr(dq),
                              _ptr(dk), _ptr(dv), _ptr(delta), _ptr(dtemp),
                              BWD_REUSE_FWD_MAPS if reuse_fwd_maps else 0, _ptr(workspace),
                              workspace.numel(), _stream(stream))
    _check(st, "capattn_bwd_ex")
    return dq, dk, dv, delta, dtemp


def ranker_bounds_from_ids(seg: torch.Tensor, history_id: int, candidate_id: int, workspace=None,
                           stream=None) -> torch.Tensor:
    """[B, L] int32 segment ids on the GPU -> [B, 4] int32 ranker bounds (hl, hu, cl, cu)."""
    B, L = seg.shape
    bounds = torch.empty(B, 4, dtype=torch.int32, device=seg.device)
    _check(lib().capattn_ranker_bounds_from_ids(_ptr(seg), B, L, int(history_id), int(candidate_id),
                                                _ptr(bounds), _ptr(workspace), _stream(stream)),
           "capattn_ranker_bounds_from_ids")
    return bounds


def capattn_device_status(workspace: torch.Tensor, stream=None) -> tuple[int, int]:
    """Synchronises the stream; returns (status, raw bits) and clears the word."""
    bits = ctypes.c_uint32(0)
    st = lib().capattn_device_status(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def capattn_check_bounded_wait(workspace: torch.Tensor, limit_ns: int, stream=None):
    """Runs the bounded-wait self-check (a wait that times out after limit_ns)."""
    _check(lib().capattn_check_bounded_wait(_ptr(workspace), int(limit_ns), _stream(stream)),
           "capattn_check_bounded_wait")


def capattn_tile_sizes(cfg: CapattnConfig):
    bq, bk = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().capattn_tile_sizes(ctypes.byref(cfg), ctypes.byref(bq), ctypes.byref(bk)),
           "capattn_tile_sizes")
    return bq.value, bk.value


def _np_ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def capattn_visit_map_host(cfg: CapattnConfig, seg=None, bounds=None, which=VISIT_Q_TILES):
    """Visit bitmap (numpy uint32) from host seg / bounds (numpy int32, C-contiguous)."""
    import numpy as np
    n = ctypes.c_size_t(0)
    _check(lib().capattn_visit_map_host(ctypes.byref(cfg), _np_ptr(seg), _np_ptr(bounds), which,
                                        None, 0, ctypes.byref(n)), "capattn_visit_map_host")
    out = np.zeros(n.value, dtype=np.uint32)
    _check(lib().capattn_visit_map_host(ctypes.byref(cfg), _np_ptr(seg), _np_ptr(bounds), which,
                                        _np_ptr(out), out.size, ctypes.byref(n)),
           "capattn_visit_map_host")
    return out


def capattn_visit_map_device(cfg: CapattnConfig, seg=None, bounds=None, which=VISIT_Q_TILES,
                             workspace=None, stream=None):
    """The same bitmap built by the device pre-pass (seg / bounds: device tensors)."""
    import numpy as np
    bq, bk = capattn_tile_sizes(cfg)
    nq, nk = -(-cfg.L // bq), -(-key_len(cfg) // bk)
    words = cfg.B * (nq * (-(-nk // 32)) if which == VISIT_Q_TILES else nk * (-(-nq // 32)))
    dev = torch.device("cuda")
    if workspace is None:
        workspace = new_workspace(cfg, dev)
    out = torch.zeros(words, dtype=torch.int32, device=dev)
    _check(lib().capattn_visit_map_device(ctypes.byref(cfg), _ptr(seg), _ptr(bounds), which,
                                          _ptr(out), words, _ptr(workspace), workspace.numel(),
                                          _stream(stream)), "capattn_visit_map_device")
    return out.cpu().numpy().view(np.uint32)


def capattn_mask_bits_host(cfg: CapattnConfig, b: int, seg=None, bounds=None):
    """Live-pair bit matrix of batch row b as a numpy bool array [L, Lk]."""
    import numpy as np
    Lk = key_len(cfg)
    wpr = -(-Lk // 64)
    bits = np.zeros(wpr * cfg.L, dtype=np.uint64)
    _check(lib().capattn_mask_bits_host(ctypes.byref(cfg), _np_ptr(seg), _np_ptr(bounds), b,
                                        _np_ptr(bits), bits.size), "capattn_mask_bits_host")
    by = bits.reshape(cfg.L, wpr).view(np.uint8)
    return np.unpackbits(by, axis=1, bitorder="little")[:, :Lk].astype(bool)


def capattn_profile_enable(on: bool = True):
    _check(lib().capattn_profile_enable(1 if on else 0), "capattn_profile_enable")


def capattn_profile_select(kinds=None):
    """Time only the given kernel kinds (names from KERNEL_KINDS; None = all)."""
    if kinds is None:
        mask = (1 << len(KERNEL_KINDS)) - 1
    else:
        mask = 0
        for k in kinds:
            mask |= 1 << KERNEL_KINDS.index(k)
    _check(lib().capattn_profile_select(mask), "capattn_profile_select")


def capattn_profile_read(reset: bool = True) -> dict:
    """{kernel kind: (milliseconds, launches)} since the last reset (synchronises)."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(lib().capattn_profile_read(ms, cnt, n, 1 if reset else 0), "capattn_profile_read")
    return {KERNEL_KINDS[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


class CapAttnFunction(torch.autograd.Function):
    """Autograd wrapper: forward saves (o, lse) and its workspace, whose spans
    and visit maps the backward (capattn_bwd_ex) reuses.  Gradients flow to q,
    k, v and, when it requires grad, to the temperature; a loss that uses the
    returned lse contributes through its gradient dlse (d lse_i / d t_ij =
    P_ij).  Segment ids and bounds are inputs only."""

    @staticmethod
    def forward(ctx, q, k, v, ap: AttnParams, temp=None, seg=None, bounds=None):
        ws = new_workspace(_config(q, k, ap), q.device)
        o, lse, _, _ = capattn_fwd(q, k, v, ap, temp, seg, bounds, workspace=ws)
        ctx.save_for_backward(q, k, v, o, lse, temp, seg, bounds)
        ctx.ws = ws
        ctx.ap = ap
        ctx.set_materialize_grads(False)
        return o, lse

    @staticmethod
    def backward(ctx, do, dlse):
        q, k, v, o, lse, temp, seg, bounds = ctx.saved_tensors
        want_dtemp = temp is not None and ctx.needs_input_grad[4]
        do = torch.zeros_like(o) if do is None else do.contiguous()
        if dlse is not None:
            dlse = dlse.to(torch.float32).contiguous()
        dq, dk, dv, _, dtemp = capattn_bwd_ex(q, k, v, o, lse, do, ctx.ap, temp, seg, bounds,
                                              dlse=dlse, want_dtemp=want_dtemp, workspace=ctx.ws,
                                              reuse_fwd_maps=True)
        return dq, dk, dv, None, dtemp, None, None


def attention(q, k, v, ap: AttnParams, temp=None, seg=None, bounds=None):
    """Soft-capped attention output O (differentiable in q, k, v)."""
    o, _ = CapAttnFunction.apply(q, k, v, ap, temp, seg, bounds)
    return o
