"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same (bf16-rounded) inputs, compare with the
stated tolerances."""

import numpy as np
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca

# Match criteria: fp32 inputs 1e-4 max-abs for O and the gradients; bf16 inputs
# O 2e-2 max-abs, LSE 1e-3 max-abs on live rows (-inf identical), gradients
# 2e-2 relative Frobenius error against the oracle on the same bf16 inputs.
TOL_FP32 = 1e-4
TOL_BF16_O = 2e-2
TOL_BF16_LSE = 1e-3
TOL_BF16_GRAD = 2e-2


def to_dev(x, dtype=None):
    if x is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


# Guard bands (a stand-in for a memory checker): every output buffer sits
# between two 4 KB bands of a sentinel byte, and one band follows the
# workspace; a write outside a buffer shows up as a changed band.
GUARD_BYTES = 4096
GUARD_BYTE = 0xA5


class Guarded:
    """A tensor of the given shape and dtype inside a byte buffer with guard bands."""

    def __init__(self, shape, dtype, device="cuda"):
        esz = torch.tensor([], dtype=dtype).element_size()
        n = int(np.prod(shape)) * esz
        self.buf = torch.full((GUARD_BYTES + n + GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8,
                              device=device)
        self.n = n
        self.tensor = self.buf[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)

    def intact(self) -> bool:
        head = self.buf[:GUARD_BYTES]
        tail = self.buf[GUARD_BYTES + self.n:]
        return bool((head == GUARD_BYTE).all()) and bool((tail == GUARD_BYTE).all())


def run_gpu(inp, ap, dtype, want_ml=False, pool=True):
    """Forward and backward through the binding with every output guarded; the
    inputs must come back unchanged and no guard band may be touched.  pool:
    a workspace that holds the dX pool (bf16: the stored-dX backward, checked
    by its launch of the delta kernel) or one without it (the backward that
    recomputes dX for dQ)."""
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("q", "k", "v", "do"))
    temp, seg, bounds = to_dev(inp.get("temp")), to_dev(inp.get("seg")), to_dev(inp.get("bounds"))
    inputs = [t for t in (q, k, v, do, temp, seg, bounds) if t is not None]
    before = [t.clone() for t in inputs]
    B, L, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    cfg = ca.make_config(ap, B, L, Hq, Hkv, D, dtype, Lk=Lk)
    ws_bytes = max(ca.workspace_bytes(cfg, ca.PASS_FWD),
                   ca.workspace_bytes(cfg, ca.PASS_BWD if pool else ca.PASS_BWD_NO_POOL))
    ws_g = Guarded((ws_bytes,), torch.uint8)
    ws_g.tensor.zero_()
    assert ws_g.tensor.data_ptr() % 256 == 0
    g = {"O": Guarded((B, L, Hq, D), dtype), "LSE": Guarded((B, Hq, L), torch.float32),
         "m": Guarded((B, Hq, L), torch.float32) if want_ml else None,
         "l": Guarded((B, Hq, L), torch.float32) if want_ml else None,
         "dQ": Guarded((B, L, Hq, D), dtype), "dK": Guarded((B, Lk, Hkv, D), dtype),
         "dV": Guarded((B, Lk, Hkv, D), dtype), "delta": Guarded((B, Hq, L), torch.float32)}
    t = {n: (None if x is None else x.tensor) for n, x in g.items()}
    o, lse, m, l = ca.capattn_fwd(q, k, v, ap, temp, seg, bounds, workspace=ws_g.tensor,
                                  out=(t["O"], t["LSE"], t["m"], t["l"]))
    ca.capattn_profile_enable(True)
    ca.capattn_profile_select([])  # launch counts only
    ca.capattn_profile_read(reset=True)
    dq, dk, dv, delta = ca.capattn_bwd(q, k, v, o, lse, do, ap, temp, seg, bounds, workspace=ws_g.tensor,
                                       out=(t["dQ"], t["dK"], t["dV"], t["delta"]))
    launches = ca.capattn_profile_read(reset=True)
    ca.capattn_profile_enable(False)
    if dtype == torch.bfloat16:
        stored_dx = ca.workspace_bytes(cfg, ca.PASS_BWD) > ca.workspace_bytes(cfg, ca.PASS_BWD_NO_POOL)
        assert launches["delta"][1] == (1 if (pool and stored_dx) else 0), launches
    st, bits = ca.capattn_device_status(ws_g.tensor)
    assert st == 0, f"device status {st} bits {bits}"
    torch.cuda.synchronize()
    for name, x in list(g.items()) + [("workspace", ws_g)]:
        assert x is None or x.intact(), f"guard band of {name} overwritten"
    for a, b in zip(inputs, before):
        assert torch.equal(a, b), "an input was modified"
    out = {"O": o, "LSE": lse, "dQ": dq, "dK": dk, "dV": dv, "delta": delta, "m": m, "l": l}
    return {k2: (None if v2 is None else v2.float().cpu().numpy()) for k2, v2 in out.items()}


def oracle_cfg(ap):
    return orc.OracleConfig(sm_scale=ap.sm_scale, cap_method=ap.cap_method, cap=ap.cap,
                            alpha=ap.alpha, beta=ap.beta, causal=ap.causal,
                            window_len=ap.window_len, z_loss_weight=ap.z_loss_weight)


def run_oracle(inp, ap):
    cfg = oracle_cfg(ap)
    O, LSE, M, Lsum = orc.forward(inp["q"], inp["k"], inp["v"], inp.get("temp"), inp.get("seg"),
                                  inp.get("bounds"), cfg)
    dQ, dK, dV, delta = orc.backward(inp["q"], inp["k"], inp["v"], inp.get("temp"), inp.get("seg"),
                                     inp.get("bounds"), O, LSE, inp["do"], cfg)
    return {"O": O, "LSE": LSE, "dQ": dQ, "dK": dK, "dV": dV, "delta": delta, "m": M, "l": Lsum}


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def check_lse(got, ref, tol):
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "fully masked rows differ"
    fin = np.isfinite(ref)
    if fin.any():
        err = float(np.max(np.abs(got[fin] - ref[fin])))
        assert err <= tol, f"LSE max-abs {err}"


def compare(got, ref, dtype):
    report = {}
    if dtype == torch.float32:
        for name in ("O", "dQ", "dK", "dV"):
            err = float(np.max(np.abs(got[name] - ref[name]))) if got[name].size else 0.0
            report[name] = err
            assert err <= TOL_FP32, f"{name} max-abs {err}"
        check_lse(got["LSE"], ref["LSE"], TOL_FP32)
    else:
        err = float(np.max(np.abs(got["O"] - ref["O"]))) if got["O"].size else 0.0
        report["O"] = err
        assert err <= TOL_BF16_O, f"O max-abs {err}"
        check_lse(got["LSE"], ref["LSE"], TOL_BF16_LSE)
        for name in ("dQ", "dK", "dV"):
            e = rel_fro(got[name], ref[name])
            report[name] = e
            assert e <= TOL_BF16_GRAD, f"{name} rel-Frobenius {e}"
    return report
