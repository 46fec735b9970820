"""The boundary is a C ABI: a plain C99 program (tests/c_abi_client.c), built
with gcc against include/capattn.h and linked to libcapattn.so, calls the
library's host-side entry points with no Python or C++ in between.  Its
live-pair and visited-tile counts are checked against the oracle and its
sizes against the same calls made through the Python binding."""

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if shutil.which("gcc") is None or not os.path.isdir(CUDA_INCLUDE):
        pytest.skip("gcc or the CUDA headers are not available")
    if not os.path.exists(ca.LIB_PATH):
        from soft_capped_attention_gb300 import build
        build.build()
    libdir = os.path.dirname(ca.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_abi") / "client")
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           os.path.join(ROOT, "tests", "c_abi_client.c"), "-I", os.path.join(ROOT, "include"),
           "-I", CUDA_INCLUDE, "-L", libdir, "-lcapattn", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _run(exe, L, window, hist, cand):
    r = subprocess.run([exe, str(L), str(window), "%d,%d" % hist, "%d,%d" % cand],
                       capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    first, name = r.stdout.splitlines()[:2]
    return dict(kv.split("=", 1) for kv in first.split()), name


@pytest.mark.parametrize("L,window,hist,cand", [
    (300, 0, (0, 300), (300, 300)),      # history covers the row: plain causal
    (300, 37, (0, 200), (200, 260)),
    (1000, 129, (0, 700), (700, 777)),
    (129, 1, (5, 60), (60, 129)),
])
def test_c_client_matches_oracle(client, L, window, hist, cand):
    out, name = _run(client, L, window, hist, cand)
    assert out["ok"] == "0" and out["bad"] == "1" and out["d96"] == "2"
    assert out["ws_null"] == "5"  # CAPATTN_ERR_WORKSPACE, returned before any launch
    lib = ca.lib()
    assert name == lib.capattn_status_string(5).decode() and name

    bounds = np.array([hist + cand], np.int32)
    ocfg = orc.OracleConfig(sm_scale=1.0, causal=True, window_len=window)
    assert int(out["live"]) == orc.pair_count(L, ocfg, None, bounds, B=1)
    bq, bk = int(out["bq"]), int(out["bk"])
    assert int(out["visited"]) == int(orc.visit_matrix(L, bq, bk, ocfg, None, bounds[0]).sum())

    # the same sizes through the Python binding's ctypes calls
    ap = ca.AttnParams(sm_scale=0.125, cap_method="tanh", cap=50.0, causal=True, window_len=window)
    cfg = ca.make_config(ap, 1, L, 4, 2, 128, torch.bfloat16)
    assert int(out["ws_fwd"]) == lib.capattn_workspace_bytes(ctypes.byref(cfg), 0)
    assert int(out["ws_bwd"]) == lib.capattn_workspace_bytes(ctypes.byref(cfg), 1)
    assert (bq, bk) == ca.capattn_tile_sizes(cfg)
