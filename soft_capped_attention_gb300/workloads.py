"""Seeded synthetic workloads for soft-capped attention.

This module only draws random inputs and describes workload shapes.  It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it without sharing any of the method's code.

Five workloads are defined, all synthetic (no dataset is involved):

1. ``tiny_fp32``: B=1, Hq=Hkv=2, L=128, D=64, fp32, no cap, non-causal.
2. ``causal_tanh``: B=2, Hq=Hkv=16, L=2048, D=128, bf16, causal, tanh cap 50.
3. ``gqa_window_alsc``: B=4, Hq=32, Hkv=8, L=4096, D=128, bf16, causal and a
   1024-key sliding window, ALSC cap (30, 2, 0.5), per-query temperature
   drawn from U[0.5, 1.5], z-loss weight 1e-4.
4. ``packed_softsign``: B=8, L=8192, Hq=Hkv=16, D=128, bf16, packed documents
   with lengths drawn from U[128, 2048] (last one truncated) as int32 segment
   ids, causal plus segment equality, soft-sign cap 20.
5. ``ranker_alsc``: B=32, Hq=8, Hkv=2, L=4096, D=128, bf16, history/candidate
   ranker bounds with hl=0, hu ~ U[1024, 3968], cl=hu,
   cu=min(hu + U[16, 128], L); ALSC cap (30, 2, 0.5).
6. ``cross_tanh``: cross attention with unequal lengths, B=2, Hq=Hkv=16,
   L=2048 queries against Lk=8192 keys, D=128, bf16, no mask, tanh cap 50.

Random streams (a stated choice; the pages fix no generator):

* Q, K, V and dO come, in that order, from ``numpy.random.PCG64(seed)`` as
  float32 standard normals.  For bf16 workloads they are rounded to bf16 with
  round-to-nearest-even and returned as float32 arrays that hold bf16 values
  exactly, so every consumer sees identical numbers.
* temperature, segment ids and ranker bounds come from a second stream,
  ``numpy.random.PCG64([seed, 1])``, so they can be drawn without the large
  tensors.  Integer draws are inclusive at both ends.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

CAP_METHODS = ("none", "tanh", "soft_sign", "alsc")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    dtype: str  # "fp32" or "bf16"
    sm_scale: float
    causal: bool = False
    window_len: int = 0
    cap_method: str = "none"
    cap: float = 0.0
    alpha: float = 0.0
    beta: float = 0.0
    temp_range: tuple | None = None  # None: temperature 1 (no array)
    doc_len_range: tuple | None = None  # None: one segment (no array)
    ranker_hu_range: tuple | None = None  # None: no ranker bounds
    ranker_cand_range: tuple | None = None
    z_loss_weight: float = 0.0
    Lk: int | None = None  # key / value length; None: equal to L

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def key_len(self) -> int:
        return self.L if self.Lk is None else self.Lk

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    1: Workload("tiny_fp32", B=1, L=128, Hq=2, Hkv=2, D=64, dtype="fp32",
                sm_scale=1.0 / 8.0),
    2: Workload("causal_tanh", B=2, L=2048, Hq=16, Hkv=16, D=128, dtype="bf16",
                sm_scale=1.0 / np.sqrt(128.0), causal=True,
                cap_method="tanh", cap=50.0),
    3: Workload("gqa_window_alsc", B=4, L=4096, Hq=32, Hkv=8, D=128,
                dtype="bf16", sm_scale=1.0 / np.sqrt(128.0), causal=True,
                window_len=1024, cap_method="alsc", cap=30.0, alpha=2.0,
                beta=0.5, temp_range=(0.5, 1.5), z_loss_weight=1e-4),
    4: Workload("packed_softsign", B=8, L=8192, Hq=16, Hkv=16, D=128,
                dtype="bf16", sm_scale=1.0 / np.sqrt(128.0), causal=True,
                cap_method="soft_sign", cap=20.0, doc_len_range=(128, 2048)),
    5: Workload("ranker_alsc", B=32, L=4096, Hq=8, Hkv=2, D=128, dtype="bf16",
                sm_scale=1.0 / np.sqrt(128.0), cap_method="alsc", cap=30.0,
                alpha=2.0, beta=0.5, ranker_hu_range=(1024, 3968),
                ranker_cand_range=(16, 128)),
    6: Workload("cross_tanh", B=2, L=2048, Lk=8192, Hq=16, Hkv=16, D=128, dtype="bf16",
                sm_scale=1.0 / np.sqrt(128.0), cap_method="tanh", cap=50.0),
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), kept as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def packed_segments(rng: np.random.Generator, B: int, L: int, lo: int, hi: int) -> np.ndarray:
    """Per batch row: document lengths ~ U[lo, hi] appended until they cover L,
    the last one cut to fit; ids 0, 1, 2, ... per row (non-decreasing)."""
    seg = np.empty((B, L), dtype=np.int32)
    for b in range(B):
        pos, doc = 0, 0
        while pos < L:
            n = int(rng.integers(lo, hi + 1))
            n = min(n, L - pos)
            seg[b, pos:pos + n] = doc
            pos += n
            doc += 1
    return seg


def ranker_bounds(rng: np.random.Generator, B: int, L: int, hu_range, cand_range) -> np.ndarray:
    """Per batch row (hl, hu, cl, cu) = (0, hu, hu, min(hu + extra, L))."""
    out = np.empty((B, 4), dtype=np.int32)
    for b in range(B):
        hu = int(rng.integers(hu_range[0], hu_range[1] + 1))
        extra = int(rng.integers(cand_range[0], cand_range[1] + 1))
        out[b] = (0, hu, hu, min(hu + extra, L))
    return out


def make_aux(w: Workload, seed: int) -> dict:
    """temperature [B, L] float32, segment ids [B, L] int32 and bounds [B, 4]
    int32 (each None when the workload does not use it)."""
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    temp = seg = bounds = None
    if w.temp_range is not None:
        temp = rng.uniform(w.temp_range[0], w.temp_range[1], size=(w.B, w.L)).astype(np.float32)
    if w.doc_len_range is not None:
        seg = packed_segments(rng, w.B, w.L, *w.doc_len_range)
    if w.ranker_hu_range is not None:
        bounds = ranker_bounds(rng, w.B, w.L, w.ranker_hu_range, w.ranker_cand_range)
    return {"temp": temp, "seg": seg, "bounds": bounds}


def make_tensors(w: Workload, seed: int) -> dict:
    """Q [B,L,Hq,D], K and V [B,Lk,Hkv,D], dO [B,L,Hq,D] as float32 arrays
    (bf16-exact for bf16 workloads)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    Lk = w.key_len
    shapes = {"q": (w.B, w.L, w.Hq, w.D), "k": (w.B, Lk, w.Hkv, w.D),
              "v": (w.B, Lk, w.Hkv, w.D), "do": (w.B, w.L, w.Hq, w.D)}
    out = {}
    for name in ("q", "k", "v", "do"):
        x = rng.standard_normal(size=shapes[name], dtype=np.float32)
        if w.dtype == "bf16":
            x = round_to_bf16(x)
        out[name] = x
    return out


def make_inputs(w: Workload, seed: int) -> dict:
    d = make_tensors(w, seed)
    d.update(make_aux(w, seed))
    return d


def small_variant(w: Workload, **kw) -> Workload:
    """The same feature set at a smaller shape (for parity tests)."""
    return w.replace(**kw)
