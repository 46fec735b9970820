"""CPU tests of the seeded input generators that both the oracle and the CUDA
path take their inputs from: bf16 rounding agrees with PyTorch's conversion,
draws are reproducible, and shapes, masks and ranges follow the stated recipe."""

import numpy as np
import pytest
import torch

from soft_capped_attention_gb300.workloads import (WORKLOADS, make_aux, make_tensors,
                                                   packed_segments, ranker_bounds, round_to_bf16)


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 100000),
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, np.inf, -np.inf],
                                 np.float32)]).astype(np.float32)
    ours = round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)
    # ties go to even: 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7
    assert round_to_bf16(np.array([1.0 + 2.0 ** -8], np.float32))[0] == 1.0
    assert round_to_bf16(np.array([1.0 + 3 * 2.0 ** -8], np.float32))[0] == 1.0 + 2.0 ** -6


@pytest.mark.parametrize("idx", sorted(WORKLOADS))
def test_shapes_and_reproducibility(idx):
    w = WORKLOADS[idx]
    small = w.replace(B=min(w.B, 2), L=min(w.L, 300), Lk=None if w.Lk is None else min(w.Lk, 500))
    a, b = make_tensors(small, seed=idx), make_tensors(small, seed=idx)
    Lk = small.key_len
    assert a["q"].shape == (small.B, small.L, small.Hq, small.D)
    assert a["k"].shape == a["v"].shape == (small.B, Lk, small.Hkv, small.D)
    assert a["do"].shape == a["q"].shape
    for n in a:
        np.testing.assert_array_equal(a[n], b[n])
        assert a[n].dtype == np.float32
        if w.dtype == "bf16":
            np.testing.assert_array_equal(a[n], round_to_bf16(a[n]))
    aux = make_aux(small, seed=idx)
    assert (aux["temp"] is None) == (w.temp_range is None)
    assert (aux["seg"] is None) == (w.doc_len_range is None)
    assert (aux["bounds"] is None) == (w.ranker_hu_range is None)
    if aux["temp"] is not None:
        lo, hi = w.temp_range
        assert aux["temp"].shape == (small.B, small.L)
        assert aux["temp"].min() >= lo and aux["temp"].max() < hi


def test_packed_segments_recipe():
    rng = np.random.default_rng(4)
    seg = packed_segments(rng, 3, 5000, 128, 2048)
    for row in seg:
        assert row[0] == 0 and np.all(np.diff(row) >= 0) and np.all(np.diff(row) <= 1)
        ids, counts = np.unique(row, return_counts=True)
        assert np.array_equal(ids, np.arange(ids.size))
        assert np.all(counts[:-1] >= 128) and np.all(counts <= 2048)  # last document may be cut
        assert counts.sum() == 5000


def test_ranker_bounds_recipe():
    rng = np.random.default_rng(5)
    bd = ranker_bounds(rng, 200, 4096, (1024, 3968), (16, 128))
    hl, hu, cl, cu = bd.T
    assert np.all(hl == 0) and np.all(cl == hu)
    assert np.all((hu >= 1024) & (hu <= 3968))
    assert np.all(cu <= 4096) and np.all(cu - cl >= 16) and np.all(cu - cl <= 128)
