"""GPU: the device pre-pass builds visit maps bit-exact with the oracle's brute force."""

import numpy as np
import pytest
import torch

from oracle import capattn_oracle as orc
from soft_capped_attention_gb300 import capattn as ca
from soft_capped_attention_gb300.workloads import WORKLOADS, make_aux

from parity_utils import to_dev
from test_boundary import CASES, _aux, _cfg, _oracle_cfg, oracle_visit_words

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("L,dtype", [(300, torch.bfloat16), (4100, torch.bfloat16),
                                     (200, torch.float32)])
def test_device_visit_maps_match_oracle(case, L, dtype):
    cs = CASES[case]
    rng = np.random.default_rng(case + 11 * L)
    B = 3
    seg, bounds = _aux(cs, B, L, rng)
    D = 128 if dtype == torch.bfloat16 else 64
    c = _cfg(B=B, L=L, D=D, dtype=dtype, causal=cs["causal"], window_len=cs["window_len"])
    bq, bk = ca.capattn_tile_sizes(c)
    ocfg = _oracle_cfg(cs["causal"], cs["window_len"])
    for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
        got = ca.capattn_visit_map_device(c, to_dev(seg), to_dev(bounds), which)
        ref = oracle_visit_words(B, L, bq, bk, ocfg, seg, bounds, which)
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_device_visit_maps_of_the_workloads(idx):
    w = WORKLOADS[idx]
    aux = make_aux(w, seed=idx)
    c = ca.make_config(ca.params_from_workload(w), w.B, w.L, w.Hq, w.Hkv, w.D, torch.bfloat16)
    bq, bk = ca.capattn_tile_sizes(c)
    ocfg = orc.config_from_workload(w)
    for which in (ca.VISIT_Q_TILES, ca.VISIT_KV_TILES):
        got = ca.capattn_visit_map_device(c, to_dev(aux["seg"]), to_dev(aux["bounds"]), which)
        ref = oracle_visit_words(w.B, w.L, bq, bk, ocfg, aux["seg"], aux["bounds"], which)
        assert np.array_equal(got, ref)
