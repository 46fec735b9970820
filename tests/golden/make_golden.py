"""Writes the stored expected values under tests/golden/ from the oracle alone.

    python tests/golden/make_golden.py

pair_counts.json: for each seeded workload, the exact number of
unmasked (query, key) pairs summed over batch and query heads (the N in the
mask-aware FLOP counts 4*D*N forward, 10*D*N backward), counted by the oracle's
brute-force mask from the seeded segment ids / ranker bounds.  Only the
oracle and the seeded input generators are used.
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from oracle import capattn_oracle as orc  # noqa: E402
from soft_capped_attention_gb300.workloads import WORKLOADS, make_aux  # noqa: E402


def main():
    out = {}
    for idx, w in WORKLOADS.items():
        aux = make_aux(w, seed=idx)
        cfg = orc.config_from_workload(w)
        per_head = orc.pair_count(w.L, cfg, aux["seg"], aux["bounds"], B=w.B, Lk=w.key_len)
        out[str(idx)] = {"name": w.name, "seed": idx, "pairs": per_head * w.Hq,
                         "pairs_per_head_summed_over_batch": per_head}
        print(idx, w.name, per_head * w.Hq)
    with open(os.path.join(HERE, "pair_counts.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
