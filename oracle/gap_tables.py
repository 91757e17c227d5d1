"""Routing-score gap enforcement for the seeded workloads -- TEST INFRASTRUCTURE.

A token whose k-th and (k+1)-th selection scores (sigmoid(logit) + bias, on the
fp32 logits) differ by less than the workload's gap (1e-3) has its row of x
re-drawn with the next attempt counter of the generator's stream, up to 64
times.  With the gap, the order in which a split-K reduction sums a logit
cannot change which experts are picked (kda page: split-K reductions differ
only in their order).

Run as a script to (re)write ``moe_inputs/gap_attempts.json`` for seed 0 of
every workload; it calls only the oracle and the input generator.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import moe_inputs as mi  # noqa: E402
from oracle.moe_oracle import router_logits, score_gap  # noqa: E402

MAX_ATTEMPTS = 64


def enforce_gap(cfg: mi.MoEConfig, seed: int = 0) -> np.ndarray:
    """Per-row attempt counters such that every token's score gap >= cfg.gap."""
    w_gate = mi.gen_w_gate(cfg, seed)
    bias = mi.gen_bias(cfg, seed)
    off = mi.gen_logit_offset(cfg, seed)
    att = np.zeros(cfg.S, np.int64)
    x = mi.gen_x(cfg, seed, att)
    bad = np.nonzero(score_gap(router_logits(x, w_gate, off), bias, cfg.k) < cfg.gap)[0]
    while len(bad):
        att[bad] += 1
        if att.max() > MAX_ATTEMPTS:
            raise RuntimeError(f"{cfg.name}: gap {cfg.gap} not reached in {MAX_ATTEMPTS} draws")
        xb = np.stack([mi.gen_x_rows(cfg, seed, np.array([t]), int(att[t]))[0] for t in bad])
        gap = score_gap(router_logits(xb, w_gate, off), bias, cfg.k)
        bad = bad[gap < cfg.gap]
    return att


def main() -> None:
    path = os.path.join(os.path.dirname(os.path.abspath(mi.__file__)), "gap_attempts.json")
    tab = {}
    for cfg in list(mi.CONFIGS) + [lc.router() for lc in mi.LATENT_CONFIGS]:
        att = enforce_gap(cfg, 0)
        rows = np.nonzero(att)[0]
        tab[f"{cfg.name}/seed0"] = {
            "shape": [cfg.S, cfg.d, cfg.E, cfg.k],
            "rows": [int(r) for r in rows],
            "attempts": [int(att[r]) for r in rows],
        }
        print(f"{cfg.name}: {len(rows)} of {cfg.S} rows re-drawn, max attempt {att.max()}")
    with open(path, "w") as f:
        json.dump(tab, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
