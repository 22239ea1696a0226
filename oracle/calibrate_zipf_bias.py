"""Find the Zipf-bias strength gamma of the skewed DeepSeek-V3-shaped batch.

The skewed workload adds b_e = -gamma * 1.2 * ln(r_e) to the router logits
(r = a seeded rank permutation; the four coldest ranks get -30).  This script
routes a sample of the workload's tokens with the oracle (fp64 logits, top-8)
and bisects gamma until the hottest expert receives 10x the mean row count.
The result is stored as workload.configs.ZIPF_GAMMA.

    python -m oracle.calibrate_zipf_bias [--tokens 4096]
"""
import argparse

import numpy as np

import workload as wl
from oracle import moe


def hot_ratio(base_logits, cfg, gamma):
    b = wl.gen_bias(cfg, gamma).double().numpy()
    ids = moe.select_topk(base_logits + b[None, :], cfg.k)
    counts, _ = moe.expert_histogram(ids, cfg.E)
    return counts.max() / counts.mean(), int((counts == 0).sum())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=4096)
    a = ap.parse_args()
    cfg = wl.DSV3_SKEW
    x = wl.gen_x(cfg, rows=a.tokens)
    lg = moe.router_logits(x, wl.gen_router(cfg))
    lo, hi = 0.0, 2.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        r, _ = hot_ratio(lg, cfg, mid)
        lo, hi = (mid, hi) if r < 10.0 else (lo, mid)
    g = round(0.5 * (lo + hi), 4)
    r, dead = hot_ratio(lg, cfg, g)
    print(f"ZIPF_GAMMA = {g}   (hottest/mean = {r:.2f}, experts with no rows = {dead}, "
          f"sample = {a.tokens} tokens)")


if __name__ == "__main__":
    main()
