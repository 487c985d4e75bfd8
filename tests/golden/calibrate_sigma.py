"""Measures alpha = E[sum_v min(p_v, q_v)] of the synthetic workloads with the
oracle's softmax and bisects the draft-noise sigma to the target alpha.
Prints one line per configuration; the sigma values it finds are the ones
written in speculative_decoding_verification_vocab_gb300/synth.py.

    python tests/golden/calibrate_sigma.py
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402
from speculative_decoding_verification_vocab_gb300 import synth  # noqa: E402


def measured_alpha(cfg, sigma, rows=24):
    c = synth.Config(**{**cfg.__dict__, "sigma_noise": sigma})
    vq, dp, _ = synth.chain_inputs(c, seed=123, B=rows // 4 if rows >= 4 else 1, N=4)
    a = []
    for b in range(vq.shape[0]):
        for i in range(4):
            q = oracle.softmax(vq[b, i].float().numpy())
            p = oracle.softmax(dp[b, i].float().numpy())
            a.append(np.minimum(p, q).sum())
    return float(np.mean(a))


def main():
    for idx in (2, 3, 4, 5):
        cfg = synth.CONFIGS[idx]
        lo, hi = 0.05, 2.0
        for _ in range(14):
            mid = 0.5 * (lo + hi)
            if measured_alpha(cfg, mid) > cfg.target_alpha:
                lo = mid
            else:
                hi = mid
        print(f"config {idx} {cfg.name}: target alpha {cfg.target_alpha} -> sigma {mid:.3f} "
              f"(alpha at synth value {cfg.sigma_noise}: {measured_alpha(cfg, cfg.sigma_noise):.3f})")
    c1 = synth.CONFIGS[1]
    print(f"config 1 {c1.name}: sigma {c1.sigma_noise} (fixed) alpha {measured_alpha(c1, c1.sigma_noise):.3f}")


if __name__ == "__main__":
    torch.manual_seed(0)
    main()
