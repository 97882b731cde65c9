"""Writes the per-expert router logit bias of the skewed-load workload.

TEST INFRASTRUCTURE: runs the CPU oracle's router only. Usage:

    python -m oracle.calibrate_skew_bias

Workload: T=32768, d=2048, E=128, K=8, seed 0 (x, W_g from the seeded input
generator). Target: expert loads follow a Zipf law with exponent s = 1.2 over
124 experts, capped at T (a token can pick an expert only once, so the largest
loads cannot exceed T); the remaining 4 experts get a bias of -1e4 and receive
no tokens. The bias is found by the fixed-point iteration
bias_e += log(target_e / observed_e) on the oracle router's selection.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import moe_oracle as O

T, D, E, K = 32768, 2048, 128, 8
N_ACTIVE = 124
ZIPF_S = 1.2


def zipf_targets(total: int, n: int, cap: int, s: float) -> np.ndarray:
    r = np.arange(1, n + 1, dtype=np.float64) ** (-s)
    lo, hi = 0.0, float(total)
    for _ in range(200):                       # bisection on the scale c
        c = 0.5 * (lo + hi)
        if np.minimum(cap, c * r).sum() > total:
            hi = c
        else:
            lo = c
    return np.minimum(cap, lo * r)


def main():
    import torch  # noqa: F401  (the input generator is torch-based)
    from token_dispatch_grouped_gb300 import inputs as I

    s = I.WORKLOADS["skew"]
    assert (s.T, s.d, s.E, s.K) == (T, D, E, K)
    inp = I.make_layer_inputs(s, seed=0, parts=("x", "Wg"))
    z, _, _, _ = O.route(inp["x"], inp["Wg"], K)        # logits without bias
    ident = np.eye(E)
    target = zipf_targets(T * K, N_ACTIVE, T, ZIPF_S)
    bias = np.zeros(E)
    bias[N_ACTIVE:] = -1e4
    for it in range(400):
        _, _, ids, _ = O.route(z, ident, K, bias)      # selection on z + bias
        load = np.bincount(ids.reshape(-1), minlength=E).astype(np.float64)
        ratio = np.log(np.maximum(target, 0.5) / np.maximum(load[:N_ACTIVE], 0.5))
        bias[:N_ACTIVE] += 0.7 * np.clip(ratio, -2.0, 2.0)
        bias[:N_ACTIVE] -= bias[:N_ACTIVE].mean()
        err = np.abs(load[:N_ACTIVE] - target).sum() / (T * K)
        if err < 0.01:
            break
    _, _, ids, _ = O.route(z, ident, K, bias)
    load = np.bincount(ids.reshape(-1), minlength=E)
    nz = load[:N_ACTIVE] > 0
    ranks = np.arange(1, N_ACTIVE + 1)[nz]
    slope = -np.polyfit(np.log(ranks), np.log(load[:N_ACTIVE][nz]), 1)[0]
    out = dict(
        E=E, T=T, d=D, K=K, seed=0, zipf_s=ZIPF_S, active_experts=N_ACTIVE,
        iterations=it + 1, l1_error=float(err), fitted_slope=float(slope),
        empty_experts=int((load == 0).sum()), loads=load.tolist(),
        bias=[float(b) for b in bias],
        written_by="python -m oracle.calibrate_skew_bias",
    )
    path = I.SKEW_BIAS_FILE
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(f"wrote {path}: slope {slope:.3f}, empty {out['empty_experts']}, "
          f"max load {load.max()}, l1 err {err:.4f}, iters {it + 1}")


if __name__ == "__main__":
    main()
