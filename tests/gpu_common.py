"""Helpers shared by the GPU parity tests (no arithmetic of the layer here)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: indices bit-exact; fp32 router logits / weights within relative
# Frobenius 1e-5; bf16 outputs and gradients within relative Frobenius 1e-2 of
# the fp64 oracle.
TOL_ROUTER = 1e-5
TOL_BF16 = 1e-2
GAP = 1e-3      # router ids are compared where the deciding logit gap exceeds this
TOL_ROW = 3e-2  # per-row bound beside the whole-tensor Frobenius check


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def cpu(t) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.numpy()


def to_dev(d: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def rel_rows(a, b) -> float:
    """Largest relative error of one row (last axis) of a against b: a wrong
    tile cannot hide inside a whole-tensor norm. Rows whose reference norm is
    below half the median row norm are measured against that floor: such
    rows can be legitimately inexact relative to themselves (a weight-gradient
    row of one token near the zero of SiLU', computed from the bf16-stored
    pre-activation), while a wrong tile errs by the size of a typical row."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    a = a.reshape(-1, a.shape[-1])
    b = b.reshape(-1, b.shape[-1])
    nb = np.linalg.norm(b, axis=1)
    if nb.size == 0:
        return 0.0
    floor = max(0.5 * float(np.median(nb)), 1e-30)
    return float(np.max(np.linalg.norm(a - b, axis=1) / np.maximum(nb, floor)))
