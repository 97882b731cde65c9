"""Numerical facts the CUDA path relies on, checked on the CPU.

The tensor-core router weight gradient stores dz as two bf16 parts,
hi = bf16(dz) and lo = bf16(dz - hi) (round to nearest even): their sum keeps
about 16 mantissa bits of dz, and x^T (hi + lo) with exact bf16 x and fp32
sums stays within the router-gradient tolerance of the fp64 x^T dz."""
import numpy as np
import torch


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).float().numpy()


def test_two_part_bf16_split_keeps_16_bits():
    rng = np.random.default_rng(0)
    dz = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    hi = _bf16(dz)
    lo = _bf16(dz.astype(np.float64) - hi.astype(np.float64))
    err = np.abs(hi.astype(np.float64) + lo - dz.astype(np.float64))
    assert np.all(err <= 2.0 ** -16 * np.abs(dz.astype(np.float64)))
    # one part alone keeps only about 8 bits
    assert np.max(np.abs(hi - dz) / np.abs(dz)) > 2.0 ** -10


def test_split_product_matches_fp64_within_tolerance():
    rng = np.random.default_rng(1)
    T, d, E, K = 2048, 64, 16, 4
    x = _bf16(rng.standard_normal((T, d)))
    dz = np.zeros((T, E))
    for t in range(T):  # K non-zeros per token that sum to zero, like the router's dz
        e = rng.choice(E, K, replace=False)
        v = rng.standard_normal(K) * 1e-3
        dz[t, e] = v - v.mean()
    dz32 = dz.astype(np.float32)
    hi = _bf16(dz32)
    lo = _bf16(dz32.astype(np.float64) - hi)
    ref = dz.T @ x.astype(np.float64)
    got = (hi.T.astype(np.float32) @ x.astype(np.float32)) + (lo.T.astype(np.float32) @ x.astype(np.float32))
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-4
    # the rows of dW_g still sum to zero over experts to the same accuracy
    assert np.abs(got.sum(axis=0)).max() <= 1e-3 * np.abs(got).max()
