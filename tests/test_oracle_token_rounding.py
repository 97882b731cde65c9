"""Pins of the token-rounding oracle (SonicMoE notes 3.4.4, Algorithm 4, NR-f)
against the guarantees the pages state, a hand-derived example, the top-K
layer it must reduce to, and finite differences. CPU only."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import token_rounding as TR
from token_dispatch_grouped_gb300 import inputs as I


def _logits(T, E, seed, skew=0.0):
    g = np.random.default_rng(seed)
    z = g.standard_normal((T, E))
    if skew:
        z = z - skew * np.log(np.arange(1, E + 1))[None, :]
    return z


@pytest.mark.parametrize("T,E,K,m,skew", [(1000, 8, 2, 128, 0.0), (3000, 16, 4, 128, 1.0),
                                          (700, 32, 6, 64, 0.5), (333, 4, 1, 128, 0.0)])
def test_counts_are_nearest_tile_multiples(T, E, K, m, skew):
    r = TR.token_rounding(_logits(T, E, T + E, skew), K, m)
    f, n = r["f"], r["n"]
    assert np.array_equal(r["final"].sum(axis=0), n)
    assert np.array_equal(r["tc"].sum(axis=0), f) and f.sum() == T * K
    for fe, ne in zip(f, n):
        if ne < T:                               # an expert capped at T is the only exception
            assert ne % m == 0
        assert abs(int(ne) - int(fe)) < m        # at most one tile away from token choice
        lo, hi = (fe // m) * m, -(-fe // m) * m
        # nearest multiple; a tie rounds down
        assert ne == min(T, hi if (hi - fe) < (fe - lo) else lo)


@pytest.mark.parametrize("seed", [1, 2])
def test_only_the_last_tile_changes(seed):
    """Rounding down drops only the lowest-scoring token-choice tokens; rounding
    up keeps every token-choice token and adds the best other tokens."""
    T, E, K, m = 1500, 12, 3, 128
    z = _logits(T, E, seed, 0.7)
    r = TR.token_rounding(z, K, m)
    p = O.softmax(z)
    for e in range(E):
        tc, fin = r["tc"][:, e], r["final"][:, e]
        if r["n"][e] <= r["f"][e]:               # rounded down (or unchanged)
            assert not (fin & ~tc).any()         # nothing added
            kept, dropped = p[tc & fin, e], p[tc & ~fin, e]
            if len(kept) and len(dropped):
                assert dropped.max() <= kept.min()
        else:                                    # rounded up
            assert (fin | ~tc).all()             # every token-choice token kept
            added, rest = p[fin & ~tc, e], p[~fin & ~tc, e]
            if len(added) and len(rest):
                assert added.min() >= rest.max()


def test_identity_when_counts_are_tile_multiples():
    """With every token-choice count a multiple of M_tile, token rounding is
    token choice, and the set-based layer is the top-K layer."""
    T, E, K, m, d, h = 256, 4, 2, 128, 8, 6
    # token t prefers experts (t % 2, 2 + t % 2): every expert gets 128 tokens
    z = np.full((T, E), -3.0)
    g = np.random.default_rng(0)
    for t in range(T):
        z[t, t % 2] = 2.0 + g.random()
        z[t, 2 + t % 2] = 1.0 + g.random()
    r = TR.token_rounding(z, K, m)
    assert np.array_equal(r["final"], r["tc"])
    ids = np.argsort(-O.softmax(z), axis=1, kind="stable")[:, :K]
    pk = np.take_along_axis(O.softmax(z), ids, axis=1)
    wk = pk / pk.sum(axis=1, keepdims=True)
    assert np.allclose(np.take_along_axis(r["w"], ids, axis=1), wk, rtol=1e-12)
    x = g.standard_normal((T, d))
    W1, W3 = g.standard_normal((E, h, d)), g.standard_normal((E, h, d))
    W2 = g.standard_normal((E, d, h))
    Wg = g.standard_normal((E, d))
    dO = g.standard_normal((T, d))
    f1 = O.layer_forward(x, W1, W3, W2, ids, wk)
    f2 = TR.layer_forward_sets(x, W1, W3, W2, r["final"], r["w"])
    assert np.allclose(f1["y"], f2["y"], rtol=1e-10, atol=1e-10)
    b1 = O.layer_backward(dO, x, Wg, W1, W3, W2, ids, wk, f1)
    b2 = TR.layer_backward_sets(dO, x, Wg, W1, W3, W2, r["final"], r["w"], f2)
    for k in ("dx", "dWg", "dW1", "dW3", "dW2"):
        assert np.allclose(b1[k], b2[k], rtol=1e-9, atol=1e-9), k


def test_hand_example():
    """T = 6, E = 3, K = 1, M_tile = 4. Token choice: tokens 0-2 pick expert 0,
    tokens 3-4 expert 1, token 5 expert 2, so f = (3, 2, 1).
    Expert 0: floor 0, ceil 4, ceil - f = 1 < f - floor = 3: pad to 4 with the
    best other token for expert 0, which is token 4 (probability 0.3 of its row
    against 0.2 for tokens 3 and 5).
    Expert 1: floor 0, ceil 4, distances 2 and 2: a tie rounds down, both
    tokens dropped. Expert 2: distances 3 and 1: rounds down, token 5 dropped.
    Final sets: tokens 0-2 and 4 keep expert 0 alone (weight 1); tokens 3 and
    5 have no expert."""
    P = np.array([[0.8, 0.1, 0.1], [0.7, 0.2, 0.1], [0.6, 0.3, 0.1],
                  [0.2, 0.7, 0.1], [0.3, 0.6, 0.1], [0.2, 0.1, 0.7]])
    z = np.log(P)
    r = TR.token_rounding(z, 1, 4)
    assert r["f"].tolist() == [3, 2, 1] and r["n"].tolist() == [4, 0, 0]
    assert r["up"].tolist() == [True, False, False]
    assert r["final"].astype(int).tolist() == [[1, 0, 0], [1, 0, 0], [1, 0, 0],
                                                [0, 0, 0], [1, 0, 0], [0, 0, 0]]
    assert np.allclose(r["w"][:, 0], [1, 1, 1, 0, 1, 0]) and not r["w"][:, 1:].any()
    rows = TR.rows_of(r["final"])
    assert rows["eti"].tolist() == [0, 1, 2, 4]
    assert rows["offsets"].tolist() == [0, 4, 4, 4]
    assert rows["tok_off"].tolist() == [0, 1, 2, 3, 3, 4, 4]
    assert rows["tok_rows"].tolist() == [0, 1, 2, 3]


def _dense_loss(Wg, x, W1, W3, W2, dO, final):
    """<dO, y> with the expert sets held fixed, through torch (an independent
    restatement of the set-based forward, for finite differences)."""
    z = x @ Wg.T
    T, E = final.shape
    y = torch.zeros_like(x)
    for t in range(T):
        sel = torch.nonzero(final[t]).flatten()
        if len(sel) == 0:
            continue
        w = torch.softmax(z[t, sel], dim=0)
        for j, e in enumerate(sel.tolist()):
            a = x[t] @ W1[e].T
            b = x[t] @ W3[e].T
            y[t] = y[t] + w[j] * ((torch.nn.functional.silu(a) * b) @ W2[e].T)
    return (dO * y).sum()


def test_router_gradient_against_autograd():
    T, E, K, d, h = 40, 6, 2, 8, 5
    g = np.random.default_rng(4)
    x = g.standard_normal((T, d))
    Wg = g.standard_normal((E, d))
    W1, W3 = g.standard_normal((E, h, d)), g.standard_normal((E, h, d))
    W2 = g.standard_normal((E, d, h))
    dO = g.standard_normal((T, d))
    r = TR.token_rounding(x @ Wg.T, K, 8)
    assert not np.array_equal(r["final"], r["tc"])          # rounding changed the sets
    b = TR.layer_backward_sets(dO, x, Wg, W1, W3, W2, r["final"], r["w"])
    t = {k: torch.tensor(v, dtype=torch.float64) for k, v in
         dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, dO=dO).items()}
    t["Wg"].requires_grad_(True)
    t["x"].requires_grad_(True)
    loss = _dense_loss(t["Wg"], t["x"], t["W1"], t["W3"], t["W2"], t["dO"],
                       torch.tensor(r["final"]))
    loss.backward()
    assert np.allclose(b["dWg"], t["Wg"].grad.numpy(), rtol=1e-9, atol=1e-9)
    assert np.allclose(b["dx"], t["x"].grad.numpy(), rtol=1e-9, atol=1e-9)


def test_planted_mistake_is_caught():
    """Renormalising the weights over all experts instead of the final set
    breaks the router gradient pin."""
    T, E, K, d, h = 30, 5, 2, 6, 4
    g = np.random.default_rng(9)
    x = g.standard_normal((T, d))
    Wg = g.standard_normal((E, d))
    W1, W3 = g.standard_normal((E, h, d)), g.standard_normal((E, h, d))
    W2 = g.standard_normal((E, d, h))
    dO = g.standard_normal((T, d))
    r = TR.token_rounding(x @ Wg.T, K, 8)
    w_bad = np.where(r["final"], O.softmax(x @ Wg.T), 0.0)
    b = TR.layer_backward_sets(dO, x, Wg, W1, W3, W2, r["final"], w_bad)
    t = {k: torch.tensor(v, dtype=torch.float64) for k, v in
         dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, dO=dO).items()}
    t["Wg"].requires_grad_(True)
    _dense_loss(t["Wg"], t["x"], t["W1"], t["W3"], t["W2"], t["dO"],
                torch.tensor(r["final"])).backward()
    assert not np.allclose(b["dWg"], t["Wg"].grad.numpy(), rtol=1e-6, atol=1e-6)


def test_rows_are_a_consistent_index():
    T, E, K = 500, 8, 2
    r = TR.token_rounding(_logits(T, E, 5, 0.3), K, 32)
    rows = TR.rows_of(r["final"])
    eti, off, tok_off, tok_exp, tok_rows = (rows[k] for k in
                                            ("eti", "offsets", "tok_off", "tok_exp", "tok_rows"))
    assert off[-1] == r["final"].sum() == tok_off[-1]
    for e in range(E):
        seg = eti[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)                          # ascending tokens
    for t in range(T):
        ex = tok_exp[tok_off[t]:tok_off[t + 1]]
        rr = tok_rows[tok_off[t]:tok_off[t + 1]]
        assert np.all(np.diff(ex) > 0)
        for e, row in zip(ex, rr):
            assert off[e] <= row < off[e + 1] and eti[row] == t
