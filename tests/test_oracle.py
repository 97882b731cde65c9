"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here touches the GPU. Each test ties the oracle to something other than
itself: a worked example printed on the pages (tests/golden/), a dense
restatement, torch fp64 autograd, finite differences, closed forms, or exact
invariants. The last tests plant mistakes in the oracle and check that the pins
catch them."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from token_dispatch_grouped_gb300 import inputs as I

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _small(T=24, d=16, E=6, K=2, h=12, seed=3):
    s = I.Shape(T, d, E, K, h)
    inp = I.make_layer_inputs(s, seed=seed)
    return s, inp


# ---------------------------------------------------------------- dispatch index
def test_fig2_worked_example():
    g = _load("moeblaze_fig2.json")
    ids = np.array(g["assignments"])
    eti, off, tim, counts = O.build_dispatch(ids, g["E"])
    assert eti.tolist() == g["expert_token_indices"]
    assert off.tolist() == g["expert_token_offsets"]
    assert tim[: g["K"]].tolist() == g["token_index_map_token0"]
    assert ids.reshape(-1)[:4].tolist() == g["token_expert_indices_prefix"]
    for e, toks in enumerate(g["tokens_per_expert"]):
        assert eti[off[e]:off[e + 1]].tolist() == toks


def test_dropless_skew_tile_example():
    g = _load("dropless_skew_batch.json")
    loads = np.array(g["loads"])
    assert loads.sum() == g["tokens"] * g["top_k"]
    tiles, rows = O.tile_rows(loads, g["block_rows"])
    assert rows.tolist() == g["rounded_loads"]
    assert rows.sum() == g["rounded_total"]
    assert tiles.sum() == 69
    assert round(100.0 * (rows.sum() / loads.sum() - 1.0), 1) == g["overhead_percent"]


@pytest.mark.parametrize("T,E,K,skew", [(1, 4, 1, 0.0), (7, 5, 5, 0.0), (300, 16, 4, 0.0),
                                        (1000, 64, 6, 1.2), (513, 8, 2, 2.5)])
def test_dispatch_invariants(T, E, K, skew):
    ids = I.random_ids(T, E, K, seed=T + E, skew=skew).numpy()
    # every token has exactly K distinct experts
    assert all(len(set(r)) == K for r in ids.tolist())
    eti, off, tim, counts = O.build_dispatch(ids, E)
    TK = T * K
    assert counts.sum() == TK and off[-1] == TK and off[0] == 0
    assert np.all(np.diff(off) == counts)
    # eti is a permutation of the multiset {t repeated K times}
    assert np.array_equal(np.sort(eti), np.repeat(np.arange(T), K))
    # tim is a bijection onto [0, TK) and inverts eti
    assert np.array_equal(np.sort(tim), np.arange(TK))
    tt = np.repeat(np.arange(T), K)
    assert np.array_equal(eti[tim], tt)
    # tokens ascend inside each expert; rows of expert e are exactly its tokens
    for e in range(E):
        seg = eti[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.array_equal(seg, np.nonzero((ids == e).any(axis=1))[0])
    # the position of (t,k) lies in the segment of expert ids[t,k]
    flat = ids.reshape(-1)
    assert np.all((tim >= off[flat]) & (tim < off[flat + 1]))


def test_dispatch_brute_force_tiny():
    # Exhaustive over all 2-of-3 assignments for 3 tokens: positions by counting.
    import itertools
    pairs = list(itertools.permutations(range(3), 2))
    for combo in itertools.product(pairs, repeat=3):
        ids = np.array(combo)
        eti, off, tim, _ = O.build_dispatch(ids, 3)
        for t in range(3):
            for k in range(2):
                e = ids[t, k]
                before = sum(1 for t2 in range(t) if e in ids[t2])
                assert tim[t * 2 + k] == sum((ids == e2).sum() for e2 in range(e)) + before


# ---------------------------------------------------------------- router
def test_router_weights_and_shift_invariance():
    s, inp = _small(T=64, E=8, K=3)
    z, p, ids, w = O.route(inp["x"], inp["Wg"], s.K)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-14)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)
    # descending order, and the chosen are the K largest
    pk = np.take_along_axis(p, ids, axis=1)
    assert np.all(np.diff(pk, axis=1) <= 0)
    assert np.all(pk[:, -1] >= np.sort(p, axis=1)[:, -s.K])
    # adding one constant to every logit changes nothing
    z2, p2, ids2, w2 = O.route(inp["x"], inp["Wg"], s.K, bias=np.full(s.E, 3.25))
    assert np.array_equal(ids, ids2)
    assert np.allclose(w, w2, rtol=1e-12)
    # renormalised weights = softmax over the chosen logits
    zk = np.take_along_axis(z, ids, axis=1)
    assert np.allclose(w, O.softmax(zk), rtol=1e-12)


def test_router_tie_break_lower_id():
    x = np.ones((3, 4))
    Wg = np.zeros((6, 4))
    Wg[[1, 4], :] = 1.0           # experts 1 and 4 tie for the top, then 0,2,3,5 tie
    z, p, ids, w = O.route(x, Wg, 3)
    assert ids.tolist() == [[1, 4, 0]] * 3
    assert np.allclose(w[:, 0], w[:, 1])


def test_router_bias_removes_expert():
    s, inp = _small(T=200, E=8, K=2)
    bias = np.zeros(8)
    bias[[2, 5]] = -1e4
    z, p, ids, w = O.route(inp["x"], inp["Wg"], 2, bias)
    assert not np.isin(ids, [2, 5]).any()


# ---------------------------------------------------------------- forward
def test_sparse_forward_matches_dense_masked():
    s, inp = _small(T=40, d=16, E=5, K=3, h=24)
    z, p, ids, w = O.route(inp["x"], inp["Wg"], s.K)
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w)
    yd = O.dense_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w)
    assert np.allclose(f["y"], yd, rtol=1e-12, atol=1e-12)


def test_forward_matches_sort_permute_pipeline():
    # The sort / gather / per-expert / weight / index-add pipeline, in torch fp64.
    s, inp = _small(T=33, d=8, E=4, K=2, h=10)
    z, p, ids, w = O.route(inp["x"], inp["Wg"], s.K)
    x = inp["x"].double()
    W1, W3, W2 = inp["W1"].double(), inp["W3"].double(), inp["W2"].double()
    te = torch.from_numpy(ids)
    tw = torch.from_numpy(w)
    flat = te.reshape(-1)
    order = torch.argsort(flat, stable=True)
    src = order // s.K
    counts = torch.bincount(flat, minlength=s.E)
    xs = x.index_select(0, src)
    outs = []
    for e, chunk in enumerate(xs.split(counts.tolist())):
        a = chunk @ W1[e].T
        b = chunk @ W3[e].T
        outs.append((torch.nn.functional.silu(a) * b) @ W2[e].T)
    ys = torch.cat(outs) * tw.reshape(-1)[order].unsqueeze(-1)
    y = torch.zeros_like(x).index_add_(0, src, ys)
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w)
    assert np.allclose(f["y"], y.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward
def _torch_expert(xe, W1e, W3e, W2e, expert):
    a = xe @ W1e.T
    if expert == "swiglu":
        A = torch.nn.functional.silu(a) * (xe @ W3e.T)
    elif expert == "silu":
        A = torch.nn.functional.silu(a)
    else:
        A = torch.relu(a)
    return A @ W2e.T


def _torch_layer(x, Wg, W1, W3, W2, ids, bias=None, expert="swiglu"):
    """Whole layer (full softmax, gather of the fixed top-K, renormalise,
    per-expert FFN, weighted sum) for torch autograd."""
    z = x @ Wg.T
    if bias is not None:
        z = z + bias
    p = torch.softmax(z, dim=1)
    pk = p.gather(1, ids)
    w = pk / pk.sum(dim=1, keepdim=True)
    T, K = ids.shape
    y = torch.zeros_like(x)
    for k in range(K):
        for e in range(W1.shape[0]):
            m = ids[:, k] == e
            if m.any():
                xe = x[m]
                Ye = _torch_expert(xe, W1[e], None if W3 is None else W3[e], W2[e], expert)
                y = y.index_add(0, torch.nonzero(m).squeeze(1), w[m, k:k + 1] * Ye)
    return y


def _autograd_reference(inp, ids, bias=None, expert="swiglu"):
    names = ("x", "Wg", "W1", "W3", "W2") if expert == "swiglu" else ("x", "Wg", "W1", "W2")
    leaves = {k: inp[k].double().clone().requires_grad_(True) for k in names}
    y = _torch_layer(leaves["x"], leaves["Wg"], leaves["W1"], leaves.get("W3"), leaves["W2"],
                     torch.from_numpy(ids), None if bias is None else torch.from_numpy(bias),
                     expert)
    (y * inp["dO"].double()).sum().backward()
    return y.detach().numpy(), {k: v.grad.numpy() for k, v in leaves.items()}


@pytest.mark.parametrize("K", [1, 2, 3])
def test_backward_matches_torch_autograd(K):
    s, inp = _small(T=30, d=12, E=5, K=K, h=16)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"], K)
    y_ref, g = _autograd_reference(inp, st["ids"])
    b = st["bwd"]
    assert np.allclose(st["fwd"]["y"], y_ref, rtol=1e-10, atol=1e-12)
    for ours, ref in (("dx", "x"), ("dWg", "Wg"), ("dW1", "W1"), ("dW3", "W3"), ("dW2", "W2")):
        assert np.allclose(b[ours], g[ref], rtol=1e-9, atol=1e-11), ours
    if K == 1:                                   # w == 1, so no router gradient
        assert np.abs(b["dWg"]).max() < 1e-14 and np.abs(b["dz"]).max() < 1e-14


def test_backward_finite_differences():
    s, inp = _small(T=10, d=6, E=4, K=2, h=8, seed=11)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"], 2)
    base = {k: O._as64(inp[k]) for k in ("x", "Wg", "W1", "W3", "W2")}
    dO = O._as64(inp["dO"])

    def loss(v):
        z, p, ids, w = O.route(v["x"], v["Wg"], 2)
        assert np.array_equal(ids, st["ids"])     # the perturbation keeps the routing
        return float(np.sum(O.layer_forward(v["x"], v["W1"], v["W3"], v["W2"], ids, w)["y"] * dO))

    rng = np.random.default_rng(0)
    eps = 1e-6
    for name, gname in (("x", "dx"), ("Wg", "dWg"), ("W1", "dW1"), ("W3", "dW3"), ("W2", "dW2")):
        for _ in range(4):
            idx = tuple(rng.integers(0, n) for n in base[name].shape)
            if name.startswith("W") and name != "Wg":
                idx = (int(st["ids"][0, 0]),) + idx[1:]     # an expert that has tokens
            vp = {k: v.copy() for k, v in base.items()}
            vm = {k: v.copy() for k, v in base.items()}
            vp[name][idx] += eps
            vm[name][idx] -= eps
            fd = (loss(vp) - loss(vm)) / (2 * eps)
            an = st["bwd"][gname][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)


def test_dS_identity_down_projection():
    # <dO_t, Y_{t,k}> = <dA'_r, A_r> with dA' = dO W2_e (SonicMoE 3.4.1)
    s, inp = _small(T=50, d=16, E=4, K=2, h=20)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"], 2)
    f = st["fwd"]
    dO = O._as64(inp["dO"])
    W2 = O._as64(inp["W2"])
    ids = st["ids"]
    for t in range(s.T):
        for k in range(2):
            r = f["tim"][t * 2 + k]
            dAp = dO[t] @ W2[ids[t, k]]
            assert np.isclose(st["bwd"]["dS"][t, k], dAp @ f["A"][r], rtol=1e-11, atol=1e-12)


def test_router_dz_closed_form_and_sum_zero():
    rng = np.random.default_rng(1)
    w = O.softmax(rng.normal(size=(20, 4)))
    dS = rng.normal(size=(20, 4))
    dz = O.router_backward_dz(w, dS)
    closed = w * (dS - np.sum(w * dS, axis=1, keepdims=True))
    assert np.allclose(dz, closed, rtol=1e-12, atol=1e-14)
    assert np.allclose(dz.sum(axis=1), 0.0, atol=1e-14)


def test_sampled_definitions_match_full_oracle():
    s, inp = _small(T=20, d=10, E=4, K=2, h=14, seed=5)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"], 2)
    toks = [0, 7, 19]
    y, dS, dx = O.tokens_forward_backward(toks, inp["x"], inp["dO"], inp["Wg"], inp["W1"],
                                          inp["W3"], inp["W2"], st["ids"], st["w"])
    assert np.allclose(y, st["fwd"]["y"][toks], rtol=1e-11, atol=1e-12)
    assert np.allclose(dS, st["bwd"]["dS"][toks], rtol=1e-11, atol=1e-12)
    assert np.allclose(dx, st["bwd"]["dx"][toks], rtol=1e-10, atol=1e-12)
    for e in range(4):
        for j in (0, 13):
            g1, g3, g2 = O.hidden_unit_grads(e, j, inp["x"], inp["dO"], inp["W1"], inp["W3"],
                                             inp["W2"], st["ids"], st["w"])
            assert np.allclose(g1, st["bwd"]["dW1"][e, j], rtol=1e-10, atol=1e-12)
            assert np.allclose(g3, st["bwd"]["dW3"][e, j], rtol=1e-10, atol=1e-12)
            assert np.allclose(g2, st["bwd"]["dW2"][e, :, j], rtol=1e-10, atol=1e-12)


def test_empty_expert_gets_zero_grads():
    s, inp = _small(T=16, d=8, E=6, K=2, h=8)
    ids = I.random_ids(16, 4, 2, seed=2).numpy()        # experts 4, 5 never chosen
    w = I.random_weights(16, 2, seed=2).numpy()
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ids, w)
    for n in ("dW1", "dW3", "dW2"):
        assert np.all(b[n][4:] == 0.0)
    assert np.all(b["dWg"][4:] == 0.0)


# ---------------------------------------------------------------- planted mistakes
def test_pins_catch_planted_silu_grad_error(monkeypatch):
    s, inp = _small(T=12, d=8, E=4, K=2, h=8)
    z, p, ids, w = O.route(inp["x"], inp["Wg"], 2)
    monkeypatch.setattr(O, "silu_grad", lambda u: O.sigmoid(u))     # dropped term
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ids, w)
    monkeypatch.undo()
    _, g = _autograd_reference(inp, ids)
    assert not np.allclose(b["dW1"], g["W1"], rtol=1e-6, atol=1e-8)


def test_pins_catch_planted_index_error(monkeypatch):
    g = _load("moeblaze_fig2.json")
    real = O.build_dispatch

    def wrong(ids, E):                      # transposed roles of the two maps
        eti, off, tim, c = real(ids, E)
        return tim, off, eti, c
    monkeypatch.setattr(O, "build_dispatch", wrong)
    eti, off, tim, _ = O.build_dispatch(np.array(g["assignments"]), g["E"])
    assert eti.tolist() != g["expert_token_indices"]


def test_pins_catch_planted_router_sign(monkeypatch):
    rng = np.random.default_rng(4)
    w = O.softmax(rng.normal(size=(5, 3)))
    dS = rng.normal(size=(5, 3))
    good = O.router_backward_dz(w, dS)
    monkeypatch.setattr(O.np, "outer", lambda a, b: -np.multiply.outer(a, b))
    bad = O.router_backward_dz(w, dS)
    monkeypatch.undo()
    assert not np.allclose(bad.sum(axis=1), 0.0)       # the sum-zero pin fails
    assert np.allclose(good.sum(axis=1), 0.0)


# ---------------------------------------------------------------- non-gated experts
@pytest.mark.parametrize("expert", ["silu", "relu"])
def test_non_gated_matches_dense_and_autograd(expert):
    s, inp = _small(T=36, d=12, E=5, K=3, h=20, seed=7)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], None, inp["W2"], inp["dO"], s.K,
                      expert=expert)
    assert st["fwd"]["H"].shape == (s.T * s.K, s.h)
    yd = O.dense_forward(inp["x"], inp["W1"], None, inp["W2"], st["ids"], st["w"], expert)
    assert np.allclose(st["fwd"]["y"], yd, rtol=1e-12, atol=1e-12)
    y_ref, g = _autograd_reference(inp, st["ids"], expert=expert)
    assert np.allclose(st["fwd"]["y"], y_ref, rtol=1e-10, atol=1e-12)
    b = st["bwd"]
    assert b["dW3"] is None
    for ours, ref in (("dx", "x"), ("dWg", "Wg"), ("dW1", "W1"), ("dW2", "W2")):
        assert np.allclose(b[ours], g[ref], rtol=1e-9, atol=1e-11), ours


def test_non_gated_finite_differences_silu():
    s, inp = _small(T=10, d=6, E=4, K=2, h=8, seed=13)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], None, inp["W2"], inp["dO"], 2,
                      expert="silu")
    base = {k: O._as64(inp[k]) for k in ("x", "Wg", "W1", "W2")}
    dO = O._as64(inp["dO"])

    def loss(v):
        z, p, ids, w = O.route(v["x"], v["Wg"], 2)
        assert np.array_equal(ids, st["ids"])
        return float(np.sum(O.layer_forward(v["x"], v["W1"], None, v["W2"], ids, w, "silu")["y"] * dO))

    rng = np.random.default_rng(3)
    eps = 1e-6
    for name, gname in (("x", "dx"), ("Wg", "dWg"), ("W1", "dW1"), ("W2", "dW2")):
        for _ in range(4):
            idx = tuple(rng.integers(0, n) for n in base[name].shape)
            if name in ("W1", "W2"):
                idx = (int(st["ids"][0, 0]),) + idx[1:]
            vp = {k: v.copy() for k, v in base.items()}
            vm = {k: v.copy() for k, v in base.items()}
            vp[name][idx] += eps
            vm[name][idx] -= eps
            fd = (loss(vp) - loss(vm)) / (2 * eps)
            an = st["bwd"][gname][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)


@pytest.mark.parametrize("expert", ["silu", "relu"])
def test_non_gated_sampled_definitions(expert):
    s, inp = _small(T=20, d=10, E=4, K=2, h=14, seed=9)
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], None, inp["W2"], inp["dO"], 2,
                      expert=expert)
    toks = [1, 8, 19]
    y, dS, dx = O.tokens_forward_backward(toks, inp["x"], inp["dO"], inp["Wg"], inp["W1"], None,
                                          inp["W2"], st["ids"], st["w"], expert)
    assert np.allclose(y, st["fwd"]["y"][toks], rtol=1e-11, atol=1e-12)
    assert np.allclose(dS, st["bwd"]["dS"][toks], rtol=1e-11, atol=1e-12)
    assert np.allclose(dx, st["bwd"]["dx"][toks], rtol=1e-10, atol=1e-12)
    for e in range(4):
        g1, g3, g2 = O.hidden_unit_grads(e, 5, inp["x"], inp["dO"], inp["W1"], None, inp["W2"],
                                         st["ids"], st["w"], expert)
        assert g3 is None
        assert np.allclose(g1, st["bwd"]["dW1"][e, 5], rtol=1e-10, atol=1e-12)
        assert np.allclose(g2, st["bwd"]["dW2"][e, :, 5], rtol=1e-10, atol=1e-12)


def test_pins_catch_planted_relu_grad_error(monkeypatch):
    s, inp = _small(T=12, d=8, E=4, K=2, h=8)
    z, p, ids, w = O.route(inp["x"], inp["Wg"], 2)
    monkeypatch.setattr(O, "relu_grad", lambda u: np.ones_like(u))     # identity slope
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], None, inp["W2"], ids, w,
                         expert="relu")
    monkeypatch.undo()
    _, g = _autograd_reference(inp, ids, expert="relu")
    assert not np.allclose(b["dW1"], g["W1"], rtol=1e-6, atol=1e-8)


def test_topk_gap_sees_membership_and_order_gaps():
    """The gap that decides which router ids the GPU tests compare: the smallest
    difference among the K+1 largest logits, so both the K-th vs (K+1)-th gap
    (set membership) and gaps inside the top K (slot order) count."""
    z = np.array([[5.0, 4.0, 3.0, 2.99995, 0.0],    # K=3: membership decided by 5e-5
                  [5.0, 4.99995, 3.0, 1.0, 0.0],    # order of slots 0/1 decided by 5e-5
                  [9.0, 7.0, 5.0, 3.0, 1.0],        # every gap 2
                  [1.0, 1.0, 0.0, -1.0, -2.0]])     # exact tie in the top K
    g = O.topk_gap(z, 3)
    assert g[0] == pytest.approx(5e-5, abs=1e-9) and g[1] == pytest.approx(5e-5, abs=1e-9)
    assert g[2] == pytest.approx(2.0) and g[3] == 0.0
    # K = E: only the order inside the top K matters
    assert O.topk_gap(np.array([[3.0, 1.0, 0.0]]), 3)[0] == pytest.approx(1.0)
    # the gap is invariant to the order of the experts
    perm = np.array([4, 2, 0, 3, 1])
    assert np.allclose(O.topk_gap(z[:, perm], 3), g)


@pytest.mark.parametrize("expert", ["swiglu", "silu", "relu"])
def test_batched_sampled_definitions_match_full_oracle(expert):
    """The batched sampled helpers (one expert at a time over the sampled rows;
    many hidden units at once) give the full oracle's values, including a token
    list with every token and an expert that no sampled token uses."""
    s, inp = _small(T=24, d=10, E=5, K=3, h=14, seed=17)
    W3 = inp["W3"] if expert == "swiglu" else None
    st = O.layer_step(inp["x"], inp["Wg"], inp["W1"], W3, inp["W2"], inp["dO"], 3,
                      expert=expert)
    for toks in ([0, 5, 23], list(range(24))):
        y, dS, dx = O.tokens_forward_backward_batched(toks, inp["x"], inp["dO"], inp["Wg"],
                                                      inp["W1"], W3, inp["W2"], st["ids"],
                                                      st["w"], expert)
        assert np.allclose(y, st["fwd"]["y"][toks], rtol=1e-11, atol=1e-12)
        assert np.allclose(dS, st["bwd"]["dS"][toks], rtol=1e-11, atol=1e-12)
        assert np.allclose(dx, st["bwd"]["dx"][toks], rtol=1e-10, atol=1e-12)
    js = [0, 6, 13]
    for e in range(5):
        g1, g3, g2 = O.hidden_units_grads(e, js, inp["x"], inp["dO"], inp["W1"], W3, inp["W2"],
                                          st["ids"], st["w"], expert)
        assert np.allclose(g1, st["bwd"]["dW1"][e][js], rtol=1e-10, atol=1e-12)
        assert np.allclose(g2, st["bwd"]["dW2"][e][:, js], rtol=1e-10, atol=1e-12)
        if expert == "swiglu":
            assert np.allclose(g3, st["bwd"]["dW3"][e][js], rtol=1e-10, atol=1e-12)
        else:
            assert g3 is None
    # an expert without tokens: exact zeros of the right shapes
    ids = np.where(st["ids"] == 4, 0, st["ids"])
    ids[:, 1:] = np.where(ids[:, 1:] == ids[:, :1], 3, ids[:, 1:])
    g1, g3, g2 = O.hidden_units_grads(4, js, inp["x"], inp["dO"], inp["W1"], W3, inp["W2"],
                                      ids, st["w"], expert)
    assert g1.shape == (3, 10) and g2.shape == (10, 3) and not g1.any() and not g2.any()
