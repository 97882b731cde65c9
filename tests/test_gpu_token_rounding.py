"""GPU token rounding (moe_token_rounding) and the layer on the rounded routing
(moe_forward_rows / moe_backward_rows) against the CPU oracle."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import token_rounding as TR
from tests.gpu_common import TOL_BF16, TOL_ROUTER, cpu, rel_fro, to_dev
from token_dispatch_grouped_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _layer(s):
    from token_dispatch_grouped_gb300.layer import MoELayer
    return MoELayer(s.T, s.d, s.E, s.K, s.h, expert=s.expert)


def _gpu_sets(rr, T, E):
    """final [T,E] and w [T,E] from the GPU's row routing, checking its index."""
    off = cpu(rr.offsets).astype(np.int64)
    N = int(off[-1])
    eti = cpu(rr.eti)[:N].astype(np.int64)
    w_row = cpu(rr.w_row)[:N].astype(np.float64)
    tok_off = cpu(rr.tok_off).astype(np.int64)
    tok_exp = cpu(rr.tok_exp)[:N].astype(np.int64)
    tok_rows = cpu(rr.tok_rows)[:N].astype(np.int64)
    assert tok_off[0] == 0 and tok_off[-1] == N and np.all(np.diff(tok_off) >= 0)
    final = np.zeros((T, E), dtype=bool)
    w = np.zeros((T, E))
    for e in range(E):
        seg = eti[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)                       # ascending tokens
        final[seg, e] = True
        w[seg, e] = w_row[off[e]:off[e + 1]]
    for t in range(T):
        ex = tok_exp[tok_off[t]:tok_off[t + 1]]
        rows = tok_rows[tok_off[t]:tok_off[t + 1]]
        assert np.all(np.diff(ex) > 0)
        assert np.array_equal(np.sort(np.nonzero(final[t])[0]), ex)
        for e, r in zip(ex, rows):
            assert off[e] <= r < off[e + 1] and eti[r] == t
    return final, w, off


def _check_against_oracle(z, ids, K, m, final, w, off):
    ref = TR.token_rounding(z, K, m, ids=ids)
    assert np.array_equal(np.diff(off), ref["n"])             # counts: exact integers
    E = z.shape[1]
    for e in range(E):
        diff = np.nonzero(final[:, e] != ref["final"][:, e])[0]
        if len(diff):
            # only a near-tie at the selection boundary may differ (fp32 scores on the GPU)
            p = ref["p"][:, e]
            cand = ~ref["tc"][:, e] if ref["up"][e] else ref["tc"][:, e]
            kept, out = p[cand & ref["final"][:, e]], p[cand & ~ref["final"][:, e]]
            edges = [v for v in (kept.min() if len(kept) else None,
                                 out.max() if len(out) else None) if v is not None]
            for t in diff:
                assert min(abs(p[t] - v) for v in edges) <= 1e-6 * max(p[t], 1e-30), (e, t)
    rows_ok = final.sum(axis=1) > 0
    for t in np.nonzero(rows_ok)[0]:
        sel = final[t]
        assert rel_fro(w[t, sel], O.softmax(z[t, sel])) <= TOL_ROUTER


CASES = [I.Shape(1000, 256, 8, 2, 256), I.Shape(3000, 128, 16, 4, 256),
         I.Shape(700, 256, 32, 6, 256), I.Shape(333, 128, 4, 1, 256),
         I.Shape(2100, 512, 4, 2, 512), I.Shape(1100, 512, 8, 2, 768, "relu")]


@pytest.mark.parametrize("s", CASES, ids=lambda s: f"T{s.T}d{s.d}E{s.E}K{s.K}h{s.h}{s.expert}")
@pytest.mark.parametrize("m", [128, 64])
def test_token_rounding_routing(s, m):
    inp = I.make_layer_inputs(s, seed=2)
    dv = to_dev(inp)
    L = _layer(s)
    r = L.route(dv["x"], dv["Wg"])
    dp = L.dispatch(r.ids)
    rr = L.round_tokens(r.logits, r, dp, m_tile=m)
    L.check_error()
    final, w, off = _gpu_sets(rr, s.T, s.E)
    counts = np.diff(off)
    f = np.diff(cpu(dp.offsets))
    assert np.all((counts % m == 0) | (counts == s.T))
    assert np.all(np.abs(counts - f) < m)
    _check_against_oracle(cpu(r.logits).astype(np.float64), cpu(r.ids), s.K, m, final, w, off)


@pytest.mark.parametrize("s", CASES[:3] + CASES[4:], ids=lambda s: f"T{s.T}d{s.d}E{s.E}K{s.K}{s.expert}")
def test_layer_on_rounded_routing(s):
    inp = I.make_layer_inputs(s, seed=3)
    dv = to_dev(inp)
    L = _layer(s)
    r = L.route(dv["x"], dv["Wg"])
    dp = L.dispatch(r.ids)
    rr = L.round_tokens(r.logits, r, dp, m_tile=64)
    y = torch.full((s.T, s.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    y, H = L.forward_rows(dv["x"], dv["W1"], dv["W3"], dv["W2"], rr, y=y)
    g = L.alloc_grads()
    for t in g.values():
        if t is not None:
            t.fill_(float("nan"))
    g = L.backward_rows(dv["dO"], dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], rr, H, g)
    L.check_error()
    final, w, off = _gpu_sets(rr, s.T, s.E)
    f = TR.layer_forward_sets(inp["x"], inp["W1"], inp["W3"], inp["W2"], final, w, s.expert)
    b = TR.layer_backward_sets(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"],
                               final, w, f, s.expert)
    assert rel_fro(cpu(y), f["y"]) <= TOL_BF16
    keys = ("dx", "dWg", "dW1", "dW2") + (("dW3",) if s.gated else ())
    for k in keys:
        assert not np.isnan(cpu(g[k])).any(), k
        assert rel_fro(cpu(g[k]), b[k]) <= TOL_BF16, k
    N = int(off[-1])
    eti = cpu(rr.eti)[:N].astype(np.int64)
    ds_ref = np.concatenate([b["dS"][eti[off[e]:off[e + 1]], e] for e in range(s.E)])
    assert rel_fro(cpu(g["dS_row"])[:N], ds_ref) <= TOL_BF16


def test_router_dwg_paths_on_rounded_routing(monkeypatch):
    """The router weight gradient of the row-format backward by the tensor-core
    path (forced) agrees with the gathered path and with the oracle."""
    s = I.Shape(1000, 256, 8, 2, 256)
    inp = I.make_layer_inputs(s, seed=3)
    dv = to_dev(inp)
    L = _layer(s)
    r = L.route(dv["x"], dv["Wg"])
    dp = L.dispatch(r.ids)
    rr = L.round_tokens(r.logits, r, dp, m_tile=64)
    dwg = {}
    for path in ("gather", "mma"):
        monkeypatch.setenv("MOE_ROUTER_DWG", path)
        y, H = L.forward_rows(dv["x"], dv["W1"], dv["W3"], dv["W2"], rr)
        g = L.backward_rows(dv["dO"], dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], rr, H)
        L.check_error()
        dwg[path] = cpu(g["dWg"]).astype(np.float64)
    monkeypatch.delenv("MOE_ROUTER_DWG")
    final, w, off = _gpu_sets(rr, s.T, s.E)
    f = TR.layer_forward_sets(inp["x"], inp["W1"], inp["W3"], inp["W2"], final, w, s.expert)
    b = TR.layer_backward_sets(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"],
                               final, w, f, s.expert)
    assert rel_fro(dwg["mma"], b["dWg"]) <= TOL_BF16
    assert rel_fro(dwg["mma"], dwg["gather"]) <= 1e-4


def test_rounding_is_identity_on_tile_multiples():
    """Every expert chosen by a multiple of M_tile tokens: the rounded routing is
    the token-choice routing and the row layer equals the top-K layer."""
    s = I.Shape(512, 256, 4, 2, 256)
    inp = I.make_layer_inputs(s, seed=4)
    dv = to_dev(inp)
    L = _layer(s)
    r = L.route(dv["x"], dv["Wg"])
    ids = torch.tensor([[t % 2, 2 + (t // 2) % 2] for t in range(s.T)], dtype=torch.int32)
    from token_dispatch_grouped_gb300.layer import Routing
    r = Routing(r.logits, ids.cuda(), r.w)
    dp = L.dispatch(r.ids)
    rr = L.round_tokens(r.logits, r, dp, m_tile=128)
    L.check_error()
    assert torch.equal(rr.offsets, dp.offsets)
    assert torch.equal(rr.eti[: s.T * s.K], dp.eti)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["skew", "fine"])
def test_rounding_full_size_properties(name):
    s = I.WORKLOADS[name]
    inp = I.make_layer_inputs(s, seed=0, with_bias=(name == "skew"))
    dv = to_dev(inp)
    L = _layer(s)
    r = L.route(dv["x"], dv["Wg"], dv["bias"])
    dp = L.dispatch(r.ids)
    rr = L.round_tokens(r.logits, r, dp, m_tile=128)
    y, H = L.forward_rows(dv["x"], dv["W1"], dv["W3"], dv["W2"], rr)
    g = L.backward_rows(dv["dO"], dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], rr, H)
    L.check_error()
    off = cpu(rr.offsets).astype(np.int64)
    counts, f = np.diff(off), np.diff(cpu(dp.offsets))
    assert np.all(counts % 128 == 0) and np.all(np.abs(counts - f) < 128)
    assert int(cpu(rr.tok_off)[-1]) == off[-1] <= rr.rows_cap
    for t in (y, g["dx"]):
        assert torch.isfinite(t).all()
