"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Small and ragged shapes are compared element by element; the full workloads are
compared on sampled tokens and hidden units (the oracle evaluates those one by
one) and on properties that hold at any size."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.gpu_common import GAP, TOL_BF16, TOL_ROUTER, TOL_ROW, cpu, rel_fro, rel_rows, to_dev
from token_dispatch_grouped_gb300 import inputs as I

pytestmark = pytest.mark.gpu

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _layer(s):
    from token_dispatch_grouped_gb300.layer import MoELayer
    return MoELayer(s.T, s.d, s.E, s.K, s.h, expert=s.expert)


def _wgrad_keys(s):
    return ("dW1", "dW3", "dW2") if s.gated else ("dW1", "dW2")


def _check_route(z_gpu, ids_gpu, w_gpu, x, Wg, K, bias, rows=None):
    xs = x if rows is None else x[rows]
    z, p, ids, w = O.route(xs, Wg, K, None if bias is None else bias)
    zg = cpu(z_gpu) if rows is None else cpu(z_gpu)[rows]
    ig = cpu(ids_gpu) if rows is None else cpu(ids_gpu)[rows]
    wg = cpu(w_gpu) if rows is None else cpu(w_gpu)[rows]
    assert rel_fro(zg, z) <= TOL_ROUTER
    sure = O.topk_gap(z, K) > GAP
    assert sure.mean() > 0.5
    assert np.array_equal(ig[sure], ids[sure])
    assert rel_fro(wg[sure], w[sure]) <= TOL_ROUTER
    assert np.allclose(wg.sum(axis=1), 1.0, atol=1e-5)


def _check_dispatch(ids_gpu, dp, E):
    eti, off, tim, counts = O.build_dispatch(cpu(ids_gpu), E)
    assert np.array_equal(cpu(dp.eti), eti)
    assert np.array_equal(cpu(dp.offsets), off)
    assert np.array_equal(cpu(dp.tim), tim)


SMALL = [
    I.WORKLOADS["tiny"],
    I.Shape(300, 256, 6, 3, 384),     # ragged tiles, h % 256 != 0 (128-wide N tiles)
    I.Shape(1, 128, 4, 4, 128),       # one token, K = E
    I.Shape(1500, 128, 16, 1, 256),   # K = 1 (router gradient is zero), 2 token chunks
    I.Shape(129, 384, 8, 8, 128),     # K = E = 8
    I.Shape(1100, 512, 8, 2, 256),    # passes split by output columns (d % 512 == 0)
    I.Shape(2100, 512, 4, 2, 512),    # ~1000 rows per expert: CTA-pair (M = 256) tiles
    # non-gated two-layer experts (SiLU / ReLU), no W3
    I.Shape(300, 256, 6, 3, 512, "silu"),    # ragged tiles, two 256-wide up tiles
    I.Shape(1500, 128, 16, 1, 256, "relu"),  # K = 1, 2 token chunks
    I.Shape(1100, 512, 8, 2, 768, "relu"),   # column-split passes, three up tiles
    I.Shape(2100, 512, 4, 2, 256, "silu"),   # CTA-pair down / dX GEMMs
    I.Shape(1200, 2048, 4, 2, 512, "silu"),  # CTA pairs at d = 2048: 128-deep dH stages
]


def _sid(s):
    return f"T{s.T}d{s.d}E{s.E}K{s.K}h{s.h}" + ("" if s.gated else f"-{s.expert}")


@pytest.mark.parametrize("s", SMALL, ids=_sid)
def test_layer_small_full_parity(s):
    inp = I.make_layer_inputs(s, seed=1)
    dv = to_dev(inp)
    L = _layer(s)
    r, dp, y, H, g = L.step(dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], dv["dO"])
    L.check_error()
    _check_route(r.logits, r.ids, r.w, inp["x"], inp["Wg"], s.K, None)
    _check_dispatch(r.ids, dp, s.E)
    # Layer parity on the GPU's own routing (ids and fp32 weights as inputs).
    ids, w = cpu(r.ids), cpu(r.w)
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w, s.expert)
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ids, w, f,
                         s.expert)
    assert H.shape == (s.TK, 2 * s.h if s.gated else s.h)
    assert rel_fro(cpu(H), f["H"]) <= TOL_BF16
    assert rel_fro(cpu(y), f["y"]) <= TOL_BF16
    assert rel_fro(cpu(g["dS"]), b["dS"]) <= TOL_BF16
    for k in ("dx",) + _wgrad_keys(s):
        assert rel_fro(cpu(g[k]), b[k]) <= TOL_BF16, k
    # every row (token, expert row, weight row) on its own
    assert rel_rows(cpu(H), f["H"]) <= TOL_ROW
    assert rel_rows(cpu(y), f["y"]) <= TOL_ROW
    for k in ("dx",) + _wgrad_keys(s):
        assert rel_rows(cpu(g[k]), b[k]) <= TOL_ROW, k
    if s.K == 1:
        assert np.all(cpu(g["dWg"]) == 0.0)
    else:
        assert rel_fro(cpu(g["dWg"]), b["dWg"]) <= TOL_BF16


def _ids_with_counts(T, K, counts, seed):
    """Top-K ids [T, K] whose per-expert counts are exactly `counts` (each at most
    T, summing to T*K): the expert-sorted labels are dealt column by column, so a
    token's K experts are distinct, then the tokens are shuffled."""
    labels = np.repeat(np.arange(len(counts)), counts)
    assert labels.size == T * K and max(counts) <= T
    ids = labels.reshape(K, T).T.copy()
    rng = np.random.default_rng(seed)
    ids = ids[rng.permutation(T)]
    for k in range(K):
        for j in range(k):
            assert not np.any(ids[:, k] == ids[:, j])
    return torch.from_numpy(ids.astype(np.int32))


# CTA-pair GEMMs run an expert's last partial tile of at most 128 rows as a
# half-height tile (M = 128 over the pair, 64 rows per CTA). Counts with
# remainders of 1 and 14 rows (half tiles), an exact multiple of 256 (none), 233
# rows (a whole tile), an expert of 100 rows (only a half tile) and an empty
# expert; forward and backward on the injected routing against the oracle, and
# against the same layer with whole tiles only (MOE_GEMM_HALF=0).
REMAINDER = [(2300, 256, 2, 512, [1025, 1038, 1280, 1257], "swiglu"),
             (2000, 384, 3, 256, [1025, 1038, 1280, 1257, 0, 1400], "swiglu"),
             (2300, 256, 2, 512, [1025, 1038, 1280, 1257], "silu"),
             (1200, 512, 2, 384, [1025, 100, 1027, 248], "swiglu")]


@pytest.mark.parametrize("T,d,K,h,counts,expert", REMAINDER,
                         ids=lambda v: str(v) if not isinstance(v, list) else "-".join(map(str, v)))
def test_partial_tiles_half_height(T, d, K, h, counts, expert, monkeypatch):
    E = len(counts)
    s = I.Shape(T, d, E, K, h, expert)
    inp = I.make_layer_inputs(s, seed=8)
    ids = _ids_with_counts(T, K, counts, seed=8)
    w = I.random_weights(T, K, seed=8)
    dv = to_dev(inp)
    from token_dispatch_grouped_gb300.layer import Routing
    out = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("MOE_GEMM_HALF", mode)
        L = _layer(s)
        r = Routing(None, ids.cuda(), w.cuda())
        dp = L.dispatch(r.ids)
        y, H = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp)
        g = L.backward(dv["dO"], dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], r, dp, H)
        L.check_error()
        out[mode] = (y, H, g)
    monkeypatch.delenv("MOE_GEMM_HALF")
    assert np.array_equal(np.diff(cpu(dp.offsets)), np.array(counts))
    y, H, g = out["1"]
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids.numpy(), w.numpy(), expert)
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"],
                         ids.numpy(), w.numpy(), f, expert)
    for name, got, ref in (("H", H, f["H"]), ("y", y, f["y"]), ("dS", g["dS"], b["dS"]),
                           ("dx", g["dx"], b["dx"]), ("dWg", g["dWg"], b["dWg"])) + \
            tuple((k, g[k], b[k]) for k in _wgrad_keys(s)):
        assert rel_fro(cpu(got), ref) <= TOL_BF16, name
        if name != "dS":
            assert rel_rows(cpu(got), ref) <= TOL_ROW, name
    # half and whole tiles sum the same products per row (the dS partials in
    # another grouping)
    y0, H0, g0 = out["0"]
    assert rel_fro(cpu(y), cpu(y0).astype(np.float64)) <= 1e-3
    assert rel_fro(cpu(H), cpu(H0).astype(np.float64)) <= 1e-3
    for k in ("dx", "dS") + _wgrad_keys(s):
        assert rel_fro(cpu(g[k]), cpu(g0[k]).astype(np.float64)) <= 1e-3, k


# Column passes: small layers split the down projection and dX into two column
# passes, larger ones into four. Forcing four passes on a small layer covers that
# path too; both runs sum every output element over the same k order, so they
# agree far inside the layer tolerance.
@pytest.mark.parametrize("s", [I.Shape(1100, 512, 8, 2, 256), I.Shape(1100, 512, 8, 2, 768, "relu")],
                         ids=_sid)
def test_column_pass_count_is_bit_identical(s, monkeypatch):
    inp = I.make_layer_inputs(s, seed=4)
    dv = to_dev(inp)
    L = _layer(s)
    outs = []
    for passes in ("2", "4"):
        monkeypatch.setenv("MOE_COLUMN_PASSES", passes)
        r, dp, y, H, g = L.step(dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], dv["dO"])
        L.check_error()
        outs.append((y, g["dx"], g["dS"], g["dWg"]))
    monkeypatch.delenv("MOE_COLUMN_PASSES")
    for a, b in zip(*outs):
        assert rel_fro(cpu(b), cpu(a).astype(np.float64)) <= 1e-3
    ids, w = cpu(r.ids), cpu(r.w)
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w, s.expert)
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ids, w, f,
                         s.expert)
    for (y, dx, _, _) in outs:
        assert rel_fro(cpu(y), f["y"]) <= TOL_BF16
        assert rel_fro(cpu(dx), b["dx"]) <= TOL_BF16


# Router weight gradient on the tensor cores (the library takes it once x exceeds
# 64 MiB): forced on small shapes -- one token chunk and several, E = K, K = 1 (dz = 0),
# CTA pairs, E = 160 (a partial second N tile) -- against the oracle and against the
# gathered per-expert path, which sums the same products in another order.
DWG = [I.WORKLOADS["tiny"], I.Shape(300, 256, 6, 3, 384), I.Shape(129, 384, 8, 8, 128),
       I.Shape(1500, 128, 16, 1, 256), I.Shape(2100, 512, 4, 2, 512),
       I.Shape(700, 256, 160, 6, 256)]


@pytest.mark.parametrize("s", DWG, ids=_sid)
def test_router_dwg_tensor_core_path(s, monkeypatch):
    inp = I.make_layer_inputs(s, seed=6)
    dv = to_dev(inp)
    out = {}
    for path in ("gather", "mma"):
        monkeypatch.setenv("MOE_ROUTER_DWG", path)
        L = _layer(s)  # the backward workspace follows the path
        r, dp, y, H, g = L.step(dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], dv["dO"])
        L.check_error()
        out[path] = (r, g)
    monkeypatch.delenv("MOE_ROUTER_DWG")
    r, g = out["mma"]
    dwg = cpu(g["dWg"])
    if s.K == 1:
        assert np.all(dwg == 0.0)
        return
    ids, w = cpu(r.ids), cpu(r.w)
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w, s.expert)
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ids, w, f,
                         s.expert)
    assert rel_fro(dwg, b["dWg"]) <= TOL_BF16
    assert rel_fro(dwg, cpu(out["gather"][1]["dWg"]).astype(np.float64)) <= 1e-4
    assert np.abs(dwg.sum(axis=0)).max() <= 1e-3 * np.abs(dwg).max()  # sum_k dz_k = 0


# Slot-wise forward (combine fused into the down projection): ragged tiles, K = 1
# (no accumulator), K = E = 8, CTA-pair shapes and a non-gated expert.
SLOTWISE = [I.Shape(300, 256, 6, 3, 512), I.Shape(1500, 128, 16, 1, 256),
            I.Shape(129, 384, 8, 8, 128), I.Shape(2100, 512, 4, 2, 512),
            I.Shape(1100, 512, 8, 2, 768, "relu")]


@pytest.mark.parametrize("s", SLOTWISE, ids=_sid)
def test_forward_slotwise_parity(s):
    inp = I.make_layer_inputs(s, seed=5)
    dv = to_dev(inp)
    L = _layer(s)
    r = L.route(dv["x"], dv["Wg"])
    dp = L.dispatch(r.ids)
    y = torch.full((s.T, s.d), float("nan"), dtype=torch.bfloat16, device="cuda")  # poison
    y, H = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp, y=y, combine="slotwise")
    y_c, H_c = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp, combine="chunked")
    y_again, _ = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp, combine="slotwise")
    L.check_error()
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], cpu(r.ids), cpu(r.w), s.expert)
    assert not np.isnan(cpu(y)).any()
    assert rel_fro(cpu(y), f["y"]) <= TOL_BF16
    assert torch.equal(H, H_c)                     # the up projection is shared
    assert rel_fro(cpu(y), cpu(y_c)) <= TOL_BF16   # same sum, one rounding fewer
    assert torch.equal(y, y_again)                 # fixed order: bit-reproducible


# Router shapes that exercise the cluster split of the reduction over d (2, 4 and
# 8 CTAs), every padded expert width (8 .. 256), E not a multiple of 8, a bias,
# and long reductions (d = 2048, 4096) at the expert counts of the workloads.
# Both paths: the tensor-core router (E <= 128, three bf16 parts of W_g) and the
# FFMA router (forced; the only one above E = 128).
ROUTER = [(256, 2048, 8, 2), (1000, 1024, 16, 4), (300, 512, 64, 6), (500, 1024, 128, 8),
          (200, 2048, 256, 8), (5000, 256, 5, 3), (777, 384, 40, 5), (4096, 4096, 8, 2),
          (1024, 4096, 16, 4), (2000, 2048, 64, 6), (3000, 2048, 128, 8), (600, 4096, 128, 8)]


@pytest.mark.parametrize("T,d,E,K", ROUTER, ids=lambda v: str(v))
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("path", ["default", "ffma"])
def test_router_shapes(T, d, E, K, with_bias, path, monkeypatch):
    from token_dispatch_grouped_gb300.layer import MoELayer
    if path == "ffma":
        monkeypatch.setenv("MOE_ROUTER", "ffma")
    s = I.Shape(T, d, E, K, 256)
    inp = I.make_layer_inputs(s, seed=3, parts=("x", "Wg"))
    bias = None
    if with_bias:
        g = torch.Generator().manual_seed(11)
        bias = (torch.rand(E, generator=g) - 0.5).float()
    L = MoELayer(T, d, E, K, 256)
    r = L.route(inp["x"].cuda(), inp["Wg"].cuda(), None if bias is None else bias.cuda())
    L.check_error()
    _check_route(r.logits, r.ids, r.w, inp["x"], inp["Wg"], K, bias)


@pytest.mark.parametrize("expert", ["swiglu", "relu"])
def test_injected_routing_skewed_and_empty_experts(expert):
    s = I.Shape(700, 256, 16, 4, 256, expert)
    inp = I.make_layer_inputs(s, seed=2)
    ids = I.random_ids(s.T, 12, s.K, seed=5, skew=1.5)      # experts 12..15 get no token
    w = I.random_weights(s.T, s.K, seed=5)
    dv = to_dev(inp)
    L = _layer(s)
    from token_dispatch_grouped_gb300.layer import Routing
    r = Routing(None, ids.cuda(), w.cuda())
    dp = L.dispatch(r.ids)
    y, H = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp)
    grads = L.alloc_grads()
    for t in grads.values():                                 # poison: every element must be written
        if t is not None:
            t.fill_(float("nan"))
    L.backward(dv["dO"], dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], r, dp, H, grads)
    L.check_error()
    _check_dispatch(r.ids, dp, s.E)
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], ids, w, expert)
    b = O.layer_backward(inp["dO"], inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], ids, w, f,
                         expert)
    assert rel_fro(cpu(y), f["y"]) <= TOL_BF16
    for k in ("dx", "dS", "dWg") + _wgrad_keys(s):
        assert not np.isnan(cpu(grads[k])).any(), k
        assert rel_fro(cpu(grads[k]), b[k]) <= TOL_BF16, k
    for k in _wgrad_keys(s):
        assert np.all(cpu(grads[k])[12:] == 0.0)


def test_fig2_worked_example_on_gpu():
    with open(os.path.join(GOLD, "moeblaze_fig2.json")) as f:
        g = json.load(f)
    s = I.Shape(5, 128, g["E"], g["K"], 128)
    L = _layer(s)
    ids = torch.tensor(g["assignments"], dtype=torch.int32, device="cuda")
    dp = L.dispatch(ids)
    L.check_error()
    assert cpu(dp.eti).tolist() == g["expert_token_indices"]
    assert cpu(dp.offsets).tolist() == g["expert_token_offsets"]
    assert cpu(dp.tim)[:2].tolist() == g["token_index_map_token0"]


@pytest.mark.parametrize("case", ["all_to_one", "two_experts", "ragged_blocks", "skew"])
def test_dispatch_adversarial(case):
    if case == "all_to_one":
        T, E, K = 1000, 8, 1
        ids = torch.full((T, K), 3, dtype=torch.int32)
    elif case == "two_experts":
        T, E, K = 777, 64, 2
        ids = torch.tensor([[5, 60]] * T, dtype=torch.int32)
    elif case == "ragged_blocks":
        T, E, K = 513, 256, 8
        ids = I.random_ids(T, E, K, seed=9)
    else:
        T, E, K = 5000, 128, 6
        ids = I.random_ids(T, E, K, seed=3, skew=2.0)
    s = I.Shape(T, 128, E, K, 128)
    L = _layer(s)
    dp = L.dispatch(ids.cuda())
    L.check_error()
    _check_dispatch(ids, dp, E)


# The single-CTA build (ids staged in shared memory; the default for E <= 16 and
# T*K <= 16384) and the three-launch build must give the same bit-exact index,
# both forced on every case. Cases at the default threshold (T*K = 16384 with
# E = 16) and just past it, at the shared-memory limit of a forced single CTA
# (T*K = 32768 with E = 256) and past T*K = 32768, token counts that leave warps
# partly or wholly idle, all tokens on one expert, and a Zipf-skewed routing
# with idle experts.
SINGLE = [(8192, 16, 2, "random"), (5462, 8, 3, "random"), (4096, 256, 8, "random"),
          (16384, 8, 2, "random"), (32769, 4, 1, "random"), (31, 8, 2, "random"),
          (1, 4, 4, "random"), (1057, 64, 6, "skew"), (8192, 8, 4, "all_to_one"),
          (4096, 8, 2, "random")]


@pytest.mark.parametrize("T,E,K,kind", SINGLE, ids=lambda v: str(v))
def test_dispatch_single_cta_and_block_builds_agree(T, E, K, kind, monkeypatch):
    if kind == "all_to_one":
        ids = torch.stack([torch.full((T,), 3, dtype=torch.int32)] +
                          [torch.full((T,), 4 + k, dtype=torch.int32) for k in range(K - 1)], 1)
    elif kind == "skew":
        ids = I.random_ids(T, E, K, seed=21, skew=1.8)
    else:
        ids = I.random_ids(T, E, K, seed=T + E)
    s = I.Shape(T, 128, E, K, 128)
    L = _layer(s)
    outs = {}
    for mode in ("single", "blocks"):
        monkeypatch.setenv("MOE_DISPATCH", mode)
        dp = L.dispatch(ids.cuda())
        L.check_error()
        outs[mode] = [t.clone() for t in (dp.eti, dp.offsets, dp.tim)]
    monkeypatch.delenv("MOE_DISPATCH")
    for a, b in zip(outs["single"], outs["blocks"]):
        assert torch.equal(a, b)
    _check_dispatch(ids, dp, E)


@pytest.mark.parametrize("mode", ["single", "blocks"])
def test_bad_expert_ids_both_dispatch_builds(mode, monkeypatch):
    from token_dispatch_grouped_gb300 import binding as B
    monkeypatch.setenv("MOE_DISPATCH", mode)
    s = I.Shape(300, 128, 8, 3, 128)
    L = _layer(s)
    B.moe_get_error()
    ids = I.random_ids(300, 8, 3, seed=2)
    ids[299, 2] = -1                                  # out of range, last token
    L.dispatch(ids.cuda())
    assert B.moe_get_error() == B.MOE_ERR_BAD_EXPERT_ID
    ids = I.random_ids(300, 8, 3, seed=2)
    ids[0, 2] = ids[0, 1]                             # repeated within the first token
    L.dispatch(ids.cuda())
    assert B.moe_get_error() == B.MOE_ERR_BAD_EXPERT_ID
    assert B.moe_get_error() == B.MOE_OK


@pytest.mark.parametrize("T,E,K,skew", [(1000, 8, 2, 0.0), (3000, 64, 6, 1.2),
                                        (513, 128, 8, 0.0), (20000, 16, 4, 2.0)])
def test_sort_dispatch_baseline_matches_oracle_and_ours(T, E, K, skew):
    """The sort-based baseline of the dispatch ablation computes the same index."""
    import bench
    ids = I.random_ids_gumbel(T, E, K, seed=7, skew=skew)
    eti, off, tim, _ = O.build_dispatch(ids.numpy(), E)
    b_eti, b_off, b_tim = bench.sort_dispatch(ids.cuda(), E)
    assert np.array_equal(cpu(b_eti), eti)
    assert np.array_equal(cpu(b_off), off)
    assert np.array_equal(cpu(b_tim), tim)
    L = _layer(I.Shape(T, 128, E, K, 128))
    dp = L.dispatch(ids.cuda())
    L.check_error()
    assert torch.equal(dp.eti, b_eti) and torch.equal(dp.offsets, b_off)
    assert torch.equal(dp.tim, b_tim)


def test_bad_expert_ids_raise_device_error():
    from token_dispatch_grouped_gb300 import binding as B
    s = I.Shape(64, 128, 8, 2, 128)
    L = _layer(s)
    B.moe_get_error()
    ids = I.random_ids(64, 8, 2, seed=1)
    ids[10, 1] = 8                                   # out of range
    L.dispatch(ids.cuda())
    assert B.moe_get_error() == B.MOE_ERR_BAD_EXPERT_ID
    ids = I.random_ids(64, 8, 2, seed=1)
    ids[3, 1] = ids[3, 0]                            # repeated within a token
    L.dispatch(ids.cuda())
    assert B.moe_get_error() == B.MOE_ERR_BAD_EXPERT_ID
    assert B.moe_get_error() == B.MOE_OK             # the word was cleared


def test_host_checks_reject_bad_calls():
    from token_dispatch_grouped_gb300 import binding as B
    s = B.shape(64, 128, 8, 2, 128)
    ids = torch.zeros(64, 2, dtype=torch.int32, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty(128, dtype=torch.int32, device="cuda")
    rc = B.moe_build_dispatch(s, ids, out, out, out, small, check=False)
    assert rc == B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert B.moe_workspace_size(B.shape(64, 100, 8, 2, 128), 2) == 0   # d % 128 != 0
    x = torch.empty(64 * 128 + 1, dtype=torch.bfloat16, device="cuda")[1:]
    Wg = torch.empty(8, 128, device="cuda")
    w = torch.empty(64, 2, device="cuda")
    assert B.moe_route(s, x, Wg, None, None, ids, w, check=False) == B.MOE_ERR_MISALIGNED


def test_determinism_bitwise():
    s = I.Shape(1200, 256, 8, 2, 512)
    inp = to_dev(I.make_layer_inputs(s, seed=4))
    L = _layer(s)
    outs = []
    for _ in range(2):
        r, dp, y, H, g = L.step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"])
        outs.append([t.clone() for t in (r.ids, r.w, dp.eti, dp.tim, y, H, *g.values())])
    L.check_error()
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ------------------------------------------------------------------ full workloads
def _full(name):
    s = I.WORKLOADS[name]
    inp = I.make_layer_inputs(s, seed=0, with_bias=(name == "skew"))
    if name == "skew":
        assert inp["bias"] is not None
    dv = to_dev(inp)
    L = _layer(s)
    bias = dv["bias"]
    r = L.route(dv["x"], dv["Wg"], bias)
    dp = L.dispatch(r.ids)
    y, H = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp)
    g = L.backward(dv["dO"], dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], r, dp, H)
    L.check_error()
    return s, inp, r, dp, y, H, g


def _stratified_rows(offsets, blk=128, all_blocks_max=16):
    """Expert-sorted rows compared at full size: for every non-empty expert, the
    first and the last row of each of its 128-row blocks (a single-CTA M tile;
    a CTA-pair tile is two of them), or of its first, middle and last block
    when it has more than 16 blocks. Partial last blocks are included."""
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        nb = (hi - lo + blk - 1) // blk
        blocks = range(nb) if nb <= all_blocks_max else sorted({0, nb // 2, nb - 1})
        for b in blocks:
            r0 = lo + b * blk
            rows += [r0, min(hi, r0 + blk) - 1]
    return np.unique(np.asarray(rows, dtype=np.int64))


def _units_per_n_tile(h, bn=256):
    """One hidden unit in every bn-wide N tile of the weight-gradient GEMMs (the
    same index serves the dW1 and the dW3 halves), at a position that moves
    from tile to tile."""
    return np.array([n * bn + (97 * n + 31) % min(bn, h - n * bn) for n in range((h + bn - 1) // bn)])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral", "fine", "skew", "long", "moeblaze_conf7",
                                  "moeblaze_conf4"])
def test_full_workload_sampled(name):
    s, inp, r, dp, y, H, g = _full(name)
    bias = inp["bias"]
    ids, w = cpu(r.ids), cpu(r.w)
    _check_dispatch(r.ids, dp, s.E)
    offsets = cpu(dp.offsets)
    counts = np.diff(offsets)
    if name == "skew":
        assert (counts == 0).sum() >= 4
    eti = cpu(dp.eti)
    rows = _stratified_rows(offsets)
    rows = np.union1d(rows, np.arange(s.TK - 4, s.TK))     # largest H offsets
    toks = np.union1d(eti[rows], [0, s.T - 1])
    _check_route(r.logits, r.ids, r.w, inp["x"], inp["Wg"], s.K, bias, rows=toks)
    ys, dSs, dxs = O.tokens_forward_backward_batched(toks, inp["x"], inp["dO"], inp["Wg"],
                                                     inp["W1"], inp["W3"], inp["W2"], ids, w,
                                                     s.expert)
    assert rel_fro(cpu(y)[toks], ys) <= TOL_BF16
    assert rel_rows(cpu(y)[toks], ys) <= TOL_ROW
    if name in ("mixtral", "skew"):  # slot-wise forward at full size (K = 2 and K = 8)
        L = _layer(s)
        dv = to_dev(inp)
        y_s, _ = L.forward(dv["x"], dv["W1"], dv["W3"], dv["W2"], r, dp, combine="slotwise")
        L.check_error()
        assert rel_fro(cpu(y_s)[toks], ys) <= TOL_BF16
        assert rel_rows(cpu(y_s)[toks], ys) <= TOL_ROW
    assert rel_fro(cpu(g["dS"])[toks], dSs) <= TOL_BF16
    assert rel_fro(cpu(g["dx"])[toks], dxs) <= TOL_BF16
    assert rel_rows(cpu(g["dx"])[toks], dxs) <= TOL_ROW
    # weight gradients: one hidden unit per 256-wide N tile (both halves of dW1/dW3)
    # of the largest and of the smallest non-empty expert
    busy = np.nonzero(counts > 0)[0]
    js = _units_per_n_tile(s.h)
    for e in sorted({int(busy[np.argmax(counts[busy])]), int(busy[np.argmin(counts[busy])])}):
        g1, g3, g2 = O.hidden_units_grads(e, js, inp["x"], inp["dO"], inp["W1"], inp["W3"],
                                          inp["W2"], ids, w, s.expert)
        pairs = [("dW1", cpu(g["dW1"][e])[js], g1), ("dW2", cpu(g["dW2"][e])[:, js].T, g2.T)]
        if s.gated:
            pairs.append(("dW3", cpu(g["dW3"][e])[js], g3))
        for k, got, ref in pairs:
            assert rel_fro(got, ref) <= TOL_BF16, (k, e)
            assert rel_rows(got, ref) <= TOL_ROW, (k, e)
    # properties at any size: dW_g rows sum to zero over experts (sum_k dz_k = 0),
    # empty experts have exact-zero weight gradients, outputs are finite
    dWg = cpu(g["dWg"])
    assert np.abs(dWg.sum(axis=0)).max() <= 1e-3 * max(1e-30, np.abs(dWg).max())
    for e in np.nonzero(counts == 0)[0]:
        assert not cpu(g["dW1"][e]).any() and not cpu(g["dW2"][e]).any()
    for t in (y, g["dx"]):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("s", [I.Shape(2100, 512, 4, 2, 512), I.Shape(1500, 128, 16, 1, 256)],
                         ids=_sid)
def test_programmatic_launch_modes_are_bit_identical(s, monkeypatch):
    """Programmatic dependent launch only overlaps launch latency: with every
    kernel launched that way (MOE_PDL=1), none (0), the small kernels only
    (small) or the default (GEMMs only), the layer's outputs are the same bits."""
    inp = to_dev(I.make_layer_inputs(s, seed=12))
    L = _layer(s)
    outs = {}
    for mode in (None, "1", "0", "small"):
        if mode is None:
            monkeypatch.delenv("MOE_PDL", raising=False)
        else:
            monkeypatch.setenv("MOE_PDL", mode)
        r, dp, y, H, g = L.step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"])
        L.check_error()
        outs[mode] = [t.clone() for t in (r.ids, r.w, dp.eti, dp.tim, y, H, *g.values())
                      if t is not None]
    monkeypatch.delenv("MOE_PDL", raising=False)
    for mode in ("1", "0", "small"):
        for a, b in zip(outs[None], outs[mode]):
            assert torch.equal(a, b), mode


# Tile order of the row-tiled GEMMs: every output element is computed by one tile
# with a fixed reduction order, so grouping an expert's M tiles (MOE_GEMM_GROUP_MB)
# moves work between CTAs but must leave every bit of every output in place.
# 2100 tokens x K = 2 over 4 experts: 4-5 M tiles of 256 rows per expert; a 1 MiB
# budget groups them by 4 (d = 512: 256 KB of A per tile), 0 walks M fastest.
@pytest.mark.parametrize("s", [I.Shape(2100, 512, 4, 2, 512), I.Shape(2100, 512, 4, 2, 256, "silu")],
                         ids=_sid)
def test_row_tile_order_is_bit_identical(s, monkeypatch):
    inp = to_dev(I.make_layer_inputs(s, seed=13))
    L = _layer(s)
    outs = {}
    for mb in ("0", "1", "32"):
        monkeypatch.setenv("MOE_GEMM_GROUP_MB", mb)
        r, dp, y, H, g = L.step(inp["x"], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"])
        L.check_error()
        outs[mb] = [t.clone() for t in (y, H, *g.values()) if t is not None]
    monkeypatch.delenv("MOE_GEMM_GROUP_MB")
    for mb in ("1", "32"):
        for a, b in zip(outs["0"], outs[mb]):
            assert torch.equal(a, b), mb
