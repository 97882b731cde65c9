"""The C-ABI library builds, loads and exports every symbol that include/*.h
declares; its pure host functions behave as documented. No compute calls."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from token_dispatch_grouped_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "moe_route" in names and "moe_backward" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_host_functions():
    from token_dispatch_grouped_gb300 import binding as B
    s = B.shape(4096, 4096, 8, 2, 14336)
    assert B.moe_chunk_tokens(s) == 2048       # T*K*d = 32 MiB: two token chunks
    assert B.moe_chunk_tokens(B.shape(32768, 2048, 128, 8, 768)) == 8192  # 512 MiB: four
    assert B.moe_chunk_tokens(B.shape(8192, 2048, 8, 4, 8192)) == 4096    # exactly 64 MiB: two
    assert B.moe_chunk_tokens(B.shape(512, 256, 8, 2, 256)) == 512        # T < 1024: one
    fwd = B.moe_workspace_size(s, B.MOE_WS_FORWARD)
    # the forward workspace holds the SwiGLU output [TK, h] and one Y chunk:
    # two column passes here (the half-width chunk is 32 MiB), so half of the
    # T*K*d routed buffer, which itself is never allocated
    TK = 4096 * 2
    assert fwd >= TK * 14336 * 2 + TK * 2048 * 2
    assert fwd < TK * 14336 * 2 + TK * 2048 * 2 + 2**20
    # larger layers keep the chunk at a quarter of T*K*d
    big = B.shape(65536, 4096, 8, 2, 14336)
    assert B.moe_workspace_size(big, B.MOE_WS_FORWARD) < 131072 * 14336 * 2 + 131072 * 1024 * 2 + 2**20
    # route: the three bf16 parts of W_g, 3 x max(16, E padded) rows of d, for the
    # tensor-core router (E <= 128); none for the FFMA router (E > 128)
    assert B.moe_workspace_size(s, B.MOE_WS_ROUTE) == 3 * 16 * 4096 * 2
    assert B.moe_workspace_size(B.shape(512, 2048, 100, 8, 768), B.MOE_WS_ROUTE) == \
        3 * 128 * 2048 * 2
    assert B.moe_workspace_size(B.shape(512, 2048, 200, 8, 768), B.MOE_WS_ROUTE) == 0
    # slot-wise forward: no chunk buffer, an fp32 [T, d] accumulator instead
    slot = B.moe_workspace_size(s, B.MOE_WS_FORWARD_SLOTWISE)
    assert slot >= TK * 14336 * 2 + 4096 * 4096 * 4
    assert slot < TK * 14336 * 2 + 4096 * 4096 * 4 + 8 * 2**20
    for bad in (B.shape(0, 128, 8, 2, 128), B.shape(8, 100, 8, 2, 128), B.shape(8, 128, 4, 5, 128),
                B.shape(8, 128, 300, 2, 128), B.shape(8, 128, 16, 9, 128)):
        assert B.moe_workspace_size(bad, B.MOE_WS_FORWARD) == 0
    assert B.status_string(B.MOE_ERR_BAD_EXPERT_ID).startswith("expert id")


def test_null_pointers_rejected_before_any_device_work():
    from token_dispatch_grouped_gb300 import binding as B
    s = B.shape(16, 128, 8, 2, 128)
    assert B.LIB.moe_route(s, None, None, None, None, None, None, None, 0, None) == \
        B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_build_dispatch(s, None, None, None, None, None, 0, None) == \
        B.MOE_ERR_INVALID_ARG
    bad = B.shape(16, 128, 8, 9, 128)
    assert B.LIB.moe_route(bad, None, None, None, None, None, None, None, 0, None) == \
        B.MOE_ERR_UNSUPPORTED_SHAPE
    # the failure-path self-test rejects a wait limit out of range before any launch
    assert B.LIB.moe_selftest_bounded_wait(0, None) == B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_selftest_bounded_wait(20_000_000_000, None) == B.MOE_ERR_INVALID_ARG


def test_oracle_is_not_imported_by_the_product():
    pkg = os.path.join(ROOT, "token_dispatch_grouped_gb300")
    for py in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        src = open(py).read()
        assert "oracle" not in re.findall(r"^\s*(?:from|import)\s+(\w+)", src, flags=re.M), py


def test_non_gated_expert_shapes():
    from token_dispatch_grouped_gb300 import binding as B
    T, d, E, K, h = 4096, 1024, 16, 4, 4096
    TK = T * K
    gated = B.moe_workspace_size(B.shape(T, d, E, K, h), B.MOE_WS_BACKWARD)
    for act in ("silu", "relu"):
        s = B.shape(T, d, E, K, h, act)
        assert s.expert == B.EXPERT_CODES[act]
        bwd = B.moe_workspace_size(s, B.MOE_WS_BACKWARD)
        # dH is [TK, h] instead of [TK, 2h]; the dX pass may also be planned differently
        assert 0 < bwd < gated
        assert bwd >= TK * h * 2 * 2           # dH and A' (bf16), each [TK, h]
        assert B.moe_workspace_size(s, B.MOE_WS_FORWARD) == \
            B.moe_workspace_size(B.shape(T, d, E, K, h), B.MOE_WS_FORWARD)
    # a non-gated up-projection tile is 256 columns wide
    assert B.moe_workspace_size(B.shape(T, d, E, K, 384, "silu"), B.MOE_WS_FORWARD) == 0
    assert B.moe_workspace_size(B.shape(T, d, E, K, 384), B.MOE_WS_FORWARD) > 0
    assert B.moe_workspace_size(B.shape(T, d, E, K, h, 3), B.MOE_WS_FORWARD) == 0


def test_gated_expert_needs_w3_before_any_device_work():
    from token_dispatch_grouped_gb300 import binding as B
    s = B.shape(16, 128, 8, 2, 256)
    fake = [256 * (i + 1) for i in range(19)]  # never dereferenced: rejected on the host
    # moe_forward pointers: x, W1, W3, W2, ids, w, eti, offsets, tim, y, H, ws
    args = [s, *fake[:2], None, *fake[3:12], 1 << 20, None]
    assert B.LIB.moe_forward(*args) == B.MOE_ERR_INVALID_ARG
    # moe_backward pointers: dy, x, Wg, W1, W3, W2, ids, w, eti, offsets, tim, H,
    # dx, dWg, dW1, dW3, dW2, dS, ws
    bw = [s, *fake[:4], None, *fake[5:19], 1 << 20, None]      # W3 missing
    assert B.LIB.moe_backward(*bw) == B.MOE_ERR_INVALID_ARG
    bw = [s, *fake[:15], None, *fake[16:19], 1 << 20, None]    # dW3 missing
    assert B.LIB.moe_backward(*bw) == B.MOE_ERR_INVALID_ARG


def test_row_routing_entry_points_host_checks():
    from token_dispatch_grouped_gb300 import binding as B
    T, d, E, K, h = 4096, 1024, 16, 4, 2048
    s = B.shape(T, d, E, K, h)
    cap = B.moe_rows_capacity(s, 128)
    assert cap == min(T * K + E * 127, T * E)
    assert B.moe_rows_capacity(s, 0) == 0
    assert B.moe_token_rounding_workspace_size(s, 128) >= 4 * T + 16 * E + 4 * cap
    fwd = B.moe_workspace_size_rows(s, cap, B.MOE_WS_FORWARD)
    bwd = B.moe_workspace_size_rows(s, cap, B.MOE_WS_BACKWARD)
    assert fwd >= cap * h * 2 and bwd >= cap * 2 * h * 2
    assert B.moe_workspace_size_rows(s, 0, B.MOE_WS_FORWARD) == 0
    # rejected on the host before any device work: nulls, bad tile, bad capacity
    nul = [None] * 11
    assert B.LIB.moe_token_rounding(s, 128, *nul, 0, None) == B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_token_rounding(s, 5000, *nul, 0, None) == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert B.LIB.moe_forward_rows(s, cap, *([None] * 13), 0, None) == B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_forward_rows(s, T * E + 1, *([None] * 13), 0, None) == \
        B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_backward_rows(s, cap, *([None] * 20), 0, None) == B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_forward_slotwise(s, *([None] * 12), 0, None) == B.MOE_ERR_INVALID_ARG


def test_workspace_follows_the_pass_and_router_gradient_rules(monkeypatch):
    """Column passes (two for small layers, four otherwise, forced by
    MOE_COLUMN_PASSES) and the router weight-gradient path (tensor cores once x
    exceeds 64 MiB, forced by MOE_ROUTER_DWG) size the workspaces as documented."""
    from token_dispatch_grouped_gb300 import binding as B
    s = B.shape(4096, 4096, 8, 2, 14336)      # Mixtral-shaped: x = 32 MiB
    TK = 4096 * 2
    A = TK * 14336 * 2                         # SwiGLU output [TK, h]
    two = B.moe_workspace_size(s, B.MOE_WS_FORWARD)
    monkeypatch.setenv("MOE_COLUMN_PASSES", "4")
    four = B.moe_workspace_size(s, B.MOE_WS_FORWARD)
    monkeypatch.delenv("MOE_COLUMN_PASSES")
    assert A + TK * 2048 * 2 <= two < A + TK * 2048 * 2 + 2**20    # half-width chunk
    assert A + TK * 1024 * 2 <= four < A + TK * 1024 * 2 + 2**20   # quarter-width chunk
    # router gradient: gathered path (P row parts per expert, P from the shape) below 64 MiB of x ...
    gather = B.moe_workspace_size(s, B.MOE_WS_BACKWARD)
    monkeypatch.setenv("MOE_ROUTER_DWG", "mma")
    mma = B.moe_workspace_size(s, B.MOE_WS_BACKWARD)
    monkeypatch.delenv("MOE_ROUTER_DWG")
    # ... the tensor-core path adds B = [dz_hi | dz_lo] [T, 128] bf16, the identity list
    # and fp32 chunk partials [chunks, d, 128] in place of [P, E, d] fp32 parts (P = 76 here)
    diff = mma - gather
    assert diff >= 4096 * 128 * 2 + 4096 * 4 + 4096 * 128 * 4 - 76 * 8 * 4096 * 4
    # skew-shaped (x = 128 MiB): the tensor-core path is the default
    k = B.shape(32768, 2048, 128, 8, 768)
    default = B.moe_workspace_size(k, B.MOE_WS_BACKWARD)
    monkeypatch.setenv("MOE_ROUTER_DWG", "mma")
    assert B.moe_workspace_size(k, B.MOE_WS_BACKWARD) == default
    monkeypatch.setenv("MOE_ROUTER_DWG", "gather")
    assert B.moe_workspace_size(k, B.MOE_WS_BACKWARD) != default
    monkeypatch.delenv("MOE_ROUTER_DWG")


def test_dispatch_entry_points_share_host_checks():
    """moe_build_dispatch and its allocation-free variant reject the same bad
    calls with the same codes, before any device work."""
    from token_dispatch_grouped_gb300 import binding as B
    bad_kind = B.shape(16, 128, 8, 2, 128, 7)            # no such expert kind
    assert B.LIB.moe_build_dispatch(bad_kind, None, None, None, None, None, 0, None) == \
        B.MOE_ERR_INVALID_ARG
    assert B.LIB.moe_build_dispatch_noalloc(bad_kind, None, None, None, None, None) == \
        B.MOE_ERR_INVALID_ARG
    too_many = B.shape(16, 128, 8, 9, 128)               # K > 8
    assert B.LIB.moe_build_dispatch(too_many, None, None, None, None, None, 0, None) == \
        B.MOE_ERR_UNSUPPORTED_SHAPE
    assert B.LIB.moe_build_dispatch_noalloc(too_many, None, None, None, None, None) == \
        B.MOE_ERR_UNSUPPORTED_SHAPE
    ok = B.shape(16, 128, 8, 2, 128)
    assert B.LIB.moe_build_dispatch_noalloc(ok, None, None, None, None, None) == \
        B.MOE_ERR_INVALID_ARG


def test_forward_buffer_never_holds_the_routed_buffer():
    """For every workload, the forward workspace beyond the [T*K, h] activation
    output (the down-projection chunk buffer and the segment tables) stays within
    half of the T*K*d bf16 routed buffer once T >= 1024 -- a quarter when that
    half exceeds 64 MiB -- so the routed buffer itself is never allocated."""
    from token_dispatch_grouped_gb300 import binding as B
    from token_dispatch_grouped_gb300 import inputs as I
    for name, s in I.WORKLOADS.items():
        if s.T < 1024:
            continue
        sh = B.shape(s.T, s.d, s.E, s.K, s.h, s.expert)
        TK = s.T * s.K
        routed = TK * s.d * 2
        extra = B.moe_workspace_size(sh, B.MOE_WS_FORWARD) - TK * s.h * 2
        bound = routed // 2 if routed // 2 <= 64 * 2**20 else routed // 4
        assert 0 < extra <= bound + 2**20, (name, extra, bound)
