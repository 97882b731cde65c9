"""ctypes binding of libmoe_gb300.so (include/moe.h), argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch
tensors (device tensors for the compute calls) and passes their data pointers
and the current CUDA stream. No computation happens in Python, and there is no
fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_BAD_EXPERT_ID = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_MISALIGNED = 7
MOE_ERR_NO_DEVICE = 8
MOE_ERR_STATIC_SCRATCH_LIMIT = 9
MOE_NOALLOC_DISPATCH_MAX_ENTRIES = 1 << 20

MOE_WS_ROUTE, MOE_WS_DISPATCH, MOE_WS_FORWARD, MOE_WS_BACKWARD = 0, 1, 2, 3
MOE_WS_FORWARD_SLOTWISE = 4

MOE_EXPERT_SWIGLU, MOE_EXPERT_SILU, MOE_EXPERT_RELU = 0, 1, 2
EXPERT_CODES = {"swiglu": MOE_EXPERT_SWIGLU, "silu": MOE_EXPERT_SILU, "relu": MOE_EXPERT_RELU}


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("h", ctypes.c_int32), ("expert", ctypes.c_int32)]


class MoeKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32),
                ("total_ms", ctypes.c_double)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        extra = ""
        if code == MOE_ERR_CUDA:
            extra = f" [{LIB.moe_last_cuda_error().decode()}]"
        super().__init__(f"{where}: {status_string(code)} (status {code}){extra}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first with "
            "`python -m token_dispatch_grouped_gb300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I, L = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_longlong
    sig = {
        "moe_workspace_size": (S, [MoeShape, I]),
        "moe_chunk_tokens": (I, [MoeShape]),
        "moe_route": (I, [MoeShape, P, P, P, P, P, P, P, S, P]),
        "moe_build_dispatch": (I, [MoeShape, P, P, P, P, P, S, P]),
        "moe_build_dispatch_noalloc": (I, [MoeShape, P, P, P, P, P]),
        "moe_forward": (I, [MoeShape, P, P, P, P, P, P, P, P, P, P, P, P, S, P]),
        "moe_forward_slotwise": (I, [MoeShape, P, P, P, P, P, P, P, P, P, P, P, P, S, P]),
        "moe_backward": (I, [MoeShape] + [P] * 19 + [S, P]),
        "moe_rows_capacity": (S, [MoeShape, I]),
        "moe_token_rounding_workspace_size": (S, [MoeShape, I]),
        "moe_token_rounding": (I, [MoeShape, I] + [P] * 11 + [S, P]),
        "moe_workspace_size_rows": (S, [MoeShape, ctypes.c_int32, I]),
        "moe_forward_rows": (I, [MoeShape, ctypes.c_int32] + [P] * 13 + [S, P]),
        "moe_backward_rows": (I, [MoeShape, ctypes.c_int32] + [P] * 20 + [S, P]),
        "moe_get_error": (I, [P]),
        "moe_selftest_bounded_wait": (I, [ctypes.c_uint64, P]),
        "moe_status_string": (ctypes.c_char_p, [I]),
        "moe_last_cuda_error": (ctypes.c_char_p, []),
        "moe_launch_count": (L, []),
        "moe_timing_enable": (I, [I]),
        "moe_timing_collect": (I, [ctypes.POINTER(MoeKernelTime), I]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


LIB = _load()


def shape(T: int, d: int, E: int, K: int, h: int, expert: str | int = "swiglu") -> MoeShape:
    code = EXPERT_CODES[expert] if isinstance(expert, str) else int(expert)
    return MoeShape(T, d, E, K, h, code)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def status_string(code: int) -> str:
    return LIB.moe_status_string(code).decode()


def moe_workspace_size(s: MoeShape, which: int) -> int:
    return int(LIB.moe_workspace_size(s, which))


def moe_chunk_tokens(s: MoeShape) -> int:
    return int(LIB.moe_chunk_tokens(s))


def moe_route(s, x, Wg, bias, logits, topk_ids, topk_w, ws=None, stream=None, check=True):
    rc = LIB.moe_route(s, _ptr(x), _ptr(Wg), _ptr(bias), _ptr(logits), _ptr(topk_ids),
                       _ptr(topk_w), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                       _stream(stream))
    if check:
        _check(rc, "moe_route")
    return rc


def moe_build_dispatch(s, topk_ids, eti, offsets, tim, ws, stream=None, check=True):
    rc = LIB.moe_build_dispatch(s, _ptr(topk_ids), _ptr(eti), _ptr(offsets), _ptr(tim), _ptr(ws),
                                0 if ws is None else ws.numel() * ws.element_size(),
                                _stream(stream))
    if check:
        _check(rc, "moe_build_dispatch")
    return rc


def moe_build_dispatch_noalloc(s, topk_ids, eti, offsets, tim, stream=None, check=True):
    """Same result as moe_build_dispatch without a workspace: for callers that
    cannot allocate device memory (the scratch is a static device array inside
    the library; calls that overlap on the GPU must not share it)."""
    rc = LIB.moe_build_dispatch_noalloc(s, _ptr(topk_ids), _ptr(eti), _ptr(offsets), _ptr(tim),
                                        _stream(stream))
    if check:
        _check(rc, "moe_build_dispatch_noalloc")
    return rc


def moe_forward(s, x, W1, W3, W2, topk_ids, topk_w, eti, offsets, tim, y, H_saved, ws,
                stream=None, check=True):
    rc = LIB.moe_forward(s, _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(topk_ids), _ptr(topk_w),
                         _ptr(eti), _ptr(offsets), _ptr(tim), _ptr(y), _ptr(H_saved), _ptr(ws),
                         0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(rc, "moe_forward")
    return rc


def moe_forward_slotwise(s, x, W1, W3, W2, topk_ids, topk_w, eti, offsets, tim, y, H_saved, ws,
                         stream=None, check=True):
    """moe_forward with the combine fused into the down projection, slot by slot."""
    rc = LIB.moe_forward_slotwise(s, _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(topk_ids),
                                  _ptr(topk_w), _ptr(eti), _ptr(offsets), _ptr(tim), _ptr(y),
                                  _ptr(H_saved), _ptr(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream(stream))
    if check:
        _check(rc, "moe_forward_slotwise")
    return rc


def moe_rows_capacity(s: MoeShape, m_tile: int) -> int:
    return int(LIB.moe_rows_capacity(s, m_tile))


def moe_token_rounding_workspace_size(s: MoeShape, m_tile: int) -> int:
    return int(LIB.moe_token_rounding_workspace_size(s, m_tile))


def moe_workspace_size_rows(s: MoeShape, rows_cap: int, which: int) -> int:
    return int(LIB.moe_workspace_size_rows(s, rows_cap, which))


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def moe_token_rounding(s, m_tile, logits, topk_ids, tc_eti, tc_offsets, eti, offsets, w_row,
                       tok_off, tok_exp, tok_rows, ws, stream=None, check=True):
    rc = LIB.moe_token_rounding(s, m_tile, _ptr(logits), _ptr(topk_ids), _ptr(tc_eti),
                                _ptr(tc_offsets), _ptr(eti), _ptr(offsets), _ptr(w_row),
                                _ptr(tok_off), _ptr(tok_exp), _ptr(tok_rows), _ptr(ws),
                                _nbytes(ws), _stream(stream))
    if check:
        _check(rc, "moe_token_rounding")
    return rc


def moe_forward_rows(s, rows_cap, x, W1, W3, W2, eti, offsets, w_row, tok_off, tok_exp, tok_rows,
                     y, H_saved, ws, stream=None, check=True):
    rc = LIB.moe_forward_rows(s, rows_cap, _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(eti),
                              _ptr(offsets), _ptr(w_row), _ptr(tok_off), _ptr(tok_exp),
                              _ptr(tok_rows), _ptr(y), _ptr(H_saved), _ptr(ws), _nbytes(ws),
                              _stream(stream))
    if check:
        _check(rc, "moe_forward_rows")
    return rc


def moe_backward_rows(s, rows_cap, dy, x, Wg, W1, W3, W2, eti, offsets, w_row, tok_off, tok_exp,
                      tok_rows, H_saved, dx, dWg, dW1, dW3, dW2, dS_row, ws, stream=None,
                      check=True):
    rc = LIB.moe_backward_rows(s, rows_cap, _ptr(dy), _ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3),
                               _ptr(W2), _ptr(eti), _ptr(offsets), _ptr(w_row), _ptr(tok_off),
                               _ptr(tok_exp), _ptr(tok_rows), _ptr(H_saved), _ptr(dx),
                               _ptr(dWg), _ptr(dW1), _ptr(dW3), _ptr(dW2), _ptr(dS_row),
                               _ptr(ws), _nbytes(ws), _stream(stream))
    if check:
        _check(rc, "moe_backward_rows")
    return rc


def moe_backward(s, dy, x, Wg, W1, W3, W2, topk_ids, topk_w, eti, offsets, tim, H_saved,
                 dx, dWg, dW1, dW3, dW2, dS, ws, stream=None, check=True):
    rc = LIB.moe_backward(s, _ptr(dy), _ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2),
                          _ptr(topk_ids), _ptr(topk_w), _ptr(eti), _ptr(offsets), _ptr(tim),
                          _ptr(H_saved), _ptr(dx), _ptr(dWg), _ptr(dW1), _ptr(dW3), _ptr(dW2),
                          _ptr(dS), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                          _stream(stream))
    if check:
        _check(rc, "moe_backward")
    return rc


def moe_get_error(stream=None) -> int:
    return int(LIB.moe_get_error(_stream(stream)))


def moe_selftest_bounded_wait(limit_ns: int, stream=None) -> int:
    """Launches the failure-path self-test (a wait that runs out); returns the
    launch status. moe_get_error() afterwards reports MOE_ERR_TIMEOUT."""
    return int(LIB.moe_selftest_bounded_wait(int(limit_ns), _stream(stream)))


def moe_launch_count() -> int:
    return int(LIB.moe_launch_count())


def moe_timing_enable(on: bool) -> None:
    LIB.moe_timing_enable(1 if on else 0)


def moe_timing_collect() -> dict:
    buf = (MoeKernelTime * 64)()
    n = LIB.moe_timing_collect(buf, 64)
    if n < 0:
        raise MoeError(-n, "moe_timing_collect")
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms))
            for i in range(min(n, 64))}
