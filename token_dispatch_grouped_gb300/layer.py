"""Buffer management around the C ABI: allocates outputs and workspaces with
torch on the device and calls the entry points in order. Argument marshalling
only; every step of the layer runs in the CUDA library."""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass
class Routing:
    logits: torch.Tensor | None
    ids: torch.Tensor
    w: torch.Tensor


@dataclass
class Dispatch:
    eti: torch.Tensor
    offsets: torch.Tensor
    tim: torch.Tensor


@dataclass
class RowRouting:
    """A routing given as rows (after token rounding)."""
    rows_cap: int
    eti: torch.Tensor
    offsets: torch.Tensor
    w_row: torch.Tensor
    tok_off: torch.Tensor
    tok_exp: torch.Tensor
    tok_rows: torch.Tensor


class MoELayer:
    """One dropless MoE layer of shape (T, d, E, K, h) on a CUDA device.

    expert: "swiglu" (W1, W3, W2), or the non-gated "silu" / "relu" (W1, W2;
    pass W3 = None). Workspaces are allocated once (the largest of the four
    calls) and reused."""

    def __init__(self, T: int, d: int, E: int, K: int, h: int, device="cuda",
                 expert: str = "swiglu"):
        self.s = B.shape(T, d, E, K, h, expert)
        self.T, self.d, self.E, self.K, self.h = T, d, E, K, h
        self.expert = expert
        self.gated = expert == "swiglu"
        self.hs = 2 * h if self.gated else h  # width of the saved pre-activation
        self.device = torch.device(device)
        sizes = [B.moe_workspace_size(self.s, w) for w in range(5)]
        if any(z == 0 for z in sizes[1:]):
            raise B.MoeError(B.MOE_ERR_UNSUPPORTED_SHAPE, "MoELayer")
        self.ws_bytes = max(sizes)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=self.device)

    # ------------------------------------------------------------------ calls
    def route(self, x, Wg, bias=None, want_logits=True) -> Routing:
        T, E, K = self.T, self.E, self.K
        logits = torch.empty(T, E, dtype=torch.float32, device=self.device) if want_logits else None
        ids = torch.empty(T, K, dtype=torch.int32, device=self.device)
        w = torch.empty(T, K, dtype=torch.float32, device=self.device)
        B.moe_route(self.s, x, Wg, bias, logits, ids, w, self.ws)
        return Routing(logits, ids, w)

    def dispatch(self, ids) -> Dispatch:
        TK = self.T * self.K
        eti = torch.empty(TK, dtype=torch.int32, device=self.device)
        off = torch.empty(self.E + 1, dtype=torch.int32, device=self.device)
        tim = torch.empty(TK, dtype=torch.int32, device=self.device)
        B.moe_build_dispatch(self.s, ids, eti, off, tim, self.ws)
        return Dispatch(eti, off, tim)

    def forward(self, x, W1, W3, W2, r: Routing, dp: Dispatch, y=None, H=None,
                combine: str = "chunked"):
        """combine: "chunked" (moe_forward) or "slotwise" (moe_forward_slotwise)."""
        if y is None:
            y = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=self.device)
        if H is None:
            H = torch.empty(self.T * self.K, self.hs, dtype=torch.bfloat16, device=self.device)
        fwd = B.moe_forward_slotwise if combine == "slotwise" else B.moe_forward
        fwd(self.s, x, W1, W3, W2, r.ids, r.w, dp.eti, dp.offsets, dp.tim, y, H, self.ws)
        return y, H

    def backward(self, dy, x, Wg, W1, W3, W2, r: Routing, dp: Dispatch, H, grads=None):
        if grads is None:
            grads = self.alloc_grads()
        B.moe_backward(self.s, dy, x, Wg, W1, W3, W2, r.ids, r.w, dp.eti, dp.offsets, dp.tim, H,
                       grads["dx"], grads["dWg"], grads["dW1"], grads["dW3"], grads["dW2"],
                       grads["dS"], self.ws)
        return grads

    def alloc_grads(self) -> dict:
        T, d, E, K, h, dev = self.T, self.d, self.E, self.K, self.h, self.device
        return dict(
            dx=torch.empty(T, d, dtype=torch.bfloat16, device=dev),
            dWg=torch.empty(E, d, dtype=torch.float32, device=dev),
            dW1=torch.empty(E, h, d, dtype=torch.bfloat16, device=dev),
            dW3=torch.empty(E, h, d, dtype=torch.bfloat16, device=dev) if self.gated else None,
            dW2=torch.empty(E, d, h, dtype=torch.bfloat16, device=dev),
            dS=torch.empty(T, K, dtype=torch.float32, device=dev),
        )

    # ---------------------------------------------------------- token rounding
    def round_tokens(self, logits, r: Routing, dp: Dispatch, m_tile: int = 128) -> RowRouting:
        """Token rounding (NR-f) of the token-choice routing r (needs its logits)."""
        dev, T, E = self.device, self.T, self.E
        cap = B.moe_rows_capacity(self.s, m_tile)
        ws = torch.empty(max(B.moe_token_rounding_workspace_size(self.s, m_tile), 256),
                         dtype=torch.uint8, device=dev)
        rr = RowRouting(cap, torch.empty(cap, dtype=torch.int32, device=dev),
                        torch.empty(E + 1, dtype=torch.int32, device=dev),
                        torch.empty(cap, dtype=torch.float32, device=dev),
                        torch.empty(T + 1, dtype=torch.int32, device=dev),
                        torch.empty(cap, dtype=torch.int32, device=dev),
                        torch.empty(cap, dtype=torch.int32, device=dev))
        B.moe_token_rounding(self.s, m_tile, logits, r.ids, dp.eti, dp.offsets, rr.eti,
                             rr.offsets, rr.w_row, rr.tok_off, rr.tok_exp, rr.tok_rows, ws)
        return rr

    def _rows_ws(self, rr: RowRouting) -> torch.Tensor:
        need = max(B.moe_workspace_size_rows(self.s, rr.rows_cap, B.MOE_WS_FORWARD),
                   B.moe_workspace_size_rows(self.s, rr.rows_cap, B.MOE_WS_BACKWARD), 256)
        if getattr(self, "_rws", None) is None or self._rws.numel() < need:
            self._rws = torch.empty(need, dtype=torch.uint8, device=self.device)
        return self._rws

    def forward_rows(self, x, W1, W3, W2, rr: RowRouting, y=None, H=None):
        if y is None:
            y = torch.empty(self.T, self.d, dtype=torch.bfloat16, device=self.device)
        if H is None:
            H = torch.empty(rr.rows_cap, self.hs, dtype=torch.bfloat16, device=self.device)
        B.moe_forward_rows(self.s, rr.rows_cap, x, W1, W3, W2, rr.eti, rr.offsets, rr.w_row,
                           rr.tok_off, rr.tok_exp, rr.tok_rows, y, H, self._rows_ws(rr))
        return y, H

    def backward_rows(self, dy, x, Wg, W1, W3, W2, rr: RowRouting, H, grads=None):
        if grads is None:
            grads = self.alloc_grads()
        dS_row = torch.empty(rr.rows_cap, dtype=torch.float32, device=self.device)
        B.moe_backward_rows(self.s, rr.rows_cap, dy, x, Wg, W1, W3, W2, rr.eti, rr.offsets,
                            rr.w_row, rr.tok_off, rr.tok_exp, rr.tok_rows, H, grads["dx"],
                            grads["dWg"], grads["dW1"], grads["dW3"], grads["dW2"], dS_row,
                            self._rows_ws(rr))
        grads["dS_row"] = dS_row
        return grads

    def step(self, x, Wg, W1, W3, W2, dy, bias=None):
        """route -> dispatch -> forward -> backward; returns all outputs."""
        r = self.route(x, Wg, bias)
        dp = self.dispatch(r.ids)
        y, H = self.forward(x, W1, W3, W2, r, dp)
        g = self.backward(dy, x, Wg, W1, W3, W2, r, dp, H)
        return r, dp, y, H, g

    def check_error(self) -> None:
        rc = B.moe_get_error()
        if rc != B.MOE_OK:
            raise B.MoeError(rc, "device")
