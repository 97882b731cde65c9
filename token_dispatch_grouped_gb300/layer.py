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
