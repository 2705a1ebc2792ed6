"""MoELayer: the user-facing handle of one layer shape.

It owns the scratch/saved device buffers (torch allocations), checks tensor
dtypes, shapes and devices, and forwards every call to the C ABI.  No
arithmetic of the layer happens here.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import binding as B


def _need(t: torch.Tensor, name: str, shape, dtype, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class MoELayer:
    """Fused MoE layer of shape (T tokens, H hidden, I expert width, E experts, top-k)."""

    def __init__(self, T: int, H: int, I: int, E: int, k: int, prec: str = "bf16",
                 device: Optional[torch.device] = None, recompute: bool = False,
                 multicast: bool = False):
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.prec = prec
        self.recompute = recompute
        self.multicast = multicast
        device = torch.device("cuda" if device is None else device)
        if device.type == "cuda" and device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = device
        self.shape = B.make_shape(T, H, I, E, k, prec, recompute, multicast)
        self.ws = B.Workspace(self.shape, self.device)

    # ---------------------------------------------------------------- checks
    def _check_weights(self, W_gate, W_up, W_down):
        d, bf = self.device, torch.bfloat16
        _need(W_gate, "W_gate", (self.E, self.I, self.H), bf, d)
        _need(W_up, "W_up", (self.E, self.I, self.H), bf, d)
        _need(W_down, "W_down", (self.E, self.H, self.I), bf, d)

    # ---------------------------------------------------------------- passes
    def forward(self, x, topk_idx, topk_w, W_gate, W_up, W_down,
                y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        d, bf = self.device, torch.bfloat16
        _need(x, "x", (self.T, self.H), bf, d)
        _need(topk_idx, "topk_idx", (self.T, self.k), torch.int32, d)
        _need(topk_w, "topk_w", (self.T, self.k), torch.float32, d)
        self._check_weights(W_gate, W_up, W_down)
        if y is None:
            y = torch.empty((self.T, self.H), dtype=bf, device=d)
        _need(y, "y", (self.T, self.H), bf, d)
        B.mm_moe_forward(self.shape, x, topk_idx, topk_w, W_gate, W_up, W_down, y,
                         self.ws.scratch, self.ws.saved, stream)
        return y

    def backward(self, dy, W_gate, W_up, W_down, out=None, stream=None, x=None
                 ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
        """Gradients (dx, dW_gate, dW_up, dW_down, dtopk_w) of the last forward.  With
        recompute=True the forward's input x must be passed again."""
        d, bf = self.device, torch.bfloat16
        _need(dy, "dy", (self.T, self.H), bf, d)
        if self.recompute:
            if x is None:
                raise ValueError("a recompute layer's backward needs the forward's x")
            _need(x, "x", (self.T, self.H), bf, d)
        self._check_weights(W_gate, W_up, W_down)
        if out is None:
            out = (torch.empty((self.T, self.H), dtype=bf, device=d),
                   torch.empty((self.E, self.I, self.H), dtype=bf, device=d),
                   torch.empty((self.E, self.I, self.H), dtype=bf, device=d),
                   torch.empty((self.E, self.H, self.I), dtype=bf, device=d),
                   torch.empty((self.T, self.k), dtype=torch.float32, device=d))
        dx, dWg, dWu, dWd, dtw = out
        _need(dx, "dx", (self.T, self.H), bf, d)
        self._check_weights(dWg, dWu, dWd)
        _need(dtw, "dtopk_w", (self.T, self.k), torch.float32, d)
        B.mm_moe_backward(self.shape, dy, self.ws.saved, W_gate, W_up, W_down,
                          x if self.recompute else None, dx, dWg, dWu, dWd, dtw,
                          self.ws.scratch, stream)
        return out

    def routing(self):
        """(offsets [E+1], perm [T*k], inv [T*k]) int32 views of the last forward's routing."""
        return B.mm_moe_get_routing(self.shape, self.ws.saved)

    def status(self, stream=None) -> int:
        """Synchronise and return the device status word (binding.STATUS names it)."""
        return B.mm_moe_read_status(self.ws.scratch, stream)


class MoERouter:
    """The top-k router in front of MoELayer: topk_idx, topk_w from x and W_router
    [E, H], and the backward from the layer's dtopk_w (adds its dx, returns
    dW_router).  Every step runs in the library (mm_moe_router_forward/backward)."""

    def __init__(self, T: int, H: int, E: int, k: int, device: Optional[torch.device] = None):
        self.T, self.H, self.E, self.k = T, H, E, k
        device = torch.device("cuda" if device is None else device)
        if device.type == "cuda" and device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = device
        self.shape = B.make_shape(T, H, 64, E, k)   # I is not used by the router
        self.logits = torch.empty((T, E), dtype=torch.float32, device=device)
        self.dlogits = torch.empty((T, E), dtype=torch.bfloat16, device=device)

    def forward(self, x, W_router, stream=None):
        """(topk_idx [T, k] int32, topk_w [T, k] fp32); the logits stay in self.logits."""
        d, bf = self.device, torch.bfloat16
        _need(x, "x", (self.T, self.H), bf, d)
        _need(W_router, "W_router", (self.E, self.H), bf, d)
        idx = torch.empty((self.T, self.k), dtype=torch.int32, device=d)
        w = torch.empty((self.T, self.k), dtype=torch.float32, device=d)
        B.mm_moe_router_forward(self.shape, x, W_router, self.logits, idx, w, stream)
        return idx, w

    def backward(self, x, W_router, topk_idx, topk_w, dtopk_w, dx, dW_router=None, stream=None):
        """Adds the router's input gradient to dx (in place) and returns dW_router."""
        d, bf = self.device, torch.bfloat16
        _need(x, "x", (self.T, self.H), bf, d)
        _need(W_router, "W_router", (self.E, self.H), bf, d)
        _need(topk_idx, "topk_idx", (self.T, self.k), torch.int32, d)
        _need(topk_w, "topk_w", (self.T, self.k), torch.float32, d)
        _need(dtopk_w, "dtopk_w", (self.T, self.k), torch.float32, d)
        _need(dx, "dx", (self.T, self.H), bf, d)
        if dW_router is None:
            dW_router = torch.empty((self.E, self.H), dtype=bf, device=d)
        _need(dW_router, "dW_router", (self.E, self.H), bf, d)
        B.mm_moe_router_backward(self.shape, x, W_router, topk_idx, topk_w, dtopk_w,
                                 self.dlogits, dx, dW_router, stream)
        return dW_router
