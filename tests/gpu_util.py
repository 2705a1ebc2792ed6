"""Helpers of the GPU tests: upload the seeded inputs, run the layer through the
C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_16_gb300 import MoELayer, build

DEV = "cuda"


def ensure_built():
    build.build()


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def upload(d):
    out = dict(
        x=bf16_dev(d["x_bits"]),
        topk_idx=torch.from_numpy(np.ascontiguousarray(d["topk_idx"], dtype=np.int32)).to(DEV),
        topk_w=torch.from_numpy(np.ascontiguousarray(d["topk_w"], dtype=np.float32)).to(DEV),
        W_gate=bf16_dev(d["W_gate_bits"]), W_up=bf16_dev(d["W_up_bits"]),
        W_down=bf16_dev(d["W_down_bits"]))
    if "dy_bits" in d:
        out["dy"] = bf16_dev(d["dy_bits"])
    return out


def run(d, backward=True, layer=None, dev=None):
    T, H = d["x"].shape
    E, I, _ = d["W_gate"].shape
    k = d["topk_idx"].shape[1]
    if layer is None:
        layer = MoELayer(T, H, I, E, k)
    if dev is None:
        dev = upload(d)
    y = layer.forward(dev["x"], dev["topk_idx"], dev["topk_w"], dev["W_gate"], dev["W_up"],
                      dev["W_down"])
    res = dict(y=y)
    if backward:
        dx, dWg, dWu, dWd, dtw = layer.backward(dev["dy"], dev["W_gate"], dev["W_up"],
                                                dev["W_down"])
        res.update(dx=dx, dW_gate=dWg, dW_up=dWu, dW_down=dWd, dtopk_w=dtw)
    torch.cuda.synchronize()
    res["status"] = layer.status()
    off, perm, inv = layer.routing()
    res.update(offsets=off, perm=perm, inv=inv)
    return res, layer, dev


def rel_err(gpu, ref) -> float:
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    den = np.abs(r).max(initial=0.0)
    if den == 0.0:
        return float(np.abs(g).max(initial=0.0))
    return float(np.abs(g - r).max(initial=0.0) / den)
