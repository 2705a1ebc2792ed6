"""Helpers of the GPU tests: upload the seeded inputs, run the layer through the
C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import oracle.moe as om
from mixture_experts_layer_16_gb300 import MoELayer, build
from mixture_experts_layer_16_gb300.inputs import CONFIGS, make_inputs

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


def run(d, backward=True, layer=None, dev=None, prec="bf16", recompute=False, multicast=False):
    T, H = d["x"].shape
    E, I, _ = d["W_gate"].shape
    k = d["topk_idx"].shape[1]
    if layer is None:
        layer = MoELayer(T, H, I, E, k, prec, recompute=recompute, multicast=multicast)
    if dev is None:
        dev = upload(d)
    y = layer.forward(dev["x"], dev["topk_idx"], dev["topk_w"], dev["W_gate"], dev["W_up"],
                      dev["W_down"])
    res = dict(y=y)
    if backward:
        dx, dWg, dWu, dWd, dtw = layer.backward(dev["dy"], dev["W_gate"], dev["W_up"],
                                                dev["W_down"], x=dev["x"])
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


def check_routing(res, topk_idx, E):
    counts, offsets, perm, inv = oracle.route(topk_idx, E)
    assert np.array_equal(res["offsets"].cpu().numpy(), offsets.astype(np.int32))
    assert np.array_equal(res["perm"].cpu().numpy(), perm.astype(np.int32))
    assert np.array_equal(res["inv"].cpu().numpy(), inv.astype(np.int32))


def full_errors(d, res, backward=True, prec="bf16"):
    """Relative errors of every output against the oracle run in precision `prec`."""
    f = oracle.forward(d["x"], d["topk_idx"], d["topk_w"], d["W_gate"], d["W_up"], d["W_down"],
                       prec)
    errs = {"y": rel_err(f32(res["y"]), f["y"])}
    if backward:
        b = oracle.backward(d["dy"], d["x"], d["topk_idx"], d["topk_w"], d["W_gate"], d["W_up"],
                            d["W_down"], prec, fwd=f)
        for key in ("dx", "dW_gate", "dW_up", "dW_down", "dtopk_w"):
            errs[key] = rel_err(f32(res[key]), b[key])
    return errs


def check_full(d, res, backward=True, tol=1e-2, prec="bf16"):
    errs = full_errors(d, res, backward, prec)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"outside tolerance: {bad} (all: {errs})"
    return errs


def sampled_check(name, tol, n_tokens=48, seed=0):
    """A full-size workload on the GPU; the oracle (in the workload's precision) on
    sampled tokens (y, dx, dtopk_w are per token) and on the weight gradients of the
    least, the median and the most loaded expert (each needs only that expert's rows;
    the median one has a mid-size token-axis K, not a multiple of the K step)."""
    cfg = CONFIGS[name]
    d = make_inputs(cfg)
    res, layer, dev = run(d, prec=cfg.prec)
    assert res["status"] == 0
    check_routing(res, d["topk_idx"], cfg.E)
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(cfg.T, size=n_tokens, replace=False))
    sub = om.token_subset(d, toks)
    f = oracle.forward(sub["x"], sub["topk_idx"], sub["topk_w"], d["W_gate"], d["W_up"],
                       d["W_down"], cfg.prec)
    b = oracle.backward(sub["dy"], sub["x"], sub["topk_idx"], sub["topk_w"], d["W_gate"],
                        d["W_up"], d["W_down"], cfg.prec, fwd=f)
    errs = {"y": rel_err(f32(res["y"][toks]), f["y"]),
            "dx": rel_err(f32(res["dx"][toks]), b["dx"]),
            "dtopk_w": rel_err(f32(res["dtopk_w"][toks]), b["dtopk_w"])}
    counts = np.bincount(d["topk_idx"].reshape(-1), minlength=cfg.E)
    order = np.argsort(counts, kind="stable")
    median = int(order[len(order) // 2])
    for e in {int(order[0]), median, int(order[-1])}:
        g, u, dd = om.expert_weight_grads(d, e, cfg.prec)
        errs[f"dW_gate[{e}]"] = rel_err(f32(res["dW_gate"][e]), g)
        errs[f"dW_up[{e}]"] = rel_err(f32(res["dW_up"][e]), u)
        errs[f"dW_down[{e}]"] = rel_err(f32(res["dW_down"][e]), dd)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"outside tolerance: {bad} (all: {errs})"
    return errs
