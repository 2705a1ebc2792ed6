"""Checks that pin the CPU oracle to something other than itself.

Each check returns the largest relative discrepancy it saw (0.0 = exact) so the
pin tests can assert a bound and the mutation tests can assert that a planted
mistake in the oracle pushes at least one check past its bound.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle.moe as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.abs(b).max(initial=0.0), 1e-300)
    return float(np.abs(a - b).max(initial=0.0) / den)


def small_problem(T=6, H=8, I=4, E=3, k=2, seed=0, idx=None, w=None):
    rng = np.random.default_rng(seed)
    d = dict(
        x=rng.standard_normal((T, H)),
        W_gate=rng.standard_normal((E, I, H)) * 0.5,
        W_up=rng.standard_normal((E, I, H)) * 0.5,
        W_down=rng.standard_normal((E, H, I)) * 0.5,
        dy=rng.standard_normal((T, H)),
    )
    if idx is None:
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    d["topk_idx"] = np.asarray(idx, dtype=np.int32)
    if w is None:
        w = rng.random((T, k)) + 0.1
    d["topk_w"] = np.asarray(w, dtype=np.float64)
    return d


def _fwd(d, prec="bf16"):
    return om.forward(d["x"], d["topk_idx"], d["topk_w"], d["W_gate"], d["W_up"],
                          d["W_down"], prec)


def _bwd(d, prec="bf16"):
    return om.backward(d["dy"], d["x"], d["topk_idx"], d["topk_w"], d["W_gate"],
                           d["W_up"], d["W_down"], prec)


# ---------------------------------------------------------------- routing
def brute_force_route(topk_idx, E):
    """O(R*E) scan: for each expert in turn, collect its flat indices in order."""
    flat = [int(v) for v in np.asarray(topk_idx).reshape(-1)]
    perm, offsets = [], [0]
    for e in range(E):
        for f, ee in enumerate(flat):
            if ee == e:
                perm.append(f)
        offsets.append(len(perm))
    inv = [0] * len(perm)
    for r, f in enumerate(perm):
        inv[f] = r
    return np.array(offsets), np.array(perm), np.array(inv)


def pin_route(topk_idx, E) -> float:
    counts, offsets, perm, inv = om.route(topk_idx, E)
    bo, bp, bi = brute_force_route(topk_idx, E)
    ok = (np.array_equal(offsets, bo) and np.array_equal(perm, bp)
          and np.array_equal(inv, bi) and np.array_equal(np.diff(offsets), counts))
    return 0.0 if ok else 1.0


# ---------------------------------------------------------------- forward
def _dense_mlp_torch(x, Wg, Wu, Wd):
    """The textbook SwiGLU MLP, written with torch.nn.functional."""
    x = torch.as_tensor(x, dtype=torch.float64)
    h = F.silu(F.linear(x, torch.as_tensor(Wg, dtype=torch.float64))) * \
        F.linear(x, torch.as_tensor(Wu, dtype=torch.float64))
    return F.linear(h, torch.as_tensor(Wd, dtype=torch.float64))


def pin_k1_dense(seed=0) -> float:
    """k = 1 and weight 1: each token's output is the dense SwiGLU MLP of its expert."""
    T, E = 10, 4
    rng = np.random.default_rng(seed + 11)
    idx = rng.integers(0, E, size=(T, 1))
    d = small_problem(T=T, E=E, k=1, idx=idx, w=np.ones((T, 1)), seed=seed)
    y = _fwd(d)["y"]
    ref = np.stack([_dense_mlp_torch(d["x"][t:t + 1], d["W_gate"][idx[t, 0]],
                                     d["W_up"][idx[t, 0]], d["W_down"][idx[t, 0]]).numpy()[0]
                    for t in range(T)])
    return rel(y, ref)


def pin_identical_experts(seed=0) -> float:
    """All experts equal: y = (sum_j w_tj) * MLP(x_t)."""
    d = small_problem(T=7, E=4, k=3, seed=seed)
    for key in ("W_gate", "W_up", "W_down"):
        d[key] = np.repeat(d[key][:1], 4, axis=0)
    y = _fwd(d)["y"]
    ref = _dense_mlp_torch(d["x"], d["W_gate"][0], d["W_up"][0], d["W_down"][0]).numpy()
    ref = ref * d["topk_w"].sum(axis=1, keepdims=True)
    return rel(y, ref)


def pin_linearity(seed=0) -> float:
    """Doubling W_down doubles y exactly (a power-of-two scale is exact in fp64)."""
    d = small_problem(seed=seed)
    y1 = _fwd(d)["y"]
    d2 = dict(d, W_down=d["W_down"] * 2.0)
    y2 = _fwd(d2)["y"]
    return 0.0 if np.array_equal(y2, 2.0 * y1) else 1.0


def pin_golden() -> float:
    """Hand-derived closed-form worked example (tests/golden)."""
    with open(os.path.join(GOLDEN, "worked_example_T1_E2_k2.json")) as fh:
        g = json.load(fh)
    d = {k: np.asarray(g[k], dtype=np.float64) for k in
         ("x", "topk_w", "W_gate", "W_up", "W_down", "dy")}
    d["topk_idx"] = np.asarray(g["topk_idx"], dtype=np.int32)
    s = lambda z: 1.0 / (1.0 + math.exp(-z))  # noqa: E731
    worst = 0.0
    f = _fwd(d)
    b = _bwd(d)
    got = dict(y=f["y"], **{k: b[k] for k in ("dtopk_w", "dx", "dW_gate", "dW_up", "dW_down")})
    for name, ent in g["expected"].items():
        val = np.asarray(ent["value"], dtype=np.float64)
        # the stored numbers are the closed forms evaluated
        if name in ("y", "dtopk_w", "dx"):
            ev = np.asarray([[eval(e, {"s": s}) for e in ent["expr"]]])
        else:
            ev = np.asarray([eval(e, {"s": s}) for e in ent["expr"]], dtype=np.float64)
        worst = max(worst, rel(val, ev), rel(got[name], val))
    return worst


def pin_permute_roundtrip(seed=0) -> float:
    d = small_problem(T=9, E=5, k=3, seed=seed)
    _, _, perm, inv = om.route(d["topk_idx"], 5)
    k = 3
    xp = d["x"][perm // k]
    back = xp[inv].reshape(9, k, -1)
    ok = all(np.array_equal(back[:, j], d["x"]) for j in range(k))
    return 0.0 if ok else 1.0


# ---------------------------------------------------------------- backward
def loss(d) -> float:
    return float(np.sum(_fwd(d)["y"] * d["dy"]))


def pin_finite_differences(seed=0, n_samples=12) -> float:
    """Central differences of L = <y, dy> against every analytic gradient."""
    d = small_problem(T=6, H=8, I=4, E=3, k=2, seed=seed)
    b = _bwd(d)
    grads = dict(x=b["dx"], W_gate=b["dW_gate"], W_up=b["dW_up"], W_down=b["dW_down"],
                 topk_w=b["dtopk_w"])
    rng = np.random.default_rng(seed + 99)
    worst = 0.0
    for name, gana in grads.items():
        theta = d[name]
        flat_idx = rng.choice(theta.size, size=min(n_samples, theta.size), replace=False)
        for fi in flat_idx:
            pos = np.unravel_index(fi, theta.shape)
            eps = 1e-5 * max(1.0, abs(theta[pos]))
            dp = {**d, name: theta.copy()}; dp[name][pos] += eps
            dm = {**d, name: theta.copy()}; dm[name][pos] -= eps
            fd = (loss(dp) - loss(dm)) / (2 * eps)
            scale = max(np.abs(gana).max(), 1e-12)
            worst = max(worst, abs(fd - gana[pos]) / scale)
    return worst


def pin_k1_autograd(seed=0) -> float:
    """k = 1, weight w: gradients equal torch autograd of w * MLP(x) for each token."""
    T, E = 8, 3
    rng = np.random.default_rng(seed + 5)
    idx = rng.integers(0, E, size=(T, 1))
    d = small_problem(T=T, E=E, k=1, idx=idx, seed=seed)
    b = _bwd(d)
    xt = torch.tensor(d["x"], requires_grad=True)
    Ws = {k: torch.tensor(d[k], requires_grad=True) for k in ("W_gate", "W_up", "W_down")}
    wt = torch.tensor(d["topk_w"], requires_grad=True)
    L = 0.0
    for t in range(T):
        e = int(idx[t, 0])
        yt = wt[t, 0] * _dense_mlp_autograd(xt[t:t + 1], Ws["W_gate"][e], Ws["W_up"][e],
                                            Ws["W_down"][e])
        L = L + (yt * torch.tensor(d["dy"][t:t + 1])).sum()
    L.backward()
    worst = rel(b["dx"], xt.grad.numpy())
    for k in Ws:
        worst = max(worst, rel(b["d" + k], Ws[k].grad.numpy()))
    worst = max(worst, rel(b["dtopk_w"], wt.grad.numpy()))
    return worst


def _dense_mlp_autograd(x, Wg, Wu, Wd):
    return F.linear(F.silu(F.linear(x, Wg)) * F.linear(x, Wu), Wd)


def pin_empty_expert_zero_grad(seed=0) -> float:
    """An expert that receives no token gets exactly zero weight gradients."""
    d = small_problem(T=6, E=4, k=2, seed=seed, idx=np.array([[0, 1], [1, 2], [2, 0],
                                                              [0, 2], [1, 0], [2, 1]]))
    b = _bwd(d)
    nz = (np.abs(b["dW_gate"][3]).max() + np.abs(b["dW_up"][3]).max()
          + np.abs(b["dW_down"][3]).max())
    live = np.abs(b["dW_gate"][:3]).max()
    return 0.0 if (nz == 0.0 and live > 0) else 1.0


ALL_PINS = dict(
    route=lambda: pin_route(np.random.default_rng(3).integers(0, 6, size=(17, 3)), 6),
    k1_dense=pin_k1_dense,
    identical_experts=pin_identical_experts,
    linearity=pin_linearity,
    golden=pin_golden,
    permute_roundtrip=pin_permute_roundtrip,
    finite_differences=pin_finite_differences,
    k1_autograd=pin_k1_autograd,
    empty_expert=pin_empty_expert_zero_grad,
)

BOUNDS = dict(route=0.0, k1_dense=1e-12, identical_experts=1e-12, linearity=0.0,
              golden=1e-12, permute_roundtrip=0.0, finite_differences=1e-6,
              k1_autograd=1e-12, empty_expert=0.0)
