"""CPU oracle of the fused MoE layer, fp64 (TEST INFRASTRUCTURE ONLY).

Follows the steps the Prime Mega MoE pages name, in their order ("Why is MoE
training communication-bound?": tokens go to a small subset of experts and the
GPU sorts them before sending; "How does the fused kernel work?": expert-parallel
dispatch, the two expert linear layers, SwiGLU, combine, and a backward pass that
the training extension adds).  On one GPU dispatch is a permutation of rows, so
the oracle is:

  route    stable sort of the flat (token, slot) indices f = t*k + j by expert
  dispatch x_perm[r] = x[perm[r] // k]
  experts  per expert e on its rows:  g = x W_gate[e]^T,  u = x W_up[e]^T,
           a = silu(g) * u,  o = a W_down[e]^T
  combine  y[t] = sum_j topk_w[t, j] * o[inv[t*k + j]]   (j ascending)

and the hand-derived backward of L = <y, dy>:

  g'  = dy W_down[e]            (per routed row, dy of its token)
  dtopk_w[t, j] = <a, g'>
  da  = w * g'
  dg  = da * u * s * (1 + g (1 - s)),  s = sigmoid(g);   du = da * silu(g)
  dx[t] = sum_j (dg W_gate[e] + du W_up[e])
  dW_gate[e] = sum_rows dg^T x,  dW_up[e] = sum_rows du^T x,
  dW_down[e] = sum_rows (w dy)^T a

Readings where the pages are silent: SwiGLU = silu(gate) * up; topk_w is used
as given (no renormalisation) and applied after the down projection; rows of one
expert keep ascending flat index; MXFP8 follows oracle.mx, each GEMM operand
quantised in 32-blocks along that GEMM's contraction axis (token-axis blocks
start at the expert's first row, the tail zero-padded); blockwise FP8 (fp8_block,
forward and backward) follows oracle.fp8block: activations in 128-blocks along the
contraction axis, weights in 128 x 128 blocks.  The layer keeps its
intermediates h = [g | u], a, w*a and dh = [dg | du] in bf16; in the modes with
an FP8 backward (mxfp8, fp8_bwd, fp8_block) the e4m3 rounding of an element is decided on
that stored bf16 value, so those modes round each of these tensors to bf16
where the layer stores it (the backward reads g, u and a as saved).  The BF16
mode keeps every intermediate in fp64.

Arithmetic is fp64 throughout; inputs are the bf16 numbers converted exactly.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from .fp8block import qdq_1d as block_qdq_1d, qdq_2d as block_qdq_2d
from .mx import bf16_round, mx_qdq

PRECISIONS = ("bf16", "mxfp8", "fp8_bwd", "fp8_block")


def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def swiglu(g, u):
    """SwiGLU activation of the gate and up projections."""
    return silu(g) * u


def swiglu_grad(g, u, da):
    """Gradients of a = silu(g) * u with respect to g and u, given da."""
    s = sigmoid(g)
    dg = da * u * s * (1.0 + g * (1.0 - s))
    du = da * silu(g)
    return dg, du


def route(topk_idx: np.ndarray, E: int):
    """Expert histogram, exclusive prefix offsets, stable permutation and its inverse.

    perm[r] = flat index t*k+j of routed row r; rows of expert e occupy
    [offsets[e], offsets[e+1]) in ascending flat index; inv[perm[r]] = r."""
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    perm = np.argsort(flat, kind="stable").astype(np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int64)
    return counts, offsets, perm, inv


def _q(v, axis, on):
    """An activation operand quantised along its contraction axis: on = False (as is),
    "mx" (MXFP8, 32-blocks) or "block" (blockwise FP8, 128-blocks)."""
    if not on:
        return v
    return block_qdq_1d(v, axis) if on == "block" else mx_qdq(v, axis)


def _qw(W, axis, on):
    """A weight operand: as an activation under MXFP8, 128 x 128 blocks (whatever the
    contraction axis) under blockwise FP8."""
    return block_qdq_2d(W) if on == "block" else _q(W, axis, on)


def _stored(v, on):
    """v as the layer stores it (bf16) when `on`, else unchanged."""
    return bf16_round(v) if on else v


def _quant_flags(prec: str):
    """The forward's and the backward's quantisation: False, "mx" or "block"."""
    if prec not in PRECISIONS:
        raise ValueError(f"unknown precision {prec!r}")
    if prec == "fp8_block":
        return "block", "block"
    return ("mx" if prec == "mxfp8" else False), ("mx" if prec in ("mxfp8", "fp8_bwd") else False)


def expert_forward(xe, Wg_e, Wu_e, Wd_e, prec: str = "bf16"):
    """One expert on its rows xe [n, H]: returns g, u, a [n, I] and o [n, H]."""
    qf, _ = _quant_flags(prec)
    xq = _q(xe, 1, qf)
    g = xq @ _qw(Wg_e, 1, qf).T
    u = xq @ _qw(Wu_e, 1, qf).T
    a = swiglu(g, u)
    o = _q(_stored(a, qf), 1, qf) @ _qw(Wd_e, 1, qf).T
    return g, u, a, o


def expert_backward(xe, dye, we, g, u, a, Wg_e, Wu_e, Wd_e, prec: str = "bf16"):
    """Backward of one expert on its rows.

    xe, dye [n, H]: the rows' inputs and their tokens' upstream gradients;
    we [n]: their routing weights; g, u, a: the forward intermediates.
    Returns dxe [n, H], dWg_e, dWu_e [I, H], dWd_e [H, I], dw [n]."""
    _, qb = _quant_flags(prec)
    g, u, a = _stored(g, qb), _stored(u, qb), _stored(a, qb)   # as the forward saved them
    gp = _q(dye, 1, qb) @ _qw(Wd_e, 0, qb)                # g' = dy W_down[e]
    dw = np.sum(a * gp, axis=1)
    da = we[:, None] * gp
    dg, du = swiglu_grad(g, u, da)
    dg, du = _stored(dg, qb), _stored(du, qb)
    dxe = _q(dg, 1, qb) @ _qw(Wg_e, 0, qb) + _q(du, 1, qb) @ _qw(Wu_e, 0, qb)
    xq = _q(xe, 0, qb)
    dWg_e = _q(dg, 0, qb).T @ xq
    dWu_e = _q(du, 0, qb).T @ xq
    dWd_e = _q(dye, 0, qb).T @ _q(_stored(we[:, None] * a, qb), 0, qb)
    return dxe, dWg_e, dWu_e, dWd_e, dw


def _as64(*arrs):
    return [np.asarray(a, dtype=np.float64) for a in arrs]


def forward(x, topk_idx, topk_w, W_gate, W_up, W_down, prec: str = "bf16") -> Dict:
    """Layer forward.  Returns y [T, H] plus the routing and per-row intermediates
    (in routed-row order) under the keys counts, offsets, perm, inv, g, u, a, o."""
    x, W_gate, W_up, W_down = _as64(x, W_gate, W_up, W_down)
    topk_idx = np.asarray(topk_idx)
    w = np.asarray(topk_w, dtype=np.float64).reshape(-1)
    T, H = x.shape
    E, I, _ = W_gate.shape
    k = topk_idx.shape[1]
    counts, offsets, perm, inv = route(topk_idx, E)
    R = T * k
    x_perm = x[perm // k]
    g = np.zeros((R, I)); u = np.zeros((R, I)); a = np.zeros((R, I))
    o = np.zeros((R, H))
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        g[lo:hi], u[lo:hi], a[lo:hi], o[lo:hi] = expert_forward(
            x_perm[lo:hi], W_gate[e], W_up[e], W_down[e], prec)
    y = np.zeros((T, H))
    for j in range(k):
        f = np.arange(T) * k + j
        y += w[f][:, None] * o[inv[f]]
    return dict(y=y, counts=counts, offsets=offsets, perm=perm, inv=inv,
                g=g, u=u, a=a, o=o)


def backward(dy, x, topk_idx, topk_w, W_gate, W_up, W_down, prec: str = "bf16",
             fwd: Optional[Dict] = None) -> Dict:
    """Layer backward of L = <y, dy>.  Returns dx [T,H], dW_gate, dW_up [E,I,H],
    dW_down [E,H,I] and dtopk_w [T,k]."""
    dy, x, W_gate, W_up, W_down = _as64(dy, x, W_gate, W_up, W_down)
    topk_idx = np.asarray(topk_idx)
    w = np.asarray(topk_w, dtype=np.float64).reshape(-1)
    if fwd is None:
        fwd = forward(x, topk_idx, topk_w, W_gate, W_up, W_down, prec)
    T, H = x.shape
    E, I, _ = W_gate.shape
    k = topk_idx.shape[1]
    offsets, perm, inv = fwd["offsets"], fwd["perm"], fwd["inv"]
    R = T * k
    x_perm = x[perm // k]
    dy_perm = dy[perm // k]
    w_perm = w[perm]
    dx_perm = np.zeros((R, H))
    dw_perm = np.zeros(R)
    dW_gate = np.zeros_like(W_gate); dW_up = np.zeros_like(W_up)
    dW_down = np.zeros_like(W_down)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue            # an expert with no rows has zero weight gradients
        s = slice(lo, hi)
        dx_perm[s], dW_gate[e], dW_up[e], dW_down[e], dw_perm[s] = expert_backward(
            x_perm[s], dy_perm[s], w_perm[s], fwd["g"][s], fwd["u"][s], fwd["a"][s],
            W_gate[e], W_up[e], W_down[e], prec)
    dx = np.zeros((T, H))
    dtopk_w = np.zeros((T, k))
    for j in range(k):
        f = np.arange(T) * k + j
        dx += dx_perm[inv[f]]
        dtopk_w[:, j] = dw_perm[inv[f]]
    return dict(dx=dx, dW_gate=dW_gate, dW_up=dW_up, dW_down=dW_down, dtopk_w=dtopk_w)


def token_subset(inputs: Dict[str, np.ndarray], tokens: Sequence[int]) -> Dict[str, np.ndarray]:
    """The layer is per token apart from the weight gradients: y[t], dx[t] and
    dtopk_w[t] of a token depend only on that token's row of x, dy, topk_idx and
    topk_w.  Returns those rows for a sampled check at full size."""
    tokens = np.asarray(tokens, dtype=np.int64)
    out = dict(inputs)
    for key in ("x", "dy", "topk_idx", "topk_w"):
        if key in inputs:
            out[key] = np.asarray(inputs[key])[tokens]
    return out


def expert_rows(topk_idx: np.ndarray, e: int) -> np.ndarray:
    """Flat indices t*k+j routed to expert e, ascending (its rows in routed order)."""
    flat = np.asarray(topk_idx).reshape(-1)
    return np.nonzero(flat == e)[0]


def expert_weight_grads(inputs: Dict[str, np.ndarray], e: int, prec: str = "bf16"):
    """dW_gate[e], dW_up[e], dW_down[e] of one expert, from its rows only."""
    k = np.asarray(inputs["topk_idx"]).shape[1]
    f = expert_rows(inputs["topk_idx"], e)
    x, dy, Wg, Wu, Wd = _as64(inputs["x"], inputs["dy"], inputs["W_gate"][e],
                              inputs["W_up"][e], inputs["W_down"][e])
    H = x.shape[1]
    I = Wg.shape[0]
    if f.size == 0:
        return np.zeros((I, H)), np.zeros((I, H)), np.zeros((H, I))
    xe = x[f // k]
    dye = dy[f // k]
    we = np.asarray(inputs["topk_w"], dtype=np.float64).reshape(-1)[f]
    g, u, a, _ = expert_forward(xe, Wg, Wu, Wd, prec)
    _, dWg, dWu, dWd, _ = expert_backward(xe, dye, we, g, u, a, Wg, Wu, Wd, prec)
    return dWg, dWu, dWd
