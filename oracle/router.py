"""CPU oracle of the top-k router in front of the MoE layer, fp64 (TEST INFRASTRUCTURE
ONLY: imported by tests/, the smoke check and bench.py's CPU baseline, never by the
library).

The Prime Mega MoE pages say only that each token goes to a small subset of the
experts ("Why is MoE training communication-bound?") and that the tested models use
128 experts with top-8 ("TL;DR"); the router itself is not described.  Readings:

  logits    s = x W_router^T                     (no bias), [T, E]
  select    the k largest logits of each token, in descending order; equal logits
            go to the lower expert index
  weights   topk_w[t, j] = softmax over the k chosen logits (equal to the full
            softmax over E renormalised over the chosen k)
  backward  only through topk_w (the selection is piecewise constant):
            ds[t, e_j] = w_j (g_j - sum_i w_i g_i),  g = dtopk_w[t], zero elsewhere;
            dW_router = ds^T x,   dx_router = ds W_router
"""
from __future__ import annotations

from typing import Dict

import numpy as np


def logits(x, W_router) -> np.ndarray:
    return np.asarray(x, dtype=np.float64) @ np.asarray(W_router, dtype=np.float64).T


def select_topk(s: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, descending; ties to the lower index."""
    s = np.asarray(s, dtype=np.float64)
    # a stable sort of (-s) keeps the lower index first among equal values
    order = np.argsort(-s, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def topk_softmax(s_chosen: np.ndarray) -> np.ndarray:
    m = s_chosen.max(axis=1, keepdims=True)
    e = np.exp(s_chosen - m)
    return e / e.sum(axis=1, keepdims=True)


def forward(x, W_router, k: int) -> Dict[str, np.ndarray]:
    s = logits(x, W_router)
    idx = select_topk(s, k)
    w = topk_softmax(np.take_along_axis(s, idx, axis=1))
    return dict(logits=s, topk_idx=idx, topk_w=w)


def backward(x, W_router, topk_idx, topk_w, dtopk_w) -> Dict[str, np.ndarray]:
    x = np.asarray(x, dtype=np.float64)
    W = np.asarray(W_router, dtype=np.float64)
    w = np.asarray(topk_w, dtype=np.float64)
    g = np.asarray(dtopk_w, dtype=np.float64)
    T = x.shape[0]
    E = W.shape[0]
    dchosen = w * (g - np.sum(w * g, axis=1, keepdims=True))    # softmax Jacobian
    ds = np.zeros((T, E))
    np.put_along_axis(ds, np.asarray(topk_idx, dtype=np.int64), dchosen, axis=1)
    return dict(dlogits=ds, dW_router=ds.T @ x, dx=ds @ W)
