"""The router oracle against independent facts: brute-force top-k with the tie rule,
the full softmax (scipy) renormalised over the chosen experts, a logit shift that
changes nothing, the softmax Jacobian's zero row sums, central finite differences of
L = sum(G * topk_w) for dW_router and dx, and planted mistakes that must fail."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle.router as orr


def brute_topk(s, k):
    out = []
    for row in s:
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))
        out.append(order[:k])
    return np.array(out)


def inputs(seed, T=24, H=64, E=16, scale=0.3):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, H)), rng.standard_normal((E, H)) * scale


@pytest.mark.parametrize("k", [1, 2, 5])
def test_topk_matches_brute_force_with_ties(k):
    rng = np.random.default_rng(k)
    s = rng.integers(-3, 4, size=(200, 12)).astype(np.float64)   # many equal logits
    assert np.array_equal(orr.select_topk(s, k), brute_topk(s, k))


def test_weights_are_the_renormalised_full_softmax():
    x, W = inputs(1)
    f = orr.forward(x, W, 4)
    full = softmax(x @ W.T, axis=1)
    chosen = np.take_along_axis(full, f["topk_idx"], axis=1)
    assert np.allclose(f["topk_w"], chosen / chosen.sum(axis=1, keepdims=True), rtol=1e-13)
    assert np.allclose(f["topk_w"].sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(np.diff(np.take_along_axis(f["logits"], f["topk_idx"], axis=1), axis=1) <= 0)


def test_shifting_every_expert_by_one_vector_changes_nothing():
    x, W = inputs(2)
    v = np.random.default_rng(3).standard_normal(W.shape[1])
    a, b = orr.forward(x, W, 3), orr.forward(x, W + v, 3)
    assert np.array_equal(a["topk_idx"], b["topk_idx"])
    assert np.allclose(a["topk_w"], b["topk_w"], rtol=1e-12)


def test_logit_gradient_rows_sum_to_zero():
    x, W = inputs(4)
    f = orr.forward(x, W, 4)
    G = np.random.default_rng(5).standard_normal(f["topk_w"].shape)
    b = orr.backward(x, W, f["topk_idx"], f["topk_w"], G)
    assert np.allclose(b["dlogits"].sum(axis=1), 0.0, atol=1e-14)
    assert np.count_nonzero(b["dlogits"]) <= f["topk_idx"].size


def _fd_check(seed=6, k=3, n=40):
    x, W = inputs(seed, scale=1.0)        # well separated logits: the selection is locally fixed
    f = orr.forward(x, W, k)
    G = np.random.default_rng(seed + 1).standard_normal(f["topk_w"].shape)
    b = orr.backward(x, W, f["topk_idx"], f["topk_w"], G)

    def L(xx, WW):
        ff = orr.forward(xx, WW, k)
        assert np.array_equal(ff["topk_idx"], f["topk_idx"])
        return float(np.sum(G * ff["topk_w"]))

    rng = np.random.default_rng(seed + 2)
    for name, arr, grad in (("W", W, b["dW_router"]), ("x", x, b["dx"])):
        for _ in range(n):
            i = tuple(rng.integers(0, d) for d in arr.shape)
            eps = 1e-6 * max(1.0, abs(arr[i]))
            p, m = arr.copy(), arr.copy()
            p[i] += eps
            m[i] -= eps
            num = (L(p, W) - L(m, W)) / (2 * eps) if name == "x" else (L(x, p) - L(x, m)) / (2 * eps)
            assert abs(num - grad[i]) <= 1e-6 * max(1.0, abs(num)), (name, i, num, grad[i])


def test_finite_differences():
    _fd_check()


def test_planted_mistakes_are_caught(monkeypatch):
    # ties to the higher index
    monkeypatch.setattr(orr, "select_topk",
                        lambda s, k: np.argsort(-np.asarray(s)[:, ::-1], axis=1,
                                                kind="stable")[:, :k] * -1 + (s.shape[1] - 1))
    with pytest.raises(AssertionError):
        test_topk_matches_brute_force_with_ties(2)
    monkeypatch.undo()
    # no renormalisation over the chosen experts
    monkeypatch.setattr(orr, "topk_softmax", lambda sc: np.exp(sc) / np.exp(sc).sum() * len(sc))
    with pytest.raises(AssertionError):
        test_weights_are_the_renormalised_full_softmax()
    monkeypatch.undo()
    # the Jacobian without the mean term
    orig = orr.backward

    def bad_backward(x, W, idx, w, g):
        out = orig(x, W, idx, w, np.asarray(g) * 0 + 0)
        ds = np.zeros_like(out["dlogits"])
        np.put_along_axis(ds, np.asarray(idx), np.asarray(w) * np.asarray(g), axis=1)
        return dict(dlogits=ds, dW_router=ds.T @ np.asarray(x), dx=ds @ np.asarray(W))
    monkeypatch.setattr(orr, "backward", bad_backward)
    with pytest.raises(AssertionError):
        _fd_check()
