"""The CPU oracle against what the mathematics and the pages' reading fix.

Pins: brute-force routing, the dense SwiGLU MLP of torch.nn.functional (k=1),
identical experts, exact linearity in W_down, a hand-derived closed-form worked
example, permute/un-permute round trip, central finite differences for every
gradient, torch autograd (k=1) and zero gradients of an empty expert.  The
mutation tests plant plausible mistakes in the oracle (on the CPU) and check
that some pin catches each one.
"""
import numpy as np
import pytest

import oracle
import oracle.moe as om
from tests import pins


@pytest.mark.parametrize("name", sorted(pins.ALL_PINS))
def test_pin(name):
    err = pins.ALL_PINS[name]()
    assert err <= pins.BOUNDS[name], f"{name}: {err}"


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 3, 3), (33, 8, 2), (64, 128, 8), (100, 4, 1)])
def test_route_brute_force(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    assert pins.pin_route(idx, E) == 0.0


def test_route_edge_cases():
    # every token to one expert; all other experts empty
    idx = np.zeros((20, 1), dtype=np.int32) + 3
    counts, offsets, perm, inv = oracle.route(idx, 5)
    assert counts.tolist() == [0, 0, 0, 20, 0]
    assert offsets.tolist() == [0, 0, 0, 0, 20, 20]
    assert perm.tolist() == list(range(20))
    # invariants on a random case
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 7, size=(50, 3))
    counts, offsets, perm, inv = oracle.route(idx, 7)
    assert counts.sum() == 150 and np.all(np.diff(offsets) >= 0)
    assert np.array_equal(inv[perm], np.arange(150))
    flat = idx.reshape(-1)
    for e in range(7):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    with pytest.raises(ValueError):
        oracle.route(np.array([[7]]), 7)


def test_finite_differences_several_seeds():
    for seed in (1, 2):
        assert pins.pin_finite_differences(seed=seed, n_samples=6) <= 1e-6


def test_subset_and_expert_grads_match_full():
    """The sampled-check helpers give the same numbers as the full oracle."""
    d = pins.small_problem(T=12, E=4, k=2, seed=4)
    full_f = pins._fwd(d)
    full_b = pins._bwd(d)
    toks = [1, 5, 11]
    sub = om.token_subset(d, toks)
    sf = pins._fwd(sub)
    sb = pins._bwd(sub)
    assert np.allclose(sf["y"], full_f["y"][toks], rtol=0, atol=1e-13)
    assert np.allclose(sb["dx"], full_b["dx"][toks], rtol=0, atol=1e-13)
    assert np.allclose(sb["dtopk_w"], full_b["dtopk_w"][toks], rtol=0, atol=1e-13)
    for e in range(4):
        g, u, dd = om.expert_weight_grads(d, e)
        assert np.allclose(g, full_b["dW_gate"][e], atol=1e-13)
        assert np.allclose(u, full_b["dW_up"][e], atol=1e-13)
        assert np.allclose(dd, full_b["dW_down"][e], atol=1e-13)


# ---------------------------------------------------------------- planted mistakes
def _sigmoid_wrong_sign(z):
    return 1.0 / (1.0 + np.exp(z))


def _swiglu_grad_dropped_term(g, u, da):
    s = om.sigmoid(g)
    return da * u * s, da * om.silu(g)            # drops the g (1 - s) term


def _swiglu_grad_swapped(g, u, da):
    dg, du = _orig_swiglu_grad(g, u, da)
    return du, dg


def _swiglu_wrong_order(g, u):
    return om.silu(u) * g                         # gate and up swapped


def _route_unstable(topk_idx, E):
    counts, offsets, perm, inv = _orig_route(topk_idx, E)
    perm = perm.copy()
    for e in range(E):                           # reverse the order inside each expert
        perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
    inv = np.empty_like(perm); inv[perm] = np.arange(perm.size)
    return counts, offsets, perm, inv


def _route_bad_inverse(topk_idx, E):
    counts, offsets, perm, inv = _orig_route(topk_idx, E)
    return counts, offsets, perm, perm.copy()     # uses perm where inv is needed


def _expert_backward_transposed_down(xe, dye, we, g, u, a, Wg_e, Wu_e, Wd_e, prec="bf16"):
    out = list(_orig_expert_backward(xe, dye, we, g, u, a, Wg_e, Wu_e, Wd_e, prec))
    out[3] = out[3][::-1].copy()                  # wrong index into dW_down
    return tuple(out)


def _expert_backward_no_weight(xe, dye, we, g, u, a, Wg_e, Wu_e, Wd_e, prec="bf16"):
    return _orig_expert_backward(xe, dye, np.ones_like(we), g, u, a, Wg_e, Wu_e, Wd_e, prec)


_orig_swiglu_grad = om.swiglu_grad
_orig_route = om.route
_orig_expert_backward = om.expert_backward

MUTANTS = {
    "sigmoid_sign": ("sigmoid", _sigmoid_wrong_sign),
    "dswiglu_dropped_term": ("swiglu_grad", _swiglu_grad_dropped_term),
    "dswiglu_swapped": ("swiglu_grad", _swiglu_grad_swapped),
    "swiglu_order": ("swiglu", _swiglu_wrong_order),
    "route_unstable": ("route", _route_unstable),
    "route_inverse": ("route", _route_bad_inverse),
    "dW_down_index": ("expert_backward", _expert_backward_transposed_down),
    "backward_drops_weight": ("expert_backward", _expert_backward_no_weight),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, monkeypatch):
    attr, fn = MUTANTS[mutant]
    monkeypatch.setattr(om, attr, fn)
    caught = []
    for name, pin in pins.ALL_PINS.items():
        try:
            err = pin()
        except Exception:
            err = float("inf")
        if not err <= pins.BOUNDS[name]:
            caught.append(name)
    assert caught, f"no pin caught the planted mistake {mutant}"
