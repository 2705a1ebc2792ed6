"""The router (mm_moe_router_forward/backward) on the GPU against the router oracle.

The selection is an integer decided by floating point, so it is also checked in the
kernel's precision: the oracle's rule (k largest, descending, ties to the lower
index) applied to the kernel's own fp32 logits must give exactly the kernel's
topk_idx.  Against the oracle's fp64 forward the choice must be valid up to fp32
rounding and equal where no near-tie exists.  Every expected value is the oracle's
own: logits within 1e-5 relative to their maximum, topk_w within 1e-5, gradients
(from the oracle's choice and weights) within 1e-2 (dlogits are rounded to bf16).  Last,
router -> layer -> layer backward -> router backward against the two oracles
composed."""
import numpy as np
import pytest
import torch

import oracle
import oracle.router as orr
from mixture_experts_layer_16_gb300 import MoERouter
from mixture_experts_layer_16_gb300.inputs import custom_inputs, router_weights
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def run_router(x_bits, Wr_bits, k, dtopk_w=None, dx_in=None):
    T, H = x_bits.shape
    E = Wr_bits.shape[0]
    r = MoERouter(T, H, E, k)
    x, Wr = G.bf16_dev(x_bits), G.bf16_dev(Wr_bits)
    idx, w = r.forward(x, Wr)
    out = dict(idx=idx, w=w, logits=r.logits.clone())
    if dtopk_w is not None:
        dx = (G.bf16_dev(dx_in) if dx_in is not None
              else torch.zeros((T, H), dtype=torch.bfloat16, device="cuda"))
        dW = r.backward(x, Wr, idx, w, torch.from_numpy(dtopk_w.astype(np.float32)).cuda(), dx)
        out.update(dx=dx, dW=dW, dlogits=r.dlogits.clone())
    torch.cuda.synchronize()
    return out


def check_selection(res, x, Wr, k):
    """The kernel's choice against the oracle's; returns the oracle's forward.  The
    selection (integers decided by floating point) is also taken in the kernel's
    precision: the oracle's rule on the kernel's fp32 logits must give exactly the
    kernel's topk_idx."""
    ro = orr.forward(x, Wr, k)
    s64 = ro["logits"]
    lg = res["logits"].double().cpu().numpy()
    assert np.abs(lg - s64).max() <= 1e-5 * np.abs(s64).max()
    idx = res["idx"].cpu().numpy().astype(np.int64)
    assert np.array_equal(orr.select_topk(lg, k), idx)
    # valid against the fp64 logits up to fp32 rounding; equal where no near-tie
    tol = 1e-5 * np.abs(s64).max()
    chosen = np.take_along_axis(s64, idx, axis=1)
    mask = np.ones_like(s64, dtype=bool)
    np.put_along_axis(mask, idx, False, axis=1)
    rest = np.where(mask, s64, -np.inf).max(axis=1) if k < s64.shape[1] else -np.inf
    assert np.all(chosen.min(axis=1) >= rest - tol)
    assert np.all(np.diff(chosen, axis=1) <= tol)
    same = np.all(idx == ro["topk_idx"], axis=1)
    w = res["w"].double().cpu().numpy()
    assert np.abs(w[same] - ro["topk_w"][same]).max(initial=0.0) <= 1e-5
    return ro, same


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


@pytest.mark.parametrize("T,H,E,k", [
    (300, 256, 16, 4), (1000, 512, 128, 8), (257, 256, 256, 8), (96, 128, 1024, 32),
    (64, 128, 8, 8),
    # dW_router's K (the tokens) split over clusters of 4 and 8 CTAs, shares of unequal
    # length; a partial M tile (E < 128) and a partial last N tile (H % 64 != 0)
    (4000, 256, 64, 4), (5000, 128, 128, 8), (3000, 200, 24, 4)])
def test_router_forward_backward(T, H, E, k):
    d = custom_inputs(T, H, 64, 8, 2, seed=T + E)
    rw = router_weights(E, H, seed=E)
    G_ = np.random.default_rng(T).standard_normal((T, k))
    res = run_router(d["x_bits"], rw["W_router_bits"], k, dtopk_w=G_)
    ro, same = check_selection(res, d["x"], rw["W_router"], k)
    assert same.all()                     # no near-tie at these seeds
    b = orr.backward(d["x"], rw["W_router"], ro["topk_idx"], ro["topk_w"], G_.astype(np.float32))
    assert rel(res["dlogits"].double().cpu().numpy(), b["dlogits"]) <= 1e-2
    assert rel(res["dW"].double().cpu().numpy(), b["dW_router"]) <= 1e-2
    assert rel(res["dx"].double().cpu().numpy(), b["dx"]) <= 1e-2


def test_router_ties_go_to_the_lower_index():
    T, H, E, k = 128, 128, 16, 4
    d = custom_inputs(T, H, 64, 8, 2, seed=3)
    rw = router_weights(E, H, seed=3)
    bits = rw["W_router_bits"].copy()
    bits[5] = bits[2]            # experts 2 and 5, 9 and 12 are identical: equal logits
    bits[12] = bits[9]
    res = run_router(d["x_bits"], bits, k)
    idx = res["idx"].cpu().numpy()
    lg = res["logits"].cpu().numpy()
    assert np.array_equal(lg[:, 5], lg[:, 2]) and np.array_equal(lg[:, 12], lg[:, 9])
    assert np.array_equal(orr.select_topk(lg.astype(np.float64), k), idx)
    # the oracle's own choice on the same tied weights (exact ties in fp64 too)
    Wt = rw["W_router"].copy()
    Wt[5], Wt[12] = Wt[2], Wt[9]
    assert np.array_equal(orr.forward(d["x"], Wt, k)["topk_idx"], idx)
    both = (np.isin(idx, [2]).any(axis=1)) & (np.isin(idx, [5]).any(axis=1))
    pos2 = np.argmax(idx == 2, axis=1)
    pos5 = np.argmax(idx == 5, axis=1)
    assert np.all(pos2[both] < pos5[both])
    only_one = np.isin(idx, [2, 5]).sum(axis=1) == 1
    assert np.all(~np.isin(idx[only_one], [5]))   # when one of the pair fits, it is 2


def test_router_dx_accumulates():
    T, H, E, k = 200, 256, 32, 4
    d = custom_inputs(T, H, 64, 8, 2, seed=5)
    rw = router_weights(E, H, seed=5)
    G_ = np.random.default_rng(6).standard_normal((T, k))
    res0 = run_router(d["x_bits"], rw["W_router_bits"], k, dtopk_w=G_)
    res1 = run_router(d["x_bits"], rw["W_router_bits"], k, dtopk_w=G_, dx_in=d["dy_bits"])
    want = res0["dx"].double().cpu().numpy() + d["dy"]
    assert rel(res1["dx"].double().cpu().numpy(), want) <= 1e-2


@pytest.mark.parametrize("routing_T", [512])
def test_router_then_layer_end_to_end(routing_T):
    T, H, I, E, k = routing_T, 256, 128, 16, 4
    d = custom_inputs(T, H, I, E, k, seed=7)
    rw = router_weights(E, H, seed=7)
    r = MoERouter(T, H, E, k)
    dev = G.upload(d)
    Wr = G.bf16_dev(rw["W_router_bits"])
    idx, w = r.forward(dev["x"], Wr)
    dev.update(topk_idx=idx, topk_w=w)
    res, layer, _ = G.run(dict(d, topk_idx=idx.cpu().numpy(), topk_w=w.cpu().numpy()), dev=dev)
    dWr = r.backward(dev["x"], Wr, idx, w, res["dtopk_w"], res["dx"])
    torch.cuda.synchronize()
    # oracles composed: the router's choice, the layer on it, the router's backward
    ro = orr.forward(d["x"], rw["W_router"], k)
    assert np.array_equal(ro["topk_idx"], idx.cpu().numpy())   # no near-ties at this seed
    f = oracle.forward(d["x"], ro["topk_idx"], ro["topk_w"], d["W_gate"], d["W_up"], d["W_down"])
    b = oracle.backward(d["dy"], d["x"], ro["topk_idx"], ro["topk_w"], d["W_gate"], d["W_up"],
                        d["W_down"], fwd=f)
    rb = orr.backward(d["x"], rw["W_router"], ro["topk_idx"], ro["topk_w"], b["dtopk_w"])
    assert rel(G.f32(res["y"]), f["y"]) <= 1e-2
    assert rel(G.f32(res["dx"]), b["dx"] + rb["dx"]) <= 1e-2
    assert rel(G.f32(dWr), rb["dW_router"]) <= 1e-2
    for key in ("dW_gate", "dW_up", "dW_down"):
        assert rel(G.f32(res[key]), b[key]) <= 1e-2


def test_router_full_size_sampled():
    T, H, E, k = 16384, 2048, 128, 8
    rng = np.random.default_rng(11)
    from mixture_experts_layer_16_gb300.inputs import bf16_bits, bf16_to_f32
    xb = bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    rw = router_weights(E, H, seed=11)
    G_ = rng.standard_normal((T, k))
    res = run_router(xb, rw["W_router_bits"], k, dtopk_w=G_)
    x = bf16_to_f32(xb).astype(np.float64)
    ro, same = check_selection(res, x, rw["W_router"], k)
    assert same.mean() > 0.999            # a near-tie may pick another valid expert
    b = orr.backward(x, rw["W_router"], ro["topk_idx"], ro["topk_w"], G_.astype(np.float32))
    assert rel(res["dW"].double().cpu().numpy(), b["dW_router"]) <= 1e-2
    toks = np.sort(rng.choice(np.nonzero(same)[0], 64, replace=False))
    assert rel(res["dx"].double().cpu().numpy()[toks], b["dx"][toks]) <= 1e-2
