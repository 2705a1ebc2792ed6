"""CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Bar: routing (offsets, perm, inv) bit-exact; every float output within
max|gpu - oracle| / max|oracle| <= 1e-2 (bf16 storage of h, a, slots and outputs
with fp32 accumulation; 1e-2 is the bound the layer's specification states).
Small shapes are compared element by element; the full-size workloads on
sampled tokens and sampled experts, which the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.moe as om
from mixture_experts_layer_16_gb300.inputs import CONFIGS, custom_inputs, make_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


check_routing = G.check_routing


def check_full(d, res, backward=True, tol=TOL):
    return G.check_full(d, res, backward, tol)


SMALL = [
    # (T, H, I, E, k, routing, seed): several tiles, ragged tails, every BN variant
    (64, 128, 64, 8, 2, "uniform", 1),       # the tiny workload's shape
    (300, 256, 192, 8, 2, "uniform", 2),     # I=192: 64-wide N tiles for the I dimension
    (1000, 384, 128, 16, 4, "uniform", 3),   # H=384: 128-wide N tiles for the H dimension
    (777, 512, 256, 32, 8, "zipf", 4),       # skewed routing
    (513, 256, 64, 12, 3, "zipf_trunc", 5),  # some experts receive no token
    # SM-pair tiles (H % 256 == 0, I % 128 == 0); experts padded to 256 rows; the
    # weight-gradient GEMMs run on pairs from 512 routed rows per expert on average
    (600, 256, 128, 8, 2, "uniform", 11),    # 128-wide pair tiles over I, single-SM wgrad
    (2200, 512, 384, 16, 4, "zipf", 12),     # I = 384: 128-wide pair tiles; pair wgrad
    (2100, 768, 256, 8, 2, "uniform", 13),   # three 256-wide N tiles over H; pair wgrad
    (900, 512, 256, 32, 8, "zipf_trunc", 14),  # pairs with empty experts
    (1200, 512, 512, 8, 2, "uniform", 20),  # two 256-wide N tiles in all four grouped GEMMs
]


@pytest.mark.parametrize("T,H,I,E,k,routing,seed", SMALL)
def test_small_parity(T, H, I, E, k, routing, seed):
    kw = dict(zipf_ranks=max(k, E - 4)) if routing == "zipf_trunc" else {}
    d = custom_inputs(T, H, I, E, k, seed=seed, routing=routing, **kw)
    res, _, _ = G.run(d)
    assert res["status"] == 0
    check_routing(res, d["topk_idx"], E)
    check_full(d, res)


def test_tiny_config():
    d = make_inputs(CONFIGS["tiny"])
    res, _, _ = G.run(d)
    assert res["status"] == 0
    check_routing(res, d["topk_idx"], CONFIGS["tiny"].E)
    check_full(d, res)


def test_all_tokens_one_expert_and_empty_experts():
    T, H, I, E, k = 400, 256, 128, 6, 1
    idx = np.full((T, 1), 4, dtype=np.int32)
    d = custom_inputs(T, H, I, E, k, seed=7, idx=idx)
    res, _, _ = G.run(d)
    check_routing(res, d["topk_idx"], E)
    errs = check_full(d, res)
    for e in (0, 1, 2, 3, 5):   # experts with no token: exact zeros
        for key in ("dW_gate", "dW_up", "dW_down"):
            assert torch.count_nonzero(res[key][e]).item() == 0
    assert errs["y"] <= TOL


def test_k1_unit_weight():
    """k = 1 with weight 1: the dense SwiGLU MLP of each token's expert."""
    T, H, I, E = 256, 128, 64, 4
    rng = np.random.default_rng(0)
    idx = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    d = custom_inputs(T, H, I, E, 1, seed=8, idx=idx)
    d["topk_w"] = np.ones((T, 1), dtype=np.float32)
    res, _, _ = G.run(d)
    check_full(d, res)


@pytest.mark.parametrize("T,H,I,E,k,routing,seed", [
    (1, 256, 128, 128, 8, "uniform", 15),     # one token: 8 experts with one row, 120 empty
    (300, 128, 64, 1024, 4, "uniform", 16),   # the largest expert count
    (40, 128, 64, 8, 8, "uniform", 17),       # k = E: every token goes to every expert
    (3, 512, 256, 4, 2, "uniform", 18),       # SM-pair tiles holding 1-2 rows
    (50, 128, 64, 16, 12, "uniform", 19),     # k > 8: the combine's general loop
])
def test_degenerate_shapes(T, H, I, E, k, routing, seed):
    d = custom_inputs(T, H, I, E, k, seed=seed, routing=routing)
    res, _, _ = G.run(d)
    assert res["status"] == 0
    check_routing(res, d["topk_idx"], E)
    check_full(d, res)


@pytest.mark.parametrize("T,E,k,how", [
    (65536, 1024, 8, "uniform"),   # 524,288 routed rows over 1,024 experts (256 routing blocks)
    (65536, 128, 1, "one"),        # every token to one expert: a 512-tile expert
    (50000, 256, 4, "zipf"),       # skewed, ragged row count
])
def test_routing_large(T, E, k, how):
    """Routing alone at sizes far above the parity shapes (H and I minimal): offsets,
    perm and inv bit-exact, y still within tolerance on sampled tokens."""
    H, I = 128, 64
    rng = np.random.default_rng(T + E + k)
    if how == "one":
        idx = np.full((T, 1), 77, dtype=np.int32)
        d = custom_inputs(T, H, I, E, k, seed=60, idx=idx)
    else:
        d = custom_inputs(T, H, I, E, k, seed=61, routing=how)
    res, _, _ = G.run(d, backward=False)
    assert res["status"] == 0
    check_routing(res, d["topk_idx"], E)
    toks = np.sort(rng.choice(T, 64, replace=False))
    sub = om.token_subset(d, toks)
    f = oracle.forward(sub["x"], sub["topk_idx"], sub["topk_w"], d["W_gate"], d["W_up"],
                       d["W_down"])
    assert G.rel_err(G.f32(res["y"][toks]), f["y"]) <= TOL


def test_determinism():
    d = custom_inputs(700, 256, 128, 16, 4, seed=9, routing="zipf")
    r1, layer, dev = G.run(d)
    snap = {k: v.clone() for k, v in r1.items() if isinstance(v, torch.Tensor)}
    r2, _, _ = G.run(d, layer=layer, dev=dev)
    for k, v in snap.items():
        assert torch.equal(v, r2[k]), k


def test_bad_expert_index_reports_status():
    """An index outside [0, E) is reported (MM_MOE_EBADIDX), dropped, and faults nothing."""
    d = custom_inputs(128, 128, 64, 8, 2, seed=10)
    d["topk_idx"][5, 1] = 8
    d["topk_idx"][9, 0] = -3
    res, layer, _ = G.run(d, backward=False)
    assert res["status"] == 3
    # the valid pairs are still routed and placed
    off = res["offsets"].cpu().numpy()
    assert off[-1] == 128 * 2 - 2


# ---------------------------------------------------------------- full-size workloads
def sampled_check(name, n_tokens=48, seed=0):
    return G.sampled_check(name, TOL, n_tokens, seed)


def test_full_qwen3_30b_4k():
    sampled_check("qwen3_30b_4k")


def test_full_qwen3_30b_16k_zipf():
    sampled_check("qwen3_30b_16k_zipf")


def test_full_qwen3_30b_16k_zipf_empty():
    sampled_check("qwen3_30b_16k_zipf_empty")


@pytest.mark.slow
def test_full_qwen3_235b_8k():
    sampled_check("qwen3_235b_8k", n_tokens=24)
