"""The A-multicast form of the grouped GEMMs (MM_MOE_MULTICAST): clusters of two SM
pairs take N tiles 2j and 2j + 1 of one M tile in step and share its A rows by TMA
multicast.  Its products are the same MMAs in the same order as the default SM-pair
kernels', so every output must match the default path bit for bit, and the oracle
within the BF16 bound; a stalled stage must unwind all four CTAs of a cluster and leave
the layer usable (the failure form of tests/test_gpu_failure.py)."""
import pytest
import torch

from mixture_experts_layer_16_gb300 import binding as B
from mixture_experts_layer_16_gb300.inputs import CONFIGS, custom_inputs, make_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

KEYS = ("y", "dx", "dW_gate", "dW_up", "dW_down", "dtopk_w")


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _same_bits(a, b):
    for key in KEYS:
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("T,H,I,E,k,routing,seed", [
    (1200, 512, 512, 8, 2, "uniform", 20),     # all four grouped GEMMs: two N tiles
    (900, 512, 256, 32, 8, "zipf_trunc", 14),  # empty experts; dgrad-down one N tile
    (3, 512, 256, 4, 2, "uniform", 18),        # pair tiles holding 1-2 rows
    (2100, 1024, 768, 16, 4, "zipf", 21),      # gate/up six N tiles, down four
])
def test_multicast_matches_oracle_and_default(T, H, I, E, k, routing, seed):
    kw = dict(zipf_ranks=max(k, E - 4)) if routing == "zipf_trunc" else {}
    d = custom_inputs(T, H, I, E, k, seed=seed, routing=routing, **kw)
    ref, _, dev = G.run(d)
    mc, _, _ = G.run(d, dev=dev, multicast=True)
    assert mc["status"] == 0
    G.check_routing(mc, d["topk_idx"], E)
    G.check_full(d, mc)
    _same_bits(mc, ref)


def test_multicast_full_size():
    # the benchmark workload: gate/up, down and dgrad-gate/up on four-CTA clusters; the
    # default path's outputs on these inputs are checked against the oracle by
    # tests/test_gpu_parity.py, and the multicast path must reproduce them exactly
    cfg = CONFIGS["qwen3_30b_16k_zipf"]
    d = make_inputs(cfg)
    ref, _, dev = G.run(d)
    mc, _, _ = G.run(d, dev=dev, multicast=True)
    assert ref["status"] == 0 and mc["status"] == 0
    G.check_routing(mc, d["topk_idx"], cfg.E)
    _same_bits(mc, ref)


def test_stalled_stage_unwinds_four_cta_clusters(monkeypatch):
    # gate/up has two N tiles (I = 256): clusters of two pairs.  The stalled stage is
    # CTA 0's, whose A half also feeds the other pair: both pairs' MMA issuers time out,
    # the abort reaches all four CTAs, and they meet at the final cluster barrier.
    d = custom_inputs(512, 512, 256, 8, 2, seed=43)
    monkeypatch.setenv("MM_MOE_TEST_STALL_GEMM", "0")
    res, layer, dev = G.run(d, backward=False, multicast=True)
    assert res["status"] == B.MM_MOE_ETIMEOUT
    monkeypatch.delenv("MM_MOE_TEST_STALL_GEMM")
    res2, _, _ = G.run(d, layer=layer, dev=dev)
    assert res2["status"] == B.MM_MOE_OK
    G.check_routing(res2, d["topk_idx"], 8)
    G.check_full(d, res2)
