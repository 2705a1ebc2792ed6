"""MM_MOE_RECOMPUTE (activation checkpointing) on the GPU: the forward keeps only the
routing, the backward re-permutes x and re-runs the gate/up GEMM.  The kernels are
deterministic, so every output must equal the mode that keeps its activations bit
for bit, in each precision; the parity of that mode against the oracle is covered by
test_gpu_parity.py and test_gpu_mx.py."""
import pytest
import torch

from mixture_experts_layer_16_gb300 import MoELayer
from mixture_experts_layer_16_gb300.inputs import CONFIGS, custom_inputs, make_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
KEYS = ("y", "dx", "dW_gate", "dW_up", "dW_down", "dtopk_w", "offsets", "perm", "inv")


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def same(a, b):
    bad = [k for k in KEYS if not torch.equal(a[k], b[k])]
    assert not bad, bad


@pytest.mark.parametrize("prec", ["bf16", "mxfp8", "fp8_bwd", "fp8_block"])
@pytest.mark.parametrize("T,H,I,E,k,routing,seed", [
    (300, 384, 128, 8, 2, "uniform", 31),      # single-SM tiles
    (900, 512, 256, 32, 8, "zipf_trunc", 32),  # SM pairs, empty experts
])
def test_recompute_matches_kept_activations(T, H, I, E, k, routing, seed, prec):
    kw = dict(zipf_ranks=max(k, E - 4)) if routing == "zipf_trunc" else {}
    d = custom_inputs(T, H, I, E, k, seed=seed, routing=routing, **kw)
    keep, _, dev = G.run(d, prec=prec)
    rc, layer, _ = G.run(d, dev=dev, prec=prec, recompute=True)
    assert keep["status"] == 0 and rc["status"] == 0
    same(keep, rc)


def test_recompute_full_size():
    cfg = CONFIGS["qwen3_30b_16k_zipf"]
    d = make_inputs(cfg)
    keep, _, dev = G.run(d)
    rc, _, _ = G.run(d, dev=dev, recompute=True)
    same(keep, rc)


def test_recompute_backward_needs_x():
    layer = MoELayer(64, 128, 64, 8, 2, recompute=True)
    dy = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((8, 64, 128), dtype=torch.bfloat16, device="cuda")
    Wd = torch.zeros((8, 128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        layer.backward(dy, W, W, Wd)
