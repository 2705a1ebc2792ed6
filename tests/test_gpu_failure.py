"""Failure detection on the GPU without a fault: a bounded wait is made to run out and
the layer must report it and stay usable.

MM_MOE_TEST_STALL_GEMM=0 makes the gate/up GEMM's first pipeline stage on CTA 0 never
fill (its barrier is armed, no copy is issued).  The MMA issuer's wait gives up after
its limit (2 s), every role of the kernel unwinds with bounded waits, the status word
reads MM_MOE_ETIMEOUT, and the CUDA context is fine: the same layer then runs the
forward and backward again and matches the oracle.  Both tile forms are covered:
single-SM tiles (H = 128) and SM pairs (H = 256, I = 128), where the CTA whose wait
ran out also stops its peer and both drain within one shared time budget."""
import pytest
import torch

from mixture_experts_layer_16_gb300 import binding as B
from mixture_experts_layer_16_gb300.inputs import custom_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def test_stalled_stage_reports_timeout_and_context_survives(monkeypatch):
    d = custom_inputs(256, 128, 64, 8, 2, seed=41)
    monkeypatch.setenv("MM_MOE_TEST_STALL_GEMM", "0")
    res, layer, dev = G.run(d, backward=False)
    assert res["status"] == B.MM_MOE_ETIMEOUT
    monkeypatch.delenv("MM_MOE_TEST_STALL_GEMM")
    res2, _, _ = G.run(d, layer=layer, dev=dev)
    assert res2["status"] == B.MM_MOE_OK
    G.check_routing(res2, d["topk_idx"], 8)
    G.check_full(d, res2)
    assert torch.cuda.is_available()


def test_stalled_stage_on_sm_pairs_unwinds_and_context_survives(monkeypatch):
    # H % 256 == 0 and I % 128 == 0: the GEMMs run on SM pairs.  The stalled stage
    # belongs to the pair's first CTA; the MMA issuer's wait runs out, the abort
    # reaches the peer CTA, both drain within one shared budget and meet at the final
    # cluster barrier.
    d = custom_inputs(512, 256, 128, 8, 2, seed=42)
    monkeypatch.setenv("MM_MOE_TEST_STALL_GEMM", "0")
    res, layer, dev = G.run(d, backward=False)
    assert res["status"] == B.MM_MOE_ETIMEOUT
    monkeypatch.delenv("MM_MOE_TEST_STALL_GEMM")
    res2, _, _ = G.run(d, layer=layer, dev=dev)
    assert res2["status"] == B.MM_MOE_OK
    G.check_routing(res2, d["topk_idx"], 8)
    G.check_full(d, res2)
