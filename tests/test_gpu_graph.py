"""A whole layer step (forward and backward through the C ABI) captured in a CUDA graph.

The library makes no host synchronisation and no allocation inside forward or
backward, and its side stream joins through events, so the step can be recorded once
and replayed.  A replay must give, bit for bit, what eager calls give on the same
inputs (the kernels are deterministic), also after new inputs are copied into the
captured buffers; the status word must stay clean.  The eager results are pinned to
the oracle by the parity tests."""
import pytest
import torch

from mixture_experts_layer_16_gb300 import MoELayer
from mixture_experts_layer_16_gb300.inputs import custom_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu
OUTS = ("y", "dx", "dW_gate", "dW_up", "dW_down", "dtopk_w")


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def eager(layer, dev):
    y = layer.forward(dev["x"], dev["topk_idx"], dev["topk_w"], dev["W_gate"], dev["W_up"],
                      dev["W_down"])
    out = layer.backward(dev["dy"], dev["W_gate"], dev["W_up"], dev["W_down"], x=dev["x"])
    torch.cuda.synchronize()
    return dict(zip(OUTS, (y,) + tuple(out)))


@pytest.mark.parametrize("prec,recompute", [("bf16", False), ("mxfp8", False),
                                            ("fp8_block", False), ("bf16", True)])
def test_step_replays_in_a_cuda_graph(prec, recompute):
    T, H, I, E, k = 1000, 512, 256, 16, 4         # SM-pair tiles, one joint wgrad launch
    d1 = custom_inputs(T, H, I, E, k, seed=61, routing="zipf")
    d2 = custom_inputs(T, H, I, E, k, seed=62, routing="uniform")
    layer = MoELayer(T, H, I, E, k, prec, recompute=recompute)
    dev1, dev2 = G.upload(d1), G.upload(d2)
    want1 = {n: t.clone() for n, t in eager(layer, dev1).items()}
    want2 = {n: t.clone() for n, t in eager(layer, dev2).items()}

    # captured buffers: inputs are copied in, outputs are read out
    cap = {n: t.clone() for n, t in dev1.items()}
    y = torch.empty_like(want1["y"])
    out = tuple(torch.empty_like(want1[n]) for n in OUTS[1:])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture's side of the device
        layer.forward(cap["x"], cap["topk_idx"], cap["topk_w"], cap["W_gate"], cap["W_up"],
                      cap["W_down"], y=y)
        layer.backward(cap["dy"], cap["W_gate"], cap["W_up"], cap["W_down"], out=out, x=cap["x"])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(cap["x"], cap["topk_idx"], cap["topk_w"], cap["W_gate"], cap["W_up"],
                      cap["W_down"], y=y)
        layer.backward(cap["dy"], cap["W_gate"], cap["W_up"], cap["W_down"], out=out, x=cap["x"])

    for dev, want in ((dev2, want2), (dev1, want1), (dev2, want2)):
        for n in cap:
            cap[n].copy_(dev[n])
        for t in (y,) + out:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = dict(zip(OUTS, (y,) + out))
        bad = [n for n in OUTS if not torch.equal(got[n], want[n])]
        assert not bad, bad
        assert layer.status() == 0
