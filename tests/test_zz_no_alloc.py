"""The routing entry point that allocates nothing (mm_moe_route_noalloc).

Some callers cannot allocate device memory at the moment they route tokens; this
entry point keeps its working memory in a fixed array inside the library.  Here it
is called through the C ABI twice in a row, on different routings, and each
result must equal both the routing the regular forward pass exports and the
oracle's stable counting sort (bit for bit: the outputs are integers).  One more
case runs at the documented limits (T * k = 262,144 routed rows over 256 experts).
The file sorts last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_16_gb300 import binding as B
from mixture_experts_layer_16_gb300.inputs import custom_inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def _noalloc(d, T, E, k):
    dev = "cuda"
    idx = torch.from_numpy(np.ascontiguousarray(d["topk_idx"], dtype=np.int32)).to(dev)
    w = torch.from_numpy(np.ascontiguousarray(d["topk_w"], dtype=np.float32)).to(dev)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((T * k,), -7, dtype=torch.int32, device=dev)
    B.mm_moe_route_noalloc(B.make_shape(T, 128, 64, E, k), idx, w, off, perm, inv)
    torch.cuda.synchronize()
    return off, perm, inv


def _check_oracle(off, perm, inv, topk_idx, E):
    _, offsets, p, i = oracle.route(topk_idx, E)
    assert np.array_equal(off.cpu().numpy(), offsets.astype(np.int32))
    assert np.array_equal(perm.cpu().numpy(), p.astype(np.int32))
    assert np.array_equal(inv.cpu().numpy(), i.astype(np.int32))


def test_noalloc_routing_matches_forward_twice():
    cases = [(3000, 256, 128, 64, 8, "zipf", 21), (1777, 256, 128, 48, 4, "uniform", 22)]
    for T, H, I, E, k, routing, seed in cases:          # two calls in a row
        d = custom_inputs(T, H, I, E, k, seed=seed, routing=routing)
        ref, _, _ = G.run(d, backward=False)            # the existing entry point
        off, perm, inv = _noalloc(d, T, E, k)
        assert torch.equal(off, ref["offsets"])
        assert torch.equal(perm, ref["perm"])
        assert torch.equal(inv, ref["inv"])
        _check_oracle(off, perm, inv, d["topk_idx"], E)


def test_noalloc_routing_at_its_limits():
    # T * k = 262,144 rows over E = 256 experts, Zipf-skewed: the largest sizes the
    # fixed array holds, against the oracle
    T, E, k = 32768, 256, 8
    rng = np.random.default_rng(23)
    p = 1.0 / np.arange(1, E + 1) ** 1.2
    g = np.log(p)[None, :] + rng.gumbel(size=(T, E))          # Gumbel-top-k draws
    idx = np.argsort(-g, axis=1)[:, :k].astype(np.int32)
    idx = rng.permutation(E).astype(np.int32)[idx]
    d = {"topk_idx": idx, "topk_w": np.full((T, k), 1.0 / k, np.float32)}
    off, perm, inv = _noalloc(d, T, E, k)
    _check_oracle(off, perm, inv, idx, E)


def test_noalloc_rejects_sizes_beyond_its_limit():
    z = torch.zeros(8, dtype=torch.int32, device="cuda")
    f = torch.zeros(8, dtype=torch.float32, device="cuda")
    for shape in (B.make_shape(65537, 128, 64, 64, 4), B.make_shape(16, 128, 64, 257, 2)):
        with pytest.raises(B.MoEError) as ei:
            B.mm_moe_route_noalloc(shape, z, f, z, z, z)
        assert ei.value.status == B.MM_MOE_EINVAL
