"""Blockwise FP8 on the GPU (MM_MOE_FP8_BLOCK, and its quantiser mm_moe_fp8_block_qdq)
against the oracle's blockwise FP8 mode (oracle/fp8block.py): power-of-two scale
2^ceil(log2(amax / 448)) per block, activations in 128-element blocks along each
GEMM's K (128-row token blocks for the weight gradients), weights in 128 x 128 blocks.

Bar: the quantiser bit for bit (the e4m3 codes and scales are integers decided on the
same bf16 inputs); routing bit-exact; float outputs within 5e-2 of the oracle's maximum,
the FP8 bound of the layer's specification; the quantised outputs follow this oracle
and not the BF16 one."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_16_gb300 import binding as B
from mixture_experts_layer_16_gb300.inputs import custom_inputs
from oracle import fp8block as fb
from tests import gpu_util as G
from tests.test_gpu_mx_quant import make

pytestmark = pytest.mark.gpu
TOL = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


# every (shape, layout) pair whose blocks are whole: rows along a row need
# cols % 128 == 0, blocks down a column rows % 128 == 0, tiles both
QUANT_CASES = [(rows, cols, layout)
               for rows, cols in [(128, 256), (384, 2048), (4096, 768), (256, 8 * 37)]
               for layout in (0, 1, 2)
               if not ((layout in (0, 2) and cols % 128) or (layout in (1, 2) and rows % 128))]


@pytest.mark.parametrize("rows,cols,layout", QUANT_CASES)
def test_quantiser_bit_exact(rows, cols, layout):
    v = make(rows, cols, seed=rows + cols + layout, axis=0 if layout == 1 else 1)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    out = torch.empty_like(t)
    B.mm_moe_fp8_block_qdq(t, out, layout)
    torch.cuda.synchronize()
    want = fb.qdq_2d(v) if layout == 2 else fb.qdq_1d(v, 1 if layout == 0 else 0)
    got = out.double().cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], want[tuple(bad[0])])


SMALL = [
    # (T, H, I, E, k, routing, seed): I % 128 == 0 (128 x 128 weight blocks)
    (300, 128, 128, 8, 2, "uniform", 51),       # single-SM tiles
    (1000, 384, 128, 16, 4, "uniform", 52),     # 128-wide N tiles over H, ragged tails
    (900, 512, 256, 32, 8, "zipf_trunc", 53),   # SM pairs, empty experts
    (2200, 512, 384, 16, 4, "zipf", 54),        # pair weight-gradient tiles
]


@pytest.mark.parametrize("T,H,I,E,k,routing,seed", SMALL)
def test_small_parity(T, H, I, E, k, routing, seed):
    kw = dict(zipf_ranks=max(k, E - 4)) if routing == "zipf_trunc" else {}
    d = custom_inputs(T, H, I, E, k, seed=seed, routing=routing, **kw)
    res, _, _ = G.run(d, prec="fp8_block")
    assert res["status"] == 0
    G.check_routing(res, d["topk_idx"], E)
    errs = G.check_full(d, res, tol=TOL, prec="fp8_block")
    ref_bf16 = G.full_errors(d, res, prec="bf16")
    for key in ("y", "dx"):
        assert errs[key] < 0.5 * ref_bf16[key], (key, errs[key], ref_bf16[key])


def test_rejects_I_not_multiple_of_128():
    with pytest.raises(B.MoEError):
        B.mm_moe_workspace_size(B.make_shape(64, 128, 64, 8, 2, "fp8_block"))


def test_full_qwen3_30b_16k_fp8block():
    G.sampled_check("qwen3_30b_16k_fp8block", TOL)
