"""Blockwise FP8 on the GPU (MM_MOE_FP8_BLOCK, and its quantisers mm_moe_fp8_block_qdq and
mm_moe_fp8_block_quantize)
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
from tests.test_gpu_mx_quant import make, scale_offset

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


@pytest.mark.parametrize("rows,cols,layout", [(128, 256, 0), (128, 256, 1), (128, 256, 2),
                                              (384, 2048, 0), (384, 2048, 1), (384, 2048, 2),
                                              (4096, 768, 0), (4096, 768, 1), (4096, 768, 2)])
def test_quantize_codes_and_scales_bit_exact(rows, cols, layout):
    """mm_moe_fp8_block_quantize (the form the blockwise GEMMs read on the block-scaled
    tensor cores) against the oracle: every scale code is ceil(log2(amax / 448)) + 127
    of its 128-block (its tile for layout 2, in both arrangements), repeated over the
    block's 32-element scale blocks, and every element's e4m3 code (decoded by torch's
    float8_e4m3fn) times its scale is the oracle's quantised value, bit for bit."""
    v = make(rows, cols, seed=11 * rows + cols + layout, axis=0 if layout == 1 else 1)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    codes = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    n = rows * cols // 32
    scales = torch.empty(n * (2 if layout == 2 else 1), dtype=torch.uint8, device="cuda")
    B.mm_moe_fp8_block_quantize(t, codes, scales, layout)
    torch.cuda.synchronize()
    elem = codes.cpu().view(torch.float8_e4m3fn).double().numpy()
    sc = scales.cpu().numpy().astype(np.int64)
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    if layout == 0:
        amax = np.abs(v.reshape(rows, cols // 128, 128)).max(axis=-1)
        want_e = fb.ue8m0_ceil_exponent(amax).repeat(128, axis=1)
        arrangements = [(r, c // 32, rows, 0)]
        want = fb.qdq_1d(v, 1)
    elif layout == 1:
        amax = np.abs(v.reshape(rows // 128, 128, cols)).max(axis=1)
        want_e = fb.ue8m0_ceil_exponent(amax).repeat(128, axis=0)
        arrangements = [(c, r // 32, cols, 0)]
        want = fb.qdq_1d(v, 0)
    else:
        amax = np.abs(v.reshape(rows // 128, 128, cols // 128, 128)).max(axis=(1, 3))
        want_e = fb.ue8m0_ceil_exponent(amax).repeat(128, axis=0).repeat(128, axis=1)
        arrangements = [(r, c // 32, rows, 0), (c, r // 32, cols, n)]
        want = fb.qdq_2d(v)
    for mn, kb, n_mn, base in arrangements:
        s = sc[base + scale_offset(mn, kb, n_mn)]           # per element
        assert np.array_equal(s, want_e + 127), (layout, base)
    s = sc[scale_offset(*arrangements[0][:3])]
    got = elem * np.exp2(s.astype(np.float64) - 127)
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
