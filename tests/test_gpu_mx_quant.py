"""The MXFP8 quantiser through the C ABI (mm_moe_mx_qdq) against the oracle's
mx_qdq, bit for bit: the e4m3 code and the block scale are integers decided by
floating point, and both sides decide them on the same bf16 input.

Inputs cover several binades per row, all-zero blocks, saturation (block maxima
with mantissa above 1.75, whose scaled value lies in (448, 512)) and exact ties
between neighbouring e4m3 values.  Values stay where every dequantised value is
at least 2^-133, so bf16 holds the result exactly."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_16_gb300 import binding as B
from oracle import mx as omx
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    G.ensure_built()


def bf16_round_np(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).double().numpy()


def make(rows, cols, seed, axis=1):
    """bf16 values whose blocks run along `axis`: binades spread far across blocks
    (from 2^-40 to 2^40) and a little within them."""
    if axis == 0:
        return np.ascontiguousarray(make(cols, rows, seed, 1).T)
    rng = np.random.default_rng(seed)
    nb = -(-cols // 32)
    binade = rng.integers(-40, 40, size=(rows, nb)).repeat(32, axis=1)[:, :cols]
    v = rng.standard_normal((rows, cols)) * np.exp2(binade)
    v *= np.exp2(rng.integers(-6, 7, size=(1, cols)))          # binades within a block
    v[rng.random((rows, cols)) < 0.02] = 0.0
    if rows >= 64 and cols >= 64:
        v[32:64, 32:64] = 0.0                                  # all-zero blocks
    # exact ties: 1.0625 lies halfway between the e4m3 values 1.0 and 1.125 (block
    # maximum 256 sets the scale to 2^0); a block maximum of 1.9 * 2^9 saturates
    # (1.9 * 2^8 > 448 after scaling)
    if rows >= 32 and cols >= 96:
        v[0:32, 64:96] = 1.0625 * np.sign(rng.standard_normal((32, 32)))
        v[0:32, 64] = 256.0
        v[5, 70] = 1.9 * 2 ** 9
        v[6, 64:96] = 1.0625 * np.sign(rng.standard_normal(32))
        v[6, 64] = 256.0
    return bf16_round_np(v)


# blocks down columns need rows % 32 == 0 (every shape here), blocks along rows
# cols % 32 == 0 (not the last shape)
QUANT_CASES = [(rows, cols, axis)
               for rows, cols in [(64, 128), (96, 2048), (4096, 768), (32, 8 * 37)]
               for axis in (0, 1) if not (axis == 1 and cols % 32)]


@pytest.mark.parametrize("rows,cols,axis", QUANT_CASES)
def test_quantiser_bit_exact(rows, cols, axis):
    v = make(rows, cols, seed=rows + cols + axis, axis=axis)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    out = torch.empty_like(t)
    B.mm_moe_mx_qdq(t, out, axis)
    torch.cuda.synchronize()
    want = omx.mx_qdq(v, axis)
    got = out.double().cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], want[tuple(bad[0])])


def test_quantiser_in_place_and_idempotent():
    v = make(128, 256, seed=3)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    B.mm_moe_mx_qdq(t, t, 1)
    once = t.clone()
    B.mm_moe_mx_qdq(t, t, 1)
    torch.cuda.synchronize()
    assert torch.equal(once, t)
    assert np.array_equal(once.double().cpu().numpy(), omx.mx_qdq(v, 1))


def test_quantiser_rejects_bad_shapes():
    t = torch.zeros((40, 48), dtype=torch.bfloat16, device="cuda")
    lib = B.lib()
    assert lib.mm_moe_mx_qdq(t.data_ptr(), t.data_ptr(), 40, 48, 1, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_qdq(t.data_ptr(), t.data_ptr(), 40, 48, 0, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_qdq(t.data_ptr(), t.data_ptr(), 40, 48, 2, None) == B.MM_MOE_EINVAL


# ---------------------------------------------------------------- e4m3 codes + scales
def scale_offset(mn, kb, n_mn):
    """Byte of the scale code of (operand row mn, k-block kb) in the arrangement the
    block-scaled tensor cores take: 512-byte atoms of 128 rows x 4 k-blocks (row mn % 32
    of 16 bytes, word (mn // 32) % 4, byte kb % 4), atoms of one 4-block group side by
    side over the n_mn // 128 row blocks."""
    return (((kb // 4) * (n_mn // 128) + mn // 128) * 512 + (mn % 32) * 16
            + ((mn // 32) % 4) * 4 + kb % 4)


@pytest.mark.parametrize("rows,cols,axis", [(128, 256, 1), (128, 256, 0), (384, 2048, 1),
                                            (384, 2048, 0), (4096, 768, 1), (4096, 768, 0)])
def test_quantize_codes_and_scales_bit_exact(rows, cols, axis):
    """mm_moe_mx_quantize (the form the MXFP8 GEMMs read) against the oracle: every
    scale code is e8m0(floor(log2 amax) - 8) of its block, and every element's e4m3
    code (decoded by torch's float8_e4m3fn) times its block scale is the oracle's
    quantised value, bit for bit."""
    v = make(rows, cols, seed=7 * rows + cols + axis, axis=axis)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    codes = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows * cols // 32, dtype=torch.uint8, device="cuda")
    B.mm_moe_mx_quantize(t, codes, scales, axis)
    torch.cuda.synchronize()
    elem = codes.cpu().view(torch.float8_e4m3fn).double().numpy()
    sc = scales.cpu().numpy().astype(np.int64)
    r = np.arange(rows)[:, None]
    c = np.arange(cols)[None, :]
    mn, kb, n_mn = (r, c // 32, rows) if axis == 1 else (c, r // 32, cols)
    s = sc[scale_offset(mn, kb, n_mn)]                       # per element
    # scale codes: the oracle's block exponent + 127
    blocks = np.moveaxis(v, axis, -1)
    blocks = blocks.reshape(blocks.shape[:-1] + (blocks.shape[-1] // 32, 32))
    want_e = omx.e8m0_scale_exponent(np.abs(blocks).max(axis=-1)) + 127
    want_s = np.repeat(want_e, 32, axis=-1)
    want_s = np.moveaxis(want_s, -1, axis) if axis == 0 else want_s
    assert np.array_equal(s, want_s)
    got = elem * np.exp2(s.astype(np.float64) - 127)
    want = omx.mx_qdq(v, axis)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], want[tuple(bad[0])])


def test_quantize_rejects_bad_shapes():
    t = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")
    u = torch.zeros((128, 96), dtype=torch.uint8, device="cuda")
    lib = B.lib()
    assert lib.mm_moe_mx_quantize(t.data_ptr(), u.data_ptr(), u.data_ptr(), 128, 96, 1,
                                  None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_quantize(t.data_ptr(), u.data_ptr(), u.data_ptr(), 128, 128, 2,
                                  None) == B.MM_MOE_EINVAL
