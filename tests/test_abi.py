"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a,
loads, exports every symbol the header declares, and rejects invalid arguments
before anything touches a device."""
import ctypes
import os
import re
import subprocess

import pytest

from mixture_experts_layer_16_gb300 import binding as B
from mixture_experts_layer_16_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.lib()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            names |= set(re.findall(r"MM_MOE_API\s+[\w\s\*]+?\b(mm_moe_\w+)\s*\(", src))
    return names


def test_exports_match_header(lib):
    decl = declared_symbols()
    assert decl == set(B.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mm_moe_\w+)", out))
    assert decl <= exported
    for name in decl:
        assert getattr(lib, name) is not None


def test_option_bits_match_header():
    src = open(os.path.join(ROOT, "include", "mm_moe.h")).read()
    bits = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (MM_MOE_\w+) (\d+)", src)}
    assert bits["MM_MOE_RECOMPUTE"] == B.MM_MOE_RECOMPUTE
    assert bits["MM_MOE_MULTICAST"] == B.MM_MOE_MULTICAST
    s = B.make_shape(64, 128, 64, 8, 2, recompute=True, multicast=True)
    assert s.flags == B.MM_MOE_RECOMPUTE | B.MM_MOE_MULTICAST


def test_multicast_option_is_accepted(lib):
    # a valid option bit: the workspace sizes do not depend on it
    a = B.mm_moe_workspace_size(B.make_shape(1024, 512, 256, 8, 2))
    b = B.mm_moe_workspace_size(B.make_shape(1024, 512, 256, 8, 2, multicast=True))
    assert a == b


def test_workspace_size_and_shape_validation(lib):
    sc, sv = B.mm_moe_workspace_size(B.make_shape(16384, 2048, 768, 128, 8))
    assert sc > 0 and sv > 0
    # the saved buffer holds x_perm and h at least: (ceil(R/128)+E)*128 padded rows
    Rp = (16384 * 8 // 128 + 128) * 128
    assert sv >= Rp * (2048 + 2 * 768) * 2
    for bad in [(0, 128, 64, 8, 2), (64, 100, 64, 8, 2), (64, 128, 48, 8, 2), (64, 128, 64, 8, 9),
                (64, 128, 64, 2048, 2), (64, 128, 64, 8, 0)]:
        with pytest.raises(B.MoEError) as ei:
            B.mm_moe_workspace_size(B.make_shape(*bad))
        assert ei.value.status == B.MM_MOE_EINVAL
    s = B.make_shape(64, 128, 64, 8, 2)
    s.flags = 4                                    # an undefined option bit
    with pytest.raises(B.MoEError):
        B.mm_moe_workspace_size(s)


def test_workspace_sizes_by_mode(lib):
    """MXFP8 modes need more scratch; recompute keeps only the routing in saved."""
    shp = (16384, 2048, 768, 128, 8)
    sc_b, sv_b = B.mm_moe_workspace_size(B.make_shape(*shp))
    sc_m, sv_m = B.mm_moe_workspace_size(B.make_shape(*shp, "mxfp8"))
    sc_f, sv_f = B.mm_moe_workspace_size(B.make_shape(*shp, "fp8_bwd"))
    sc_r, sv_r = B.mm_moe_workspace_size(B.make_shape(*shp, recompute=True))
    assert sc_m > sc_b and sc_f > sc_b
    assert sv_m > sv_b                        # the backward's quantised weights
    assert sv_f == sv_b
    Rp = (16384 * 8 // 256 + 128) * 256       # padded rows (SM-pair tiles)
    acts = Rp * (2048 + 2 * 768 + 768) * 2    # x_perm, h, a in bf16
    assert sv_b - sv_r >= acts                # they leave saved ...
    assert sc_r >= sc_b + acts                # ... for scratch
    assert sv_r < 16 << 20                    # routing and weights per row only


def test_forward_backward_reject_before_launch(lib):
    """NULL / misaligned pointers and unknown precisions return before any CUDA call."""
    s = B.make_shape(64, 128, 64, 8, 2)
    null = [None] * 10
    st = lib.mm_moe_forward(ctypes.byref(s), *([None] * 10))
    assert st == B.MM_MOE_EINVAL
    st = lib.mm_moe_backward(ctypes.byref(s), *([None] * 13))
    assert st == B.MM_MOE_EINVAL
    # recompute needs x in the backward
    rc = B.make_shape(64, 128, 64, 8, 2, recompute=True)
    args = [4096 * (i + 1) for i in range(13)]
    args[5] = None                                  # x
    assert lib.mm_moe_backward(ctypes.byref(rc), *args) == B.MM_MOE_EINVAL
    fake = [4096 * (i + 1) for i in range(10)]
    mis = list(fake)
    mis[0] += 2                                    # x misaligned
    assert lib.mm_moe_forward(ctypes.byref(s), *mis) == B.MM_MOE_EINVAL
    bad_prec = B.make_shape(64, 128, 64, 8, 2, 4)
    assert lib.mm_moe_forward(ctypes.byref(bad_prec), *fake) == B.MM_MOE_EINVAL
    assert lib.mm_moe_get_routing(ctypes.byref(s), None, None, None, None) == B.MM_MOE_EINVAL
    # the router: NULL pointers, k above 32, E not a multiple of 8
    r = B.make_shape(64, 128, 64, 16, 4)
    assert lib.mm_moe_router_forward(ctypes.byref(r), *([None] * 6)) == B.MM_MOE_EINVAL
    assert lib.mm_moe_router_backward(ctypes.byref(r), *([None] * 9)) == B.MM_MOE_EINVAL
    fake6 = [4096 * (i + 1) for i in range(6)]
    for bad in (B.make_shape(64, 128, 64, 64, 33), B.make_shape(64, 128, 64, 12, 4)):
        assert lib.mm_moe_router_forward(ctypes.byref(bad), *fake6) == B.MM_MOE_EINVAL
    # the quantiser: NULL, misaligned, ragged blocks and unknown axes
    assert lib.mm_moe_mx_qdq(None, None, 32, 32, 1, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_qdq(4096, 4098, 32, 32, 1, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_qdq(4096, 8192, 32, 48, 1, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_qdq(4096, 8192, 40, 32, 0, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_mx_qdq(4096, 8192, 32, 32, 2, None) == B.MM_MOE_EINVAL
    assert lib.mm_moe_read_status(None, None) == B.MM_MOE_EINVAL
    del null


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError):
        B.lib()
