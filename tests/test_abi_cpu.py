"""The C ABI on the host: the library loads, exports what include/moe.h declares,
and rejects bad arguments before touching the GPU.  No kernel runs here."""
import ctypes
import os
import re

import pytest

from sparse_moe_transformer_selected_b300 import build, moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load()


def declared_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(moe.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # exported with C linkage: the plain name resolves through dlsym
    for name in declared_functions():
        ctypes.CDLL(moe.LIB_PATH)[name]


def test_workspace_bytes(lib):
    assert moe.moe_workspace_bytes(0, 256, 256, 8, 4) == 0
    n = moe.moe_workspace_bytes(64, 256, 256, 8, 4)
    R = 256
    assert n >= R * 256 * 2 + 2 * R * 256 * 2 + R * 256 * 4  # x_perm + h pair + y
    assert moe.moe_workspace_bytes(64, 250, 256, 8, 4) == 0       # d % 32
    assert moe.moe_workspace_bytes(64, 256, 250, 8, 4) == 0       # W % 32
    assert moe.moe_workspace_bytes(64, 256, 256, 257, 4) == 0     # E > 256
    assert moe.moe_workspace_bytes(64, 256, 256, 8, 9) == 0       # k > 8
    assert moe.moe_workspace_bytes(64, 256, 256, 3, 4) == 0       # k > E
    assert "k = 4" in moe.moe_last_error()


def test_workspace_regions_disjoint_and_aligned(lib):
    T, d, W, E, k = 77, 96, 160, 5, 3
    total = moe.moe_workspace_bytes(T, d, W, E, k)
    spans = []
    for name in moe.REGIONS:
        off, nb = moe.moe_workspace_region(T, d, W, E, k, name)
        assert off % 256 == 0 and off >= 256 and off + nb <= total, name
        spans.append((off, off + nb))
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    with pytest.raises(moe.MoEError):
        moe.moe_workspace_region(T, d, W, E, k, 99)


def _forward(lib, T=64, d=256, W=256, E=8, k=4, ws_bytes=None, **ptrs):
    good = dict(x=16, rw=16, rb=16, wgu=16, wgus=16, bgu=16, wdn=16, wdns=16, bdn=16,
                out=16, ws=16)
    good.update(ptrs)
    if ws_bytes is None:
        ws_bytes = max(1, moe.moe_workspace_bytes(T, d, W, E, k))
    p = {k_: ctypes.c_void_p(v) for k_, v in good.items()}
    return lib.moe_forward(p["x"], T, d, W, p["rw"], p["rb"], p["wgu"], p["wgus"], p["bgu"],
                           p["wdn"], p["wdns"], p["bdn"], E, k, 7.0, 1.702, p["out"], p["ws"],
                           ws_bytes, None)


def test_argument_errors_return_before_any_launch(lib):
    # every case below is rejected on the host; the fake addresses are never used
    assert _forward(lib, d=100) == 2                              # MOE_ERR_SHAPE
    assert _forward(lib, W=48) == 2
    assert _forward(lib, E=0) == 2
    assert _forward(lib, k=0) == 2
    assert _forward(lib, T=-1) == 2
    assert _forward(lib, x=0) == 1                                # MOE_ERR_NULL
    assert "x is NULL" in moe.moe_last_error()
    assert _forward(lib, ws=0) == 1
    assert _forward(lib, wgu=24) == 3                             # MOE_ERR_ALIGN
    assert "w_gu" in moe.moe_last_error()
    assert _forward(lib, ws_bytes=1024) == 4                      # MOE_ERR_WORKSPACE
    assert _forward(lib, T=0) == 0                                # nothing to do


def test_nan_limit_rejected(lib):
    p = [ctypes.c_void_p(16)] * 11
    st = lib.moe_forward(p[0], 64, 256, 256, p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8],
                         8, 4, float("nan"), 1.0, p[9], p[10], 1 << 30, None)
    assert st == 2


def test_route_argument_errors(lib):
    v = ctypes.c_void_p
    assert lib.moe_route(v(16), 64, 100, v(16), v(16), 8, 4, None, None, None, None, None,
                         v(16), 1 << 20, None) == 2
    assert lib.moe_route(None, 64, 256, v(16), v(16), 8, 4, None, None, None, None, None,
                         v(16), 1 << 20, None) == 1
    assert lib.moe_route(v(16), 64, 256, v(16), v(16), 8, 4, v(20), None, None, None, None,
                         v(16), 1 << 20, None) == 3
    assert lib.moe_route(v(16), 0, 256, v(16), v(16), 8, 4, None, None, None, None, None,
                         v(16), 0, None) == 0


def test_binding_raises_on_error(lib):
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_forward(0, 64, 256, 256, 16, 16, 16, 16, 16, 16, 16, 16, 8, 4, 7.0, 1.702,
                        16, 16, 1 << 30, stream=0)
    assert ei.value.status == 1


# ------------------------------------------------- GEMM design selection --
# moe_hidden_format reports how h is carried, which names the design moe_forward
# picks for a shape and clamp; the choice is host logic, checked here without a GPU.

@pytest.mark.parametrize("shape,limit,want", [
    # decode-sized loads (at most 8 routed rows per expert) with a bounded clamp:
    # block-scaled MXFP4 GEMMs, h as four E4M3 terms scaled by 2^-3 at limit 7
    ((32, 2880, 2880, 32, 4), 7.0, (moe.HIDDEN_E4M3_TERMS, -3)),
    ((64, 2880, 2880, 128, 4), 7.0, (moe.HIDDEN_E4M3_TERMS, -3)),
    ((32, 2048, 768, 128, 8), 7.0, (moe.HIDDEN_E4M3_TERMS, -3)),
    ((24, 448, 320, 16, 4), 7.0, (moe.HIDDEN_E4M3_TERMS, -3)),      # K % 128 = 64 tails
    ((32, 2880, 2880, 32, 4), 1.0, (moe.HIDDEN_E4M3_TERMS, -7)),    # |h| <= 2: 2^7 scale
    # more rows per expert: TMEM-dequantised GEMMs with an f16 pair
    ((8192, 2880, 2880, 32, 4), 7.0, (moe.HIDDEN_F16_PAIR, 0)),
    ((64, 256, 256, 8, 4), 7.0, (moe.HIDDEN_F16_PAIR, 0)),
    # block-scaled design excluded: a clamp too wide for a fixed scale, no clamp,
    # a reduction length whose 4-bit tail map would be misaligned, K < 128
    ((32, 2880, 2880, 32, 4), 20.0, (moe.HIDDEN_F16_PAIR, 0)),
    ((32, 2880, 2880, 32, 4), float("inf"), (moe.HIDDEN_BF16_PAIR, 0)),
    ((16, 416, 256, 8, 4), 7.0, (moe.HIDDEN_F16_PAIR, 0)),
    ((45, 96, 160, 5, 4), 7.0, (moe.HIDDEN_F16_PAIR, 0)),
])
def test_gemm_design_selection(lib, shape, limit, want):
    assert moe.moe_hidden_format(*shape, limit) == want


def test_gemm_design_override(lib, monkeypatch):
    decode = (32, 2880, 2880, 32, 4)
    monkeypatch.setenv("MOE_GEMM", "tmem")
    assert moe.moe_hidden_format(*decode, 7.0)[0] == moe.HIDDEN_F16_PAIR
    monkeypatch.setenv("MOE_GEMM", "anything-else")                 # ignored
    assert moe.moe_hidden_format(*decode, 7.0)[0] == moe.HIDDEN_E4M3_TERMS


def _block(lib, T=64, d=256, W=256, E=8, k=4, eps=1e-5, ws_bytes=None, **ptrs):
    good = dict(x=16, g=16, rw=16, rb=16, wgu=16, wgus=16, bgu=16, wdn=16, wdns=16, bdn=16,
                out=16, ws=16)
    good.update(ptrs)
    if ws_bytes is None:
        ws_bytes = max(1, moe.moe_workspace_bytes(T, d, W, E, k))
    p = {k_: ctypes.c_void_p(v) for k_, v in good.items()}
    return lib.moe_block_forward(p["x"], T, d, W, p["g"], eps, p["rw"], p["rb"], p["wgu"],
                                 p["wgus"], p["bgu"], p["wdn"], p["wdns"], p["bdn"], E, k, 7.0,
                                 1.702, p["out"], p["ws"], ws_bytes, None)


def test_block_argument_errors_return_before_any_launch(lib):
    # every case below is rejected on the host; the fake addresses are never used
    assert _block(lib, g=0) == 1                                  # MOE_ERR_NULL
    assert "norm_w" in moe.moe_last_error()
    assert _block(lib, g=24) == 3                                 # MOE_ERR_ALIGN
    assert _block(lib, eps=float("nan")) == 2                     # MOE_ERR_SHAPE
    assert _block(lib, eps=-1.0) == 2
    assert _block(lib, eps=float("inf")) == 2
    assert _block(lib, d=100) == 2
    assert _block(lib, x=0) == 1
    assert _block(lib, ws_bytes=1024) == 4                        # MOE_ERR_WORKSPACE
    assert _block(lib, T=0, g=0) == 0                             # nothing to do
    assert _block(lib, T=0, g=24) == 3                            # still checked at T = 0


def test_failure_hooks_check_their_arguments(lib):
    with pytest.raises(moe.MoEError):
        moe.moe_set_wait_limit(1e-6)
    with pytest.raises(moe.MoEError):
        moe.moe_set_wait_limit(120.0)
    with pytest.raises(moe.MoEError):
        moe.moe_set_fault_injection(2)
    assert moe.moe_set_wait_limit(0.5) == 0
    assert moe.moe_set_wait_limit(0) == 0
    assert moe.moe_set_fault_injection(0) == 0
    # the combine launcher rejects shapes on the host (fake addresses unused)
    assert lib.moe_debug_combine(16, 16, 16, 16, 4, 100, 4, 16, 16, 1 << 20, None) == 2
    assert lib.moe_debug_combine(16, 16, 16, 16, 4, 128, 4, 16, 16, 8, None) == 4


def test_mma_peak_checks_its_arguments(lib):
    out = ctypes.c_double(0.0)
    assert lib.moe_mma_peak(4, 10, ctypes.byref(out), 16, None) == 2
    assert lib.moe_mma_peak(-1, 10, ctypes.byref(out), 16, None) == 2
    assert lib.moe_mma_peak(0, 0, ctypes.byref(out), 16, None) == 2
    assert lib.moe_mma_peak(1, 10, None, 16, None) == 1
