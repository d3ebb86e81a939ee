"""moe_forward_noalloc: the MoE block for callers that cannot allocate device
memory while it runs (an engine plugin whose host forbids allocation during
serving, a real-time loop, code handed only its input and output buffers).
It brings its own scratch, a fixed array inside the library, and must give
the same results as moe_forward with a caller workspace.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import numpy as np
import pytest

from sparse_moe_transformer_selected_b300 import build, moe
from sparse_moe_transformer_selected_b300 import inputs as gen

from . import parity


def _call_noalloc(dev, x, out):
    moe.moe_forward_noalloc(x, dev.T, dev.d, dev.W, dev.router_w, dev.router_b, dev.w_gu,
                            dev.w_gu_scale, dev.b_gu, dev.w_dn, dev.w_dn_scale, dev.b_dn, dev.E,
                            dev.k, dev.limit, dev.alpha, out)


def test_oversize_shape_is_rejected_before_any_gpu_work():
    build.build()
    lib = moe.load()
    # 4096 tokens at d = W = 2880 need far more than the built-in scratch; the
    # call must fail on the host (the fake addresses below are never used)
    v = [16] * 11
    st = lib.moe_forward_noalloc(v[0], 4096, 2880, 2880, v[1], v[2], v[3], v[4], v[5], v[6],
                                 v[7], v[8], 32, 4, 7.0, 1.702, v[9], None)
    assert st == 4                                              # MOE_ERR_WORKSPACE
    assert "built-in array" in moe.moe_last_error()
    assert moe.moe_workspace_bytes(4096, 2880, 2880, 32, 4) > moe.NOALLOC_SCRATCH_BYTES
    assert lib.moe_forward_noalloc(v[0], 64, 100, 2880, v[1], v[2], v[3], v[4], v[5], v[6],
                                   v[7], v[8], 32, 4, 7.0, 1.702, v[9], None) == 2


def test_scratch_fits_the_stated_decode_sizes():
    """The header's size statement: the built-in scratch holds the workspace of
    up to 144 tokens at d = W = 2880, k = 4, for 32 and for 128 experts."""
    moe.load()
    for E in (32, 128):
        assert moe.moe_workspace_bytes(144, 2880, 2880, E, 4) <= moe.NOALLOC_SCRATCH_BYTES
        assert moe.moe_workspace_bytes(145, 2880, 2880, E, 4) > moe.NOALLOC_SCRATCH_BYTES


def test_zero_tokens_gets_the_same_argument_checks():
    """With T = 0 the call enqueues nothing but still rejects what moe_forward
    rejects (the fake addresses are never used)."""
    lib = moe.load()
    v = [16] * 11
    args = lambda x, lim: (x, 0, 2880, 2880, v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8],
                           32, 4, lim, 1.702, v[9], None)
    assert lib.moe_forward_noalloc(*args(v[0], 7.0)) == 0
    assert lib.moe_forward_noalloc(*args(24, 7.0)) == 3            # misaligned x
    assert lib.moe_forward_noalloc(*args(v[0], float("nan"))) == 2
    assert lib.moe_forward_noalloc(24, 0, 100, 2880, *([16] * 8), 32, 4, 7.0, 1.702, 16,
                                   None) == 2                        # d % 32


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "gptoss20b_decode"])
def test_noalloc_matches_moe_forward_on_two_calls(name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_moe_transformer_selected_b300.device import DeviceMoE, bf16_to_f64

    wl = gen.WORKLOADS[name]
    assert moe.moe_workspace_bytes(wl.T, wl.d, wl.W, wl.E, wl.k) <= moe.NOALLOC_SCRATCH_BYTES
    dev = DeviceMoE.upload(gen.make_inputs(wl))
    # a second batch of tokens for the second call, so stale scratch from the
    # first call could not go unnoticed
    x2 = gen.make_inputs(wl.with_(seed=wl.seed + 101)).x
    x_b = torch.from_numpy(x2.view(np.int16)).to(dev.x.device).view(torch.bfloat16)
    for x in (dev.x, x_b):
        ref = bf16_to_f64(dev.forward(x=x).clone())
        out = torch.full_like(dev.out, float("nan"))
        _call_noalloc(dev, x, out)
        torch.cuda.synchronize()
        assert moe.moe_poll_status_noalloc() == 0       # its own status word: no failure
        got = bf16_to_f64(out)
        parity.check_output(got, ref, what=f"{name} no-alloc vs workspace")
        # same kernels, same order of arithmetic: the results agree bit for bit
        assert np.array_equal(got, ref)
