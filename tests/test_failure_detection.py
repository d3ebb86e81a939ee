"""Failure detection on the GPU, without a GPU fault.

The grouped GEMMs bound every wait.  A test hook makes gate_up's weight
producer issue nothing, so the MMA's wait for its first stage has nothing to
wait for; with a short wait limit the kernel records MOE_ERR_TIMEOUT, its roles
stop, and the call completes.  The next normal call on the same workspace must
succeed and be correct.  The fused combine's bounds check is driven through a
test launcher with host tables that hold one permuted-row index out of range.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import moe_oracle as O  # noqa: E402
from sparse_moe_transformer_selected_b300 import inputs as gen  # noqa: E402
from sparse_moe_transformer_selected_b300 import moe  # noqa: E402
from sparse_moe_transformer_selected_b300.device import DeviceMoE, bf16_to_f64  # noqa: E402

from . import parity  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()
    yield
    moe.moe_set_fault_injection(0)
    moe.moe_set_wait_limit(0)


DESIGNS = {
    "tmem": (gen.WORKLOADS["tiny"], moe.HIDDEN_F16_PAIR),
    "block_scaled": (gen.Workload("fd_decode", T=16, d=256, W=256, E=16, router_bias="normal",
                                  seed=41), moe.HIDDEN_E4M3_TERMS),
}


@pytest.mark.parametrize("design", sorted(DESIGNS))
def test_withheld_stage_times_out_and_the_next_call_recovers(design):
    wl, fmt = DESIGNS[design]
    inp = gen.make_inputs(wl)
    dev = DeviceMoE.upload(inp)
    assert dev.hidden_format()[0] == fmt
    moe.moe_set_wait_limit(0.02)
    moe.moe_set_fault_injection(1)
    try:
        dev.forward()
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_poll_status(dev.workspace)
        assert ei.value.status == 7                            # MOE_ERR_TIMEOUT
    finally:
        moe.moe_set_fault_injection(0)
        moe.moe_set_wait_limit(0)
    out = bf16_to_f64(dev.forward())
    assert moe.moe_poll_status(dev.workspace) == 0
    ref = O.moe_forward_inputs(inp)
    parity.check_output(out, ref["out"])


def _combine_tables(T, k, d, seed):
    rng = np.random.default_rng(seed)
    R = T * k
    y = rng.normal(0, 50, size=(R, d)).astype(np.float32)
    perm = rng.permutation(R).astype(np.int32)              # permuted row -> t k + j
    inv = np.empty(R, dtype=np.int32)
    inv[perm] = np.arange(R, dtype=np.int32)
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    return y, perm, inv, w


def _combine_ref(y, inv, w, T, k, skip=None):
    out = np.zeros((T, y.shape[1]))
    for t in range(T):
        for s in range(k):
            if (t, s) != skip:
                out[t] += np.float64(w[t, s]) * y[inv[t * k + s]].astype(np.float64)
    return out


@pytest.mark.parametrize("corrupt", [False, True])
def test_combine_reports_and_skips_a_row_out_of_range(corrupt):
    T, k, d = 40, 4, 320
    y, perm, inv, w = _combine_tables(T, k, d, seed=43)
    skip = None
    if corrupt:
        inv[7 * k + 2] = T * k + 5                          # outside [0, T k)
        skip = (7, 2)
    dv = "cuda"
    yt, pt, it, wt = (torch.from_numpy(a).to(dv) for a in (y, perm, inv, w))
    out = torch.full((T, d), float("nan"), dtype=torch.bfloat16, device=dv)
    nb = 256 + 4 * T * ((d + 127) // 128)
    ws = torch.empty(nb, dtype=torch.uint8, device=dv)
    moe.moe_debug_combine(yt, pt, it, wt, T, d, k, out, ws, nb)
    if corrupt:
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_poll_status(ws)
        assert ei.value.status == 8                         # MOE_ERR_DEVICE_BOUNDS
    else:
        assert moe.moe_poll_status(ws) == 0
    got = bf16_to_f64(out)
    ref = _combine_ref(y, inv, w, T, k, skip)
    # one rounding to bf16 of an fp32 sum: within a bf16 half-ulp plus fp32 noise
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-4)
