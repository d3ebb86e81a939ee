"""CUDA path vs the CPU oracle, through the C ABI, on one GPU.

Every layer is compared element by element, the full gpt-oss layer shapes
included: they run at full size in the launch configuration the benchmark
times, and the oracle computes every token (its experts on all host cores).
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import moe_oracle as O  # noqa: E402
from sparse_moe_transformer_selected_b300 import inputs as gen  # noqa: E402
from sparse_moe_transformer_selected_b300 import moe  # noqa: E402
from sparse_moe_transformer_selected_b300.device import DeviceMoE, bf16_to_f64  # noqa: E402

from . import parity  # noqa: E402

pytestmark = pytest.mark.gpu

FULL = ["gptoss20b_decode", "gptoss20b_prefill", "gptoss120b_prefill",
        "gptoss120b_skew16k", "gptoss120b_skew64"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()
    yield
    torch.cuda.synchronize()


def _run(inp, tokens=None, keep_hidden=False):
    dev = DeviceMoE.upload(inp)
    out = dev.forward()
    moe.moe_poll_status(dev.workspace)
    ref = O.moe_forward_inputs(inp, tokens=tokens, keep_hidden=keep_hidden)
    return dev, bf16_to_f64(out), ref


def _check_full(dev, out, ref, k):
    idx = dev.region("topk_idx").cpu().numpy()
    w = dev.region("topk_w").cpu().numpy()
    excused = parity.check_routing(ref, idx, w, k)
    parity.check_permutation(O.expert_permutation, idx, dev.E,
                             dev.region("offsets").cpu().numpy(),
                             dev.region("perm").cpu().numpy(),
                             dev.region("inv").cpu().numpy())
    keep = np.setdiff1d(np.arange(ref["out"].shape[0]), excused)
    return parity.check_output(out[keep], ref["out"][keep])


# ---------------------------------------------------------------- routing --

@pytest.mark.parametrize("name", ["tiny"] + FULL)
def test_route_parity(name):
    wl = gen.WORKLOADS[name]
    x, rw, rb = gen.make_router_inputs(wl)
    dev = "cuda"
    xt = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    rwt, rbt = torch.from_numpy(rw).to(dev), torch.from_numpy(rb).to(dev)
    nb = moe.moe_workspace_bytes(wl.T, wl.d, 32, wl.E, wl.k)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    T, k, E = wl.T, wl.k, wl.E
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty((T, k), dtype=torch.int32, device=dev)
    moe.moe_route(xt, T, wl.d, rwt, rbt, E, k, idx, w, off, perm, inv, ws, nb)
    moe.moe_poll_status(ws)
    logits = O.router_logits(O.bf16_bits_to_f64(x), rw, rb)
    ridx, gap = O.select_topk(logits, k)
    ref = dict(topk_idx=ridx, gap=gap, logits=logits,
               topk_w=O.selected_softmax(np.take_along_axis(logits, ridx, axis=1)))
    idx_h = idx.cpu().numpy()
    excused = parity.check_routing(ref, idx_h, w.cpu().numpy(), k)
    assert len(excused) <= max(2, T // 2000), f"too many near-tie differences: {excused}"
    parity.check_permutation(O.expert_permutation, idx_h, E, off.cpu().numpy(),
                             perm.cpu().numpy(), inv.cpu().numpy())
    if excused == []:
        counts, offsets, p, iv = O.expert_permutation(ridx, E)
        assert np.array_equal(off.cpu().numpy(), offsets)
    if name == "gptoss120b_skew16k":
        counts = np.diff(off.cpu().numpy())
        assert (counts == 0).sum() >= 1 and (counts > 0.10 * T).sum() >= 1


# ------------------------------------------------------------ whole block --

def test_forward_tiny_with_intermediates():
    inp = gen.make_inputs(gen.WORKLOADS["tiny"])
    dev, out, ref = _run(inp, keep_hidden=True)
    rel, worst = _check_full(dev, out, ref, 4)
    # hidden activations h (carried as hi + lo bf16) and expert outputs y
    perm = dev.region("perm").cpu().numpy()
    h = dev.hidden().cpu().numpy().astype(np.float64)
    y = dev.region("y").cpu().numpy().astype(np.float64)
    for row, q in enumerate(perm):
        t, j = divmod(int(q), 4)
        z_ref, h_ref, y_ref = ref["hidden"][(t, j)]
        assert np.allclose(h[row], h_ref, rtol=1e-4, atol=1e-4 * np.abs(h_ref).max()), (t, j)
        assert np.allclose(y[row], y_ref, rtol=1e-4, atol=1e-4 * np.abs(y_ref).max()), (t, j)


def test_forward_decode_20b_all_tokens():
    inp = gen.make_inputs(gen.WORKLOADS["gptoss20b_decode"])
    dev, out, ref = _run(inp)
    _check_full(dev, out, ref, 4)


@pytest.mark.parametrize("name", ["gptoss20b_prefill", "gptoss120b_prefill",
                                  "gptoss120b_skew16k", "gptoss120b_skew64"])
def test_forward_full_size_every_token(name):
    """The full gpt-oss layers in the launch configuration the benchmark times,
    every output element of every token against the oracle (its experts on all
    host cores): every work unit of both GEMMs, every chunk boundary and every
    expert segment's last partial chunk is compared."""
    wl = gen.WORKLOADS[name]
    inp = gen.make_inputs(wl)
    dev = DeviceMoE.upload(inp)
    out = bf16_to_f64(dev.forward())
    moe.moe_poll_status(dev.workspace)
    ref = O.moe_forward_inputs(inp, workers=os.cpu_count() or 1)
    rel, worst = _check_full(dev, out, ref, wl.k)
    # deterministic: a second run is bitwise identical
    first = dev.out.clone()
    dev.forward()
    assert torch.equal(first.view(torch.int16), dev.out.view(torch.int16))


# ----------------------------------------------------------- edge cases --

EDGE = {
    "T1": gen.Workload("T1", T=1, d=256, W=256, E=8, router_bias="normal"),
    "ragged77": gen.Workload("ragged77", T=77, d=256, W=256, E=8, router_bias="normal", seed=3),
    "T33": gen.Workload("T33", T=33, d=128, W=192, E=6, router_bias="normal", seed=4),
    "E1k1": gen.Workload("E1k1", T=40, d=128, W=128, E=1, k=1, seed=5),
    "k1": gen.Workload("k1", T=50, d=128, W=128, E=16, k=1, router_bias="normal", seed=6),
    "k8": gen.Workload("k8", T=50, d=128, W=128, E=16, k=8, router_bias="normal", seed=7),
    "d32": gen.Workload("d32", T=45, d=32, W=32, E=4, router_bias="normal", seed=8),
    "d96_w160": gen.Workload("d96_w160", T=70, d=96, W=160, E=5, router_bias="normal", seed=9),
    "E256": gen.Workload("E256", T=300, d=64, W=64, E=256, router_bias="normal", seed=10),
    "rows_over_tile": gen.Workload("rows_over_tile", T=600, d=256, W=256, E=4, k=2,
                                   router_bias="normal", seed=11),
    # more than 8 router tiles with d not a multiple of 64: the CUDA-core
    # split-K logits kernel instead of the tensor-core one
    "split_d96": gen.Workload("split_d96", T=300, d=96, W=64, E=8, router_bias="normal", seed=13),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_shapes(name):
    inp = gen.make_inputs(EDGE[name])
    dev, out, ref = _run(inp)
    _check_full(dev, out, ref, EDGE[name].k)


def test_plain_swiglu_special_case():
    inp = gen.make_inputs(gen.WORKLOADS["tiny"].with_(seed=12), limit=float("inf"), alpha=1.0)
    dev, out, ref = _run(inp)
    _check_full(dev, out, ref, 4)


def test_all_tokens_one_expert():
    """One expert takes every token (a segment much longer than a row tile);
    the others are empty."""
    wl = gen.Workload("hot", T=300, d=128, W=128, E=8, k=1, router_bias="normal", seed=13)
    inp = gen.make_inputs(wl)
    inp.router_b[:] = -100.0
    inp.router_b[5] = 100.0
    dev, out, ref = _run(inp)
    assert np.all(ref["topk_idx"] == 5)
    _check_full(dev, out, ref, 1)


@pytest.mark.parametrize("n0,n1", [(192, 160), (193, 161), (384, 1)])
def test_chunk_boundaries(n0, n1):
    """Two experts take exactly n0 and n1 rows, so the TMEM design's token
    chunks (192 rows for gate_up, 160 for down, above 32 rows per expert)
    end exactly at an expert's last row, or one row before it; the tokens of
    the two experts are interleaved at random."""
    wl = gen.Workload("split", T=n0 + n1, d=256, W=256, E=2, k=1, seed=16)
    inp = gen.make_inputs(wl)
    # route on the sign of feature 0 alone: +1 -> expert 0, -1 -> expert 1
    sign = np.ones(wl.T, dtype=np.float32)
    sign[np.random.default_rng(17).permutation(wl.T)[:n1]] = -1.0
    inp.x[:, 0] = gen.f32_to_bf16_bits(sign)
    inp.router_w[:] = 0.0
    inp.router_w[0, 0], inp.router_w[1, 0] = 10.0, -10.0
    inp.router_b[:] = 0.0
    dev, out, ref = _run(inp)
    assert np.bincount(ref["topk_idx"].ravel(), minlength=2).tolist() == [n0, n1]
    _check_full(dev, out, ref, 1)


def test_identical_experts_give_router_independent_output():
    wl = gen.Workload("same", T=64, d=128, W=128, E=8, router_bias="normal", seed=14)
    inp = gen.make_inputs(wl)
    for arr in (inp.w_gu, inp.w_gu_scale, inp.b_gu, inp.w_dn, inp.w_dn_scale, inp.b_dn):
        arr[:] = arr[0]
    dev, out, ref = _run(inp)
    _check_full(dev, out, ref, 4)
    inp.router_b = np.random.default_rng(0).normal(0, 5, wl.E).astype(np.float32)
    dev2, out2, _ = _run(inp)
    parity.check_output(out2, ref["out"])


def test_deterministic_and_status_ok():
    inp = gen.make_inputs(gen.WORKLOADS["tiny"].with_(T=200, seed=15))
    dev = DeviceMoE.upload(inp)
    a = dev.forward().clone()
    b = dev.forward().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_poll_status(dev.workspace) == 0


def test_zero_tokens_is_a_no_op():
    inp = gen.make_inputs(gen.WORKLOADS["tiny"])
    dev = DeviceMoE.upload(inp)
    sentinel = torch.full_like(dev.out, 3.0)
    moe.moe_forward(dev.x, 0, dev.d, dev.W, dev.router_w, dev.router_b, dev.w_gu, dev.w_gu_scale,
                    dev.b_gu, dev.w_dn, dev.w_dn_scale, dev.b_dn, dev.E, dev.k, 7.0, 1.702,
                    sentinel, dev.workspace, 0)
    torch.cuda.synchronize()
    assert torch.all(sentinel == 3.0)


# ---------------------------------------- the TMEM design on small shapes --

@pytest.mark.parametrize("name", ["T1", "T33", "d32", "k8"])
def test_edge_shapes_forced_tmem_design(name, monkeypatch):
    """MOE_GEMM=tmem runs K3/K4 with the dequantised weights in tensor memory
    on shapes the block-scaled design would otherwise take (or on its fallback
    shapes); it must meet the same bar."""
    monkeypatch.setenv("MOE_GEMM", "tmem")
    inp = gen.make_inputs(EDGE[name])
    dev, out, ref = _run(inp)
    assert dev.hidden_format()[0] != moe.HIDDEN_E4M3_TERMS
    _check_full(dev, out, ref, EDGE[name].k)


# ----------------------------------- the pre-norm block: RMSNorm + residual --

def _run_block(inp, tokens=None):
    dev = DeviceMoE.upload(inp)
    out = dev.forward()
    moe.moe_poll_status(dev.workspace)
    ref = O.moe_block_forward_inputs(inp, tokens=tokens, workers=os.cpu_count() or 1)
    return dev, bf16_to_f64(out), ref


@pytest.mark.parametrize("name,want", [("tiny", moe.HIDDEN_F16_PAIR),
                                       ("gptoss20b_decode", moe.HIDDEN_E4M3_TERMS),
                                       ("ragged77", moe.HIDDEN_F16_PAIR),
                                       ("E256", moe.HIDDEN_F16_PAIR)])
def test_block_forward_parity(name, want):
    """out = x + MoE(RMSNorm(x)) against the oracle's block, on both GEMM
    designs: routing (from the normalised x) bit-exact up to flagged near-ties,
    every output element within the tolerances."""
    wl = gen.WORKLOADS.get(name) or EDGE[name]
    inp = gen.make_block_inputs(wl)
    dev, out, ref = _run_block(inp)
    assert dev.hidden_format()[0] == want
    _check_full(dev, out, ref, wl.k)


def test_block_forward_prefill_every_token():
    """The 20b prefill shape through the block entry point (its RMSNorm runs as
    a pass of its own for more than 256 tokens), every token compared."""
    wl = gen.WORKLOADS["gptoss20b_prefill"]
    inp = gen.make_block_inputs(wl)
    dev, out, ref = _run_block(inp)
    _check_full(dev, out, ref, wl.k)


def test_block_forward_in_place():
    """out may be the input buffer itself (an in-place residual update)."""
    inp = gen.make_block_inputs(gen.WORKLOADS["gptoss20b_decode"])
    dev = DeviceMoE.upload(inp)
    want = dev.forward().clone()
    x = dev.x.clone()
    dev.forward(x=x, out=x)
    moe.moe_poll_status(dev.workspace)
    assert torch.equal(x.view(torch.int16), want.view(torch.int16))


def test_cuda_graph_replay_matches_eager_call():
    """moe_forward captured into a CUDA graph (the benchmark's end-to-end path)
    gives the eager call's output bit for bit, and follows new inputs."""
    inp = gen.make_inputs(gen.WORKLOADS["gptoss20b_decode"])
    dev = DeviceMoE.upload(inp)
    eager = dev.forward().clone()
    graph = dev.capture_graph()
    dev.out.fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), dev.out.view(torch.int16))
    x2 = gen.make_inputs(gen.WORKLOADS["gptoss20b_decode"].with_(seed=77)).x
    dev.x.copy_(torch.from_numpy(x2.view(np.int16)).view(torch.bfloat16))
    graph.replay()
    second = dev.out.clone()
    assert torch.equal(second.view(torch.int16), dev.forward().view(torch.int16))
    moe.moe_poll_status(dev.workspace)


# ------------------------------------------------ the block-scaled design --

def test_block_scaled_path_intermediates():
    """A decode-sized load with K % 128 = 64 on both GEMMs (the tail box read
    through the second tensor map) and a partial down tile (d % 128 = 64) runs
    on the block-scaled design; its h (four E4M3 terms) and y match the oracle
    row by row."""
    wl = gen.Workload("mx_tail", T=24, d=448, W=320, E=16, router_bias="normal", seed=21)
    inp = gen.make_inputs(wl)
    dev, out, ref = _run(inp, keep_hidden=True)
    fmt, ex = dev.hidden_format()
    assert fmt == moe.HIDDEN_E4M3_TERMS and ex == -3
    _check_full(dev, out, ref, 4)
    perm = dev.region("perm").cpu().numpy()
    h = dev.hidden().cpu().numpy().astype(np.float64)
    y = dev.region("y").cpu().numpy().astype(np.float64)
    for row, q in enumerate(perm):
        t, j = divmod(int(q), 4)
        z_ref, h_ref, y_ref = ref["hidden"][(t, j)]
        assert np.allclose(h[row], h_ref, rtol=1e-4, atol=1e-4 * np.abs(h_ref).max()), (t, j)
        assert np.allclose(y[row], y_ref, rtol=1e-4, atol=1e-4 * np.abs(y_ref).max()), (t, j)


def test_block_scaled_and_tmem_designs_agree_on_decode(monkeypatch):
    """MOE_GEMM=tmem forces the dequantise-into-TMEM design on the 20b decode
    layer; it and the default block-scaled design agree within the oracle bar."""
    inp = gen.make_inputs(gen.WORKLOADS["gptoss20b_decode"])
    dev = DeviceMoE.upload(inp)
    assert dev.hidden_format()[0] == moe.HIDDEN_E4M3_TERMS
    a = bf16_to_f64(dev.forward().clone())
    monkeypatch.setenv("MOE_GEMM", "tmem")
    assert dev.hidden_format()[0] == moe.HIDDEN_F16_PAIR
    b = bf16_to_f64(dev.forward().clone())
    moe.moe_poll_status(dev.workspace)
    parity.check_output(a, b, what="block-scaled vs tmem design")


@pytest.mark.parametrize("case", ["k_tail_32", "wide_clamp"])
def test_block_scaled_design_falls_back(case):
    """Decode-sized loads the block-scaled design cannot take run on the TMEM
    design: a reduction length with K % 128 = 32 (the 4-bit tail map's base
    would not be 32-byte aligned) and a clamp too wide for a fixed h scale."""
    if case == "k_tail_32":
        wl = gen.Workload("k_tail_32", T=16, d=416, W=256, E=8, router_bias="normal", seed=22)
        inp = gen.make_inputs(wl)
    else:
        wl = gen.Workload("wide_clamp", T=16, d=256, W=256, E=8, router_bias="normal", seed=23)
        inp = gen.make_inputs(wl, limit=20.0)
    dev, out, ref = _run(inp)
    assert dev.hidden_format()[0] != moe.HIDDEN_E4M3_TERMS
    _check_full(dev, out, ref, 4)


# ------------------------------------------------ a second MoE shape (stress) --

@pytest.mark.parametrize("name", sorted(gen.STRESS_WORKLOADS))
def test_stress_shape_d2048_w768_e128_top8(name):
    """Another model's MoE layer shape (d 2048, expert width 768, 128 experts,
    top-8) through the same kernels: the decode size takes the block-scaled
    design, the prefill size the TMEM design; every token compared."""
    wl = gen.STRESS_WORKLOADS[name]
    inp = gen.make_inputs(wl)
    dev = DeviceMoE.upload(inp)
    out = bf16_to_f64(dev.forward())
    moe.moe_poll_status(dev.workspace)
    ref = O.moe_forward_inputs(inp, workers=os.cpu_count() or 1)
    fmt = dev.hidden_format()[0]
    assert (fmt == moe.HIDDEN_E4M3_TERMS) == (wl.T <= 64)
    _check_full(dev, out, ref, wl.k)


def test_block_scaled_design_with_16_byte_aligned_weights():
    """Weight buffers aligned to 16 but not 32 bytes: the 4-bit TMA maps want
    32-byte bases, so the call takes the TMEM design instead and still meets
    the oracle bar (same layer, same result up to rounding)."""
    wl = gen.Workload("aligned16", T=16, d=256, W=256, E=8, router_bias="normal", seed=24)
    inp = gen.make_inputs(wl)
    dev = DeviceMoE.upload(inp)
    assert dev.hidden_format()[0] == moe.HIDDEN_E4M3_TERMS
    ref = O.moe_forward_inputs(inp)

    def shifted(t):
        buf = torch.empty(t.numel() + 16, dtype=torch.uint8, device=t.device)
        view = buf[16:16 + t.numel()]
        view.copy_(t.view(-1))
        assert view.data_ptr() % 32 == 16
        return view

    w_gu, w_dn = shifted(dev.w_gu), shifted(dev.w_dn)
    out = torch.empty_like(dev.out)
    moe.moe_forward(dev.x, dev.T, dev.d, dev.W, dev.router_w, dev.router_b, w_gu, dev.w_gu_scale,
                    dev.b_gu, w_dn, dev.w_dn_scale, dev.b_dn, dev.E, dev.k, dev.limit, dev.alpha,
                    out, dev.workspace, dev.workspace.numel())
    moe.moe_poll_status(dev.workspace)
    _check_full(dev, bf16_to_f64(out), ref, 4)
    # the aligned call (block-scaled design) agrees with it
    parity.check_output(bf16_to_f64(dev.forward()), bf16_to_f64(out), what="aligned vs 16-byte-aligned weights")


# ------------------------------------ the TMEM design at extreme weight scales --

def _scale_extreme_inputs(limit):
    """A layer the TMEM design takes (128 rows per expert) whose E8M0 weight
    scales reach past the old limits of its number formats (f16: bytes above
    240; bf16: above 142) and span far more than 2^14 within a row."""
    wl = gen.Workload("scale_extremes", T=256, d=256, W=256, E=4, k=2, router_bias="normal",
                      seed=51)
    inp = gen.make_inputs(wl, limit=limit)
    W, nsb = wl.W, wl.d // 32
    gus, dns = inp.w_gu_scale, inp.w_dn_scale
    if np.isfinite(limit):                     # (the clamp bounds h whatever z is)
        gus[0, 0:16, 0] = 244                  # gate rows: one block near the top of E8M0
    gus[0, 16:48, 1::2] = gus[0, 16:48, 0::2] - 20   # blocks 2^20 below their neighbours
    gus[1, W:W + 32, 2] = 1                    # up rows: a block at the bottom of E8M0
    dns[1, 0:64, 3] = dns[1, 0:64, 0] - 18      # down rows spanning 2^18
    if not np.isfinite(limit):
        dns[2, 0:32, 0] = 150                  # bf16 form: above 2^(142 - 127)
    return inp


@pytest.mark.parametrize("limit", [7.0, float("inf")])
def test_tmem_design_extreme_weight_scales(limit):
    """The dequantiser's per-row power-of-two factors stay exact for scale bytes
    up to 254 (the f16 form for the clamped layer, the bf16 form for the
    unclamped one); blocks more than 2^14 below their row's largest are left
    out in the f16 form, an error far inside the tolerance."""
    inp = _scale_extreme_inputs(limit)
    dev, out, ref = _run(inp)
    fmt = dev.hidden_format()[0]
    assert fmt == (moe.HIDDEN_F16_PAIR if np.isfinite(limit) else moe.HIDDEN_BF16_PAIR)
    assert np.all(np.isfinite(ref["out"]))
    _check_full(dev, out, ref, 2)
