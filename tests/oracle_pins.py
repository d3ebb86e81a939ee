"""Pins of the CPU oracle to facts outside itself.

Each check_* function takes an oracle module (the real one, or a mutant built
by test_oracle_mutations.py) and raises AssertionError when the oracle
disagrees with what the pages, the number formats or the mathematics fix.
None of them re-types the oracle's own formula: each compares against a
closed form, a brute force, a printed value or an invariant.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

from sparse_moe_transformer_selected_b300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ----------------------------------------------------------------- formats --

def check_e2m1_table(O):
    """All 16 codes against the printed table and the E2M1 bit-field formula."""
    table = {int(c): float(v) for c, v in _golden_rows("e2m1_table.txt")}
    got = O.decode_e2m1(np.arange(16, dtype=np.uint8))
    for c in range(16):
        # bit fields: sign = bit 3, exponent = bits 2..1 (bias 1), mantissa = bit 0
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        closed = (m * 0.5) if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        closed = -closed if s else closed
        assert got[c] == table[c] == closed, (c, got[c], table[c], closed)
        assert math.copysign(1.0, got[c]) == math.copysign(1.0, table[c]), c


def check_e8m0(O):
    for s in (1, 121, 122, 123, 124, 127, 128, 200, 254):
        assert O.decode_e8m0(np.array([s]))[0] == math.ldexp(1.0, s - 127), s
    assert np.isnan(O.decode_e8m0(np.array([255]))[0])


def check_mxfp4_layout(O):
    """Nibble order and scale-block extent, element by element."""
    rng = np.random.Generator(np.random.PCG64(7))
    rows, K = 3, 96
    codes = rng.integers(0, 16, size=(rows, K), dtype=np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = rng.integers(100, 150, size=(rows, K // 32), dtype=np.uint8)
    table = {int(c): float(v) for c, v in _golden_rows("e2m1_table.txt")}
    got = O.dequant_mxfp4(packed, scales)
    assert got.shape == (rows, K)
    for r in range(rows):
        for kk in range(K):
            want = table[int(codes[r, kk])] * math.ldexp(1.0, int(scales[r, kk // 32]) - 127)
            assert got[r, kk] == want, (r, kk, got[r, kk], want)


def check_bits_per_param(O):
    """MXFP4 = 4.25 bits per parameter (weight-quantisation bullet)."""
    for n in (32, 2880 * 5760, 2880 * 2880):
        assert O.mxfp4_storage_bytes(n) * 8 / n == 4.25


def check_bf16_decode(O):
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x0000: 0.0, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x3E80: 0.25, 0x4049: 3.140625}
    for bits, v in cases.items():
        assert O.bf16_bits_to_f64(np.array([bits], np.uint16))[0] == v, hex(bits)


# ------------------------------------------------------------ param counts --

def check_param_arithmetic(O):
    rows = {r[0]: tuple(int(v) for v in r[1:]) for r in _golden_rows("param_arithmetic.txt")}
    d, h, fc1 = rows["fc1"]
    assert O.ffn_params(d, h) == 2 * fc1
    d, h, n = rows["ffn"]
    assert O.ffn_params(d, h) == n == 8_388_608
    d, h, n = rows["glu"]
    assert O.glu_params(d, h) == n == 3 * 1_048_576


def check_model_sizes(O):
    """Expert parameters and MXFP4 storage against the pages' model figures."""
    for name, blocks, experts, dm, width, total, active, ckpt in _golden_rows("model_sizes.txt"):
        blocks, experts, dm, width = int(blocks), int(experts), int(dm), int(width)
        total, active, ckpt = float(total), float(active), float(ckpt)
        per_expert = O.glu_params(dm, width)
        assert per_expert == 24_883_200
        moe = blocks * experts * per_expert
        assert 0.9 * total <= moe <= total, (name, moe)          # "MoE 占总参 90%+"
        assert blocks * 4 * per_expert <= active, name            # top-4 fits the active count
        gib = O.mxfp4_storage_bytes(moe) / 2 ** 30
        assert gib < ckpt, (name, gib)                            # experts fit the checkpoint
        assert gib > 0.7 * ckpt, (name, gib)                      # and are most of it


# ----------------------------------------------------------------- routing --

def check_topk_bruteforce(O):
    rng = np.random.Generator(np.random.PCG64(11))
    # small integers force many exact ties
    logits = rng.integers(-3, 4, size=(200, 9)).astype(np.float64)
    for k in (1, 2, 4, 9):
        idx, gap = O.select_topk(logits, k)
        for t in range(logits.shape[0]):
            want = [e for _, e in sorted((-logits[t, e], e) for e in range(9))][:k]
            assert list(idx[t]) == want, (t, k, list(idx[t]), want)
            srt = sorted(logits[t], reverse=True)
            g = srt[k - 1] - srt[k] if k < 9 else math.inf
            assert gap[t] == g


def check_router_logits(O):
    """logits = x·Wr + b by an exact rational brute force."""
    rng = np.random.Generator(np.random.PCG64(12))
    x = rng.integers(-8, 8, size=(5, 6)).astype(np.float64) / 4
    w = rng.integers(-8, 8, size=(3, 6)).astype(np.float64) / 8
    b = np.array([0.5, -0.25, 1.0])
    got = O.router_logits(x, w, b)
    for t in range(5):
        for e in range(3):
            want = sum(Fraction(x[t, i]) * Fraction(w[e, i]) for i in range(6)) + Fraction(b[e])
            assert Fraction(got[t, e]) == want


def check_selected_softmax(O):
    rng = np.random.Generator(np.random.PCG64(13))
    logits = rng.normal(0, 2, size=(300, 16))
    idx, _ = O.select_topk(logits, 4)
    sel = np.take_along_axis(logits, idx, axis=1)
    w = O.selected_softmax(sel)
    assert np.all(np.abs(w.sum(axis=1) - 1) <= 1e-15)
    assert np.all(np.diff(w, axis=1) <= 0)                 # slots in descending weight
    # renormalising the softmax over all 16 experts gives the same weights
    for t in range(300):
        full = [math.exp(v) for v in logits[t]]
        tot = sum(full)
        p = [full[e] / tot for e in idx[t]]
        ren = [v / sum(p) for v in p]
        assert np.allclose(w[t], ren, rtol=1e-13, atol=0)
    # two equal selected logits get equal weight; one dominant logit gets ~1
    w2 = O.selected_softmax(np.array([[3.0, 3.0, 1.0, 1.0], [50.0, 0.0, 0.0, 0.0]]))
    assert w2[0, 0] == w2[0, 1] and w2[0, 2] == w2[0, 3]
    assert abs(w2[0, 0] - math.e ** 2 / (2 * math.e ** 2 + 2)) < 1e-15
    assert w2[1, 0] == 1.0 and abs(w2[1, 1] - math.exp(-50.0)) < 1e-35


def check_permutation(O):
    rng = np.random.Generator(np.random.PCG64(14))
    for T, E, k in ((1, 4, 4), (50, 8, 4), (37, 32, 4), (100, 6, 2), (20, 5, 1)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        counts, offsets, perm, inv = O.expert_permutation(idx, E)
        # brute-force recount and ordering
        assert sorted(perm.tolist()) == list(range(T * k))        # bijection
        assert int(counts.sum()) == T * k and offsets[E] == T * k and offsets[0] == 0
        row = 0
        for e in range(E):
            members = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
            assert counts[e] == len(members) and offsets[e] == row
            for (t, j) in members:                                # (expert, token, slot) order
                assert perm[row] == t * k + j and inv[t, j] == row
                row += 1
            toks = [perm[r] // k for r in range(offsets[e], offsets[e + 1])]
            assert all(a < b for a, b in zip(toks, toks[1:]))   # strictly ascending


def check_skew_workload(O):
    """The Zipf(1.2) router bias leaves empty experts and a few hot ones."""
    wl = gen.WORKLOADS["gptoss120b_skew16k"]
    x, rw, rb = gen.make_router_inputs(wl)
    logits = O.router_logits(O.bf16_bits_to_f64(x), rw, rb)
    idx, _ = O.select_topk(logits, 4)
    counts, *_ = O.expert_permutation(idx, wl.E)
    frac = counts / wl.T
    assert (counts == 0).sum() >= 1
    assert (frac > 0.10).sum() >= 1


# -------------------------------------------------------------- activation --

def check_activation_spots(O):
    limit, alpha = 7.0, 1.702
    for zg, zu in ((0.3, -0.7), (-2.0, 1.5), (6.9, 6.9), (7.0, 7.0), (7.5, -7.0),
                   (12.0, -9.0), (-30.0, 0.0), (1.0, -1.0), (-7.0, 100.0)):
        g = zg if zg < limit else limit                 # gate clamped from above only
        u = -limit if zu < -limit else (limit if zu > limit else zu)
        want = g * (1.0 / (1.0 + math.exp(-alpha * g))) * (u + 1.0)
        got = O.clamped_swiglu(np.array([zg]), np.array([zu]), limit, alpha)[0]
        assert abs(got - want) <= 1e-15 * max(1.0, abs(want)), (zg, zu, got, want)


def check_plain_swiglu(O):
    """limit = inf, alpha = 1 and z_up shifted by -1 gives Swish(g)·u."""
    rng = np.random.Generator(np.random.PCG64(15))
    zg, zu = rng.normal(0, 3, 200), rng.normal(0, 3, 200)
    got = O.clamped_swiglu(zg, zu - 1.0, math.inf, 1.0)
    for i in range(200):
        swish = zg[i] / (1.0 + math.exp(-zg[i]))        # x·σ(x)
        assert abs(got[i] - swish * zu[i]) <= 1e-13 * max(1.0, abs(swish * zu[i]))


# ------------------------------------------------------------ whole block --

def _tiny_inputs(T, d, W, E, seed, k=4, router_bias="normal"):
    wl = gen.Workload("pin", T=T, d=d, W=W, E=E, k=k, router_bias=router_bias, seed=seed)
    return gen.make_inputs(wl)


def _decode_row(O, packed_row, scale_row):
    """Plain per-element decode via the printed table (independent of dequant_mxfp4)."""
    table = {int(c): float(v) for c, v in _golden_rows("e2m1_table.txt")}
    out = []
    for j, byte in enumerate(packed_row):
        for c in (int(byte) & 15, int(byte) >> 4):
            kk = len(out)
            out.append(table[c] * math.ldexp(1.0, int(scale_row[kk // 32]) - 127))
    return out


def check_e1_k1_dense(O):
    """E = 1, k = 1: the block is one dense gated FFN with weight 1."""
    inp = _tiny_inputs(T=3, d=32, W=32, E=1, seed=21, k=1)
    res = O.moe_forward_inputs(inp)
    assert np.all(res["topk_w"] == 1.0)
    xb = O.bf16_bits_to_f64(inp.x)
    bgu = O.bf16_bits_to_f64(inp.b_gu[0])
    bdn = O.bf16_bits_to_f64(inp.b_dn[0])
    wgu = [_decode_row(O, inp.w_gu[0, n], inp.w_gu_scale[0, n]) for n in range(64)]
    wdn = [_decode_row(O, inp.w_dn[0, n], inp.w_dn_scale[0, n]) for n in range(32)]
    for t in range(3):
        z = [sum(wgu[n][i] * xb[t, i] for i in range(32)) + bgu[n] for n in range(64)]
        h = []
        for n in range(32):
            g = min(z[n], 7.0)
            u = max(-7.0, min(7.0, z[32 + n]))
            h.append(g / (1 + math.exp(-1.702 * g)) * (u + 1))
        for o in range(32):
            y = sum(wdn[o][n] * h[n] for n in range(32)) + bdn[o]
            assert abs(res["out"][t, o] - y) <= 1e-12 * max(1.0, abs(y)), (t, o)


def check_identical_experts(O):
    """All experts equal: the output does not depend on the router."""
    inp = _tiny_inputs(T=6, d=64, W=32, E=5, seed=22)
    for arr in (inp.w_gu, inp.w_gu_scale, inp.b_gu, inp.w_dn, inp.w_dn_scale, inp.b_dn):
        arr[:] = arr[0]
    a = O.moe_forward_inputs(inp)["out"]
    rng = np.random.Generator(np.random.PCG64(23))
    inp.router_w = rng.normal(0, 1, inp.router_w.shape).astype(np.float32)
    inp.router_b = rng.normal(0, 3, inp.router_b.shape).astype(np.float32)
    b = O.moe_forward_inputs(inp)["out"]
    inp1 = _tiny_inputs(T=6, d=64, W=32, E=1, seed=22, k=1)
    for name in ("w_gu", "w_gu_scale", "b_gu", "w_dn", "w_dn_scale", "b_dn"):
        setattr(inp1, name, getattr(inp, name)[:1].copy())
    inp1.x = inp.x
    c = O.moe_forward_inputs(inp1)["out"]
    assert np.allclose(a, b, rtol=1e-13, atol=1e-13)
    assert np.allclose(a, c, rtol=1e-13, atol=1e-13)


def check_preactivation_exact(O):
    """Tiny GEMMs against an exact rational computation (no rounding at all).

    With d = 32, bf16 inputs (8 significant bits) times E2M1·2^s weights (2 bits)
    span well under 53 bits, so the fp64 sums are exact in any order.
    """
    inp = _tiny_inputs(T=2, d=32, W=32, E=4, seed=24)
    res = O.moe_forward_inputs(inp, keep_hidden=True)
    xb = O.bf16_bits_to_f64(inp.x)
    for (t, j), (z, h, y) in res["hidden"].items():
        e = int(res["topk_idx"][t, j])
        bgu = O.bf16_bits_to_f64(inp.b_gu[e])
        for n in range(64):
            row = _decode_row(O, inp.w_gu[e, n], inp.w_gu_scale[e, n])
            want = sum(Fraction(row[i]) * Fraction(xb[t, i]) for i in range(32)) + Fraction(bgu[n])
            assert Fraction(z[n]) == want, (t, j, n)


def check_weighted_combine(O):
    """out = Σ_j w_j·y_j with the expert bias inside y_j, checked on one token by
    recomputing each selected expert as its own E = 1 layer."""
    inp = _tiny_inputs(T=4, d=64, W=64, E=6, seed=25)
    res = O.moe_forward_inputs(inp)
    for t in range(4):
        acc = np.zeros(64)
        for j in range(4):
            e = int(res["topk_idx"][t, j])
            one = _tiny_inputs(T=4, d=64, W=64, E=1, seed=25, k=1)
            for name in ("w_gu", "w_gu_scale", "b_gu", "w_dn", "w_dn_scale", "b_dn"):
                setattr(one, name, getattr(inp, name)[e:e + 1].copy())
            one.x = inp.x
            y = O.moe_forward_inputs(one)["out"][t]
            acc += res["topk_w"][t, j] * y
        assert np.allclose(res["out"][t], acc, rtol=1e-12, atol=1e-12)
    # which experts: the four largest logits of an independent dot product
    xb = O.bf16_bits_to_f64(inp.x)
    for t in range(4):
        lg = [sum(float(xb[t, i]) * float(inp.router_w[e, i]) for i in range(64))
              + float(inp.router_b[e]) for e in range(6)]
        want = sorted(range(6), key=lambda e: (-lg[e], e))[:4]
        assert list(res["topk_idx"][t]) == want


def check_sampled_tokens(O):
    """Computing a sample of tokens gives the same rows as the full run."""
    inp = _tiny_inputs(T=16, d=64, W=32, E=8, seed=26)
    full = O.moe_forward_inputs(inp)["out"]
    sub = O.moe_forward_inputs(inp, tokens=[13, 2, 7])["out"]
    # BLAS may block a 3-row product differently from a 16-row one
    assert np.allclose(sub, full[[13, 2, 7]], rtol=1e-13, atol=1e-13)


def check_threaded_experts(O):
    """Running the experts on several threads changes nothing, bit for bit."""
    inp = _tiny_inputs(T=24, d=64, W=32, E=8, seed=27)
    a = O.moe_forward_inputs(inp)["out"]
    b = O.moe_forward_inputs(inp, workers=4)["out"]
    assert np.array_equal(a, b)


# --------------------------------------------------------- the step before --

def _decimal_rms_norm(row, weight, eps):
    """x / sqrt(mean(x²) + eps) · g in 50-digit decimal arithmetic from the exact
    binary values: an independent brute force of RMSNorm ([P3] 2.7.1)."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    xs = [Fraction(float(v)) for v in row]
    ms = sum(v * v for v in xs) / len(xs) + Fraction(float(eps))
    rms = (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
    return [float(Decimal(v.numerator) / Decimal(v.denominator) / rms * Decimal(float(g)))
            for v, g in zip(xs, weight)]


def _bf16_value(bits):
    """A bf16 bit pattern's value, through the float32 byte layout (struct)."""
    import struct
    return struct.unpack(">f", struct.pack(">I", int(bits) << 16))[0]


def check_rms_norm_decimal(O):
    rng = np.random.Generator(np.random.PCG64(31))
    cases = [(rng.normal(0, 1, 16), rng.normal(1, 0.1, 16), 1e-5),
             (rng.normal(0, 30, 48), rng.normal(1, 0.5, 48), 0.5),
             (np.concatenate([rng.normal(0, 1e-3, 31), [250.0]]), np.ones(32), 0.0),
             (np.full(8, -3.0), rng.normal(0, 2, 8), 1e-5)]
    for row, g, eps in cases:
        got = O.rms_norm(row[None, :], g, eps)[0]
        want = _decimal_rms_norm(row, g, eps)
        for i in range(len(row)):
            assert abs(got[i] - want[i]) <= 1e-14 * max(1e-300, abs(want[i])), (i, got[i], want[i])


def check_rms_norm_no_mean_no_bias(O):
    """RMSNorm subtracts no mean and adds no bias ([P3] 2.7.1; [P5] "RMSNorm 替换
    LayerNorm"): a constant row maps to ±1 (a mean-subtracting norm gives 0), a
    zero row stays zero, scaling a row by a power of two changes nothing, and
    with g = 1 and eps = 0 every output row has RMS 1."""
    d = 24
    for c in (2.5, -0.75):
        assert np.array_equal(O.rms_norm(np.full((1, d), c), np.ones(d), 0.0)[0],
                              np.full(d, math.copysign(1.0, c)))
    assert np.array_equal(O.rms_norm(np.zeros((1, d)), np.ones(d), 1e-5)[0], np.zeros(d))
    rng = np.random.Generator(np.random.PCG64(32))
    x = rng.normal(0, 1, (5, d))
    g = rng.normal(1, 0.2, d)
    assert np.array_equal(O.rms_norm(8.0 * x, g, 0.0), O.rms_norm(x, g, 0.0))
    y = O.rms_norm(x, np.ones(d), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-15, atol=0)


def _bf16_round_bits(v):
    """Nearest bf16 of a float64 by integer arithmetic on its IEEE bits: keep
    the sign, exponent and top 7 fraction bits, and round the 45 dropped bits
    half to even (normal range only)."""
    import struct
    b = struct.unpack(">Q", struct.pack(">d", float(v)))[0]
    keep, drop = b >> 45, b & ((1 << 45) - 1)
    half = 1 << 44
    if drop > half or (drop == half and keep & 1):
        keep += 1
    return struct.unpack(">d", struct.pack(">Q", keep << 45))[0]


def check_round_bf16(O):
    """bf16 rounding against integer rounding of the IEEE bits, at random
    values and at constructed midpoints (ties go to the even neighbour)."""
    rng = np.random.Generator(np.random.PCG64(37))
    vals = np.concatenate([rng.normal(0, 1, 400), rng.normal(0, 1e3, 100),
                           [1.0, -2.5, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8),
                            1 + 2.0 ** -8 + 2.0 ** -40, 0.0]])
    got = O.round_bf16(vals)
    for v, r in zip(vals, got):
        assert r == _bf16_round_bits(v), (v, r)
    assert O.round_bf16(1 + 2.0 ** -8) == 1.0                     # tie, even below
    assert O.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6       # tie, even above


def check_block_rounds_moe_input(O):
    """E = 1, k = 1 block on a tiny layer against a brute force: RMSNorm in
    50-digit decimal, rounded to bf16 by integer bit arithmetic, then the dense
    gated FFN in plain Python; block - x must equal it."""
    inp = _block_inputs(T=3, d=32, W=32, E=1, seed=38, k=1)
    res = O.moe_block_forward_inputs(inp)
    xb = [[_bf16_value(b) for b in row] for row in inp.x]
    bgu = [_bf16_value(b) for b in inp.b_gu[0]]
    bdn = [_bf16_value(b) for b in inp.b_dn[0]]
    wgu = [_decode_row(O, inp.w_gu[0, n], inp.w_gu_scale[0, n]) for n in range(64)]
    wdn = [_decode_row(O, inp.w_dn[0, n], inp.w_dn_scale[0, n]) for n in range(32)]
    for t in range(3):
        xn = [_bf16_round_bits(v) for v in _decimal_rms_norm(xb[t], inp.norm_w, inp.eps)]
        z = [sum(wgu[n][i] * xn[i] for i in range(32)) + bgu[n] for n in range(64)]
        h = []
        for n in range(32):
            g = min(z[n], 7.0)
            u = max(-7.0, min(7.0, z[32 + n]))
            h.append(g / (1 + math.exp(-1.702 * g)) * (u + 1))
        for o in range(32):
            y = sum(wdn[o][n] * h[n] for n in range(32)) + bdn[o]
            got = res["out"][t, o] - xb[t][o]
            assert abs(got - y) <= 1e-12 * max(1.0, abs(y)), (t, o, got, y)


def _block_inputs(T, d, W, E, seed, k=4):
    wl = gen.Workload("pin", T=T, d=d, W=W, E=E, k=k, router_bias="normal", seed=seed)
    return gen.make_block_inputs(wl)


def check_block_residual(O):
    """The block adds the MoE output to the un-normalised input: with every
    expert's output zero (down codes 0, down bias 0) the block returns x
    exactly; with rows of RMS 1 (entries ±1), g = 1 and eps = 0 the norm is the
    identity and the block is x plus the MoE of x."""
    inp = _block_inputs(T=5, d=64, W=32, E=6, seed=33)
    inp.w_dn[:] = 0
    inp.b_dn[:] = 0
    out = O.moe_block_forward_inputs(inp)["out"]
    for t in range(5):
        for i in range(64):
            assert out[t, i] == _bf16_value(inp.x[t, i]), (t, i)
    inp = _block_inputs(T=6, d=64, W=32, E=6, seed=34)
    signs = np.random.Generator(np.random.PCG64(35)).integers(0, 2, size=(6, 64))
    inp.x = np.where(signs == 1, 0x3F80, 0xBF80).astype(np.uint16)      # +1.0 / -1.0
    inp.norm_w = np.ones(64, dtype=np.float32)
    inp.eps = 0.0
    blk = O.moe_block_forward_inputs(inp)["out"]
    moe = O.moe_forward_inputs(inp)["out"]
    xv = np.where(signs == 1, 1.0, -1.0)
    assert np.allclose(blk, xv + moe, rtol=1e-13, atol=1e-13)


def check_block_scale_invariance(O):
    """With eps = 0, scaling the input by 4 scales the residual part only: the
    MoE reads RMSNorm(x), which does not change, so block(4x) - 4x equals
    block(x) - x."""
    inp = _block_inputs(T=6, d=64, W=32, E=6, seed=36)
    inp.eps = 0.0
    a = O.moe_block_forward_inputs(inp)
    xa = np.array([[_bf16_value(b) for b in row] for row in inp.x])
    inp.x = (inp.x.astype(np.int64) + (2 << 7)).astype(np.uint16)   # exponent + 2: times 4
    b = O.moe_block_forward_inputs(inp)
    assert np.allclose(b["out"] - 4.0 * xa, a["out"] - xa, rtol=1e-12, atol=1e-12)
    assert np.array_equal(a["topk_idx"], b["topk_idx"])


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
