"""The activation number formats of the block-scaled GEMM design, checked on the
host with torch's E4M3 conversion (round to nearest even): the two-term split
of bf16 x with a power-of-two scale per 32-element block is exact, and the
four-term split of h with one fixed scale keeps about 16 significant bits.
These are properties of the formats, independent of any kernel."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def e4m3(v: torch.Tensor) -> torch.Tensor:
    """Round to E4M3 (nearest even) and back to float64."""
    return v.to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64)


def all_bf16_below(m: float) -> torch.Tensor:
    """Every finite bf16 value with magnitude <= m, as float64."""
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).to(torch.float64)
    v = v[torch.isfinite(v)]
    return v[v.abs() <= m]


@pytest.mark.parametrize("m", [1.0, 1.75, 3.0, 300.0, 2.0 ** -20])
def test_two_term_split_of_bf16_is_exact_within_the_block(m):
    """x = (hi + lo/16) 2^e_b with e_b = floor(log2 m) - 7 for the block's
    largest |x| = m: every bf16 value within 2^-7 of m (relative) is exact, and
    smaller ones are off by at most 2^-13 of m (E4M3 subnormals)."""
    e_b = int(np.floor(np.log2(m))) - 7
    v = all_bf16_below(m)
    s = v * 2.0 ** (-e_b)
    assert s.abs().max() < 448
    hi = e4m3(s)
    lo = e4m3((s - hi) * 16.0)
    rec = (hi + lo / 16.0) * 2.0 ** e_b
    big = v.abs() >= m * 2.0 ** -7
    assert torch.equal(rec[big], v[big])
    assert (rec - v).abs().max() <= m * 2.0 ** -13


def four_terms(h: torch.Tensor, e: int) -> torch.Tensor:
    v = h * 2.0 ** (-e)
    rec = torch.zeros_like(v)
    r = v.clone()
    for t in range(4):
        q = e4m3(r)
        rec += q / 16.0 ** t
        r = (r - q) * 16.0
    return rec * 2.0 ** e


@pytest.mark.parametrize("limit", [7.0, 1.0, 16.0])
def test_four_term_split_of_h_keeps_16_bits(limit):
    """h = (t0 + t1/16 + t2/256 + t3/4096) 2^e with 2^-e the largest power of
    two that keeps limit (limit + 1) within E4M3's 448: relative error at most
    2^-16 over the 14 binades below the bound; below that, absolute error at
    most 2^(e - 21) (the last term's E4M3 subnormal step)."""
    bound = limit * (limit + 1)
    e = 0
    while bound * 2.0 ** (-e) > 448:
        e += 1
    while bound * 2.0 ** (-(e - 1)) <= 448:
        e -= 1
    rng = np.random.default_rng(0)
    mags = bound * 2.0 ** rng.uniform(-14, 0, 200000)
    h = torch.from_numpy(mags * rng.choice([-1.0, 1.0], mags.size))
    err = (four_terms(h, e) - h).abs()
    assert (err / h.abs()).max() <= 2.0 ** -16
    tiny = torch.from_numpy(bound * 2.0 ** rng.uniform(-30, -14, 20000))
    assert (four_terms(tiny, e) - tiny).abs().max() <= 2.0 ** (e - 21)


def test_scale_exponent_matches_the_library():
    """The exponent above is the one moe_hidden_format reports (limit 7: 2^-3)."""
    from sparse_moe_transformer_selected_b300 import build, moe
    build.build()
    moe.load()
    fmt, ex = moe.moe_hidden_format(32, 2880, 2880, 32, 4, 7.0)
    assert fmt == moe.HIDDEN_E4M3_TERMS and ex == -3
