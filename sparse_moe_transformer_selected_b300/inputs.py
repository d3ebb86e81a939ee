"""Seeded synthetic inputs for the gpt-oss MoE MLP block.

This module only draws random numbers and packs them into the storage formats
the library consumes (bf16 bit patterns, packed E2M1 nibbles, E8M0 bytes).  It
holds none of the block's arithmetic: no decoding of those formats, no routing,
no matrix products.  Both the CPU oracle (through the tests) and the CUDA path
are fed from here, so the two sides always see the same bytes.

Draw order (one numpy PCG64 stream per workload, seed 0 unless stated):
x, router_w, router_b, W_gu codes, W_gu scales, b_gu, W_dn codes, W_dn scales,
b_dn.

Shapes follow the pages' gpt-oss layer: d_model = expert width = 2880
("更深对比更宽" section of "OpenAI 最新开源模型 gpt-oss 架构与训练解析"),
E = 32 (20b) or 128 (120b) experts, top-4 ("模型架构", MoE bullet, same page).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named MoE-layer shape plus the recipe of its synthetic values."""

    name: str
    T: int            # tokens
    d: int            # d_model
    W: int            # expert (intermediate) width
    E: int            # experts
    k: int = 4        # experts per token
    router_bias: str = "zero"      # "zero" | "normal" | "zipf"
    router_bias_std: float = 0.1   # for "normal"
    zipf_s: float = 1.2            # for "zipf": popularity p_e ∝ e^-s
    zipf_c: float = 1.0            # for "zipf": router_b[π(e)] = c·ln p_e
    scale_lo: int = -6             # E8M0 scale = 127 + U{scale_lo..scale_hi}
    scale_hi: int = -3
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the gpt-oss MoE layer used for parity and timing.
WORKLOADS = {
    "tiny": Workload("tiny", T=64, d=256, W=256, E=8, router_bias="normal"),
    "gptoss20b_decode": Workload("gptoss20b_decode", T=32, d=2880, W=2880, E=32),
    "gptoss20b_prefill": Workload("gptoss20b_prefill", T=8192, d=2880, W=2880, E=32),
    "gptoss120b_prefill": Workload("gptoss120b_prefill", T=4096, d=2880, W=2880, E=128),
    "gptoss120b_skew16k": Workload("gptoss120b_skew16k", T=16384, d=2880, W=2880, E=128,
                                   router_bias="zipf"),
    "gptoss120b_skew64": Workload("gptoss120b_skew64", T=64, d=2880, W=2880, E=128,
                                  router_bias="zipf"),
}

# A second MoE shape as a stress of the same kernels (another model's layer:
# d = 2048, expert width 768, 128 experts, top-8); not a pages' configuration.
STRESS_WORKLOADS = {
    "qwen3_30b_a3b_decode": Workload("qwen3_30b_a3b_decode", T=32, d=2048, W=768, E=128, k=8,
                                     seed=31),
    "qwen3_30b_a3b_prefill": Workload("qwen3_30b_a3b_prefill", T=2048, d=2048, W=768, E=128,
                                      k=8, seed=32),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return uint16 bits.

    Inputs here are finite draws, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


@dataclasses.dataclass
class MoEInputs:
    """Host copies of every argument of the block, in the library's layouts.

    x          uint16 [T, d]          bf16 bit patterns, row-major
    router_w   float32 [E, d]
    router_b   float32 [E]
    w_gu       uint8  [E, 2W, d/2]    rows [0,W) gate, [W,2W) up; byte j holds
                                      K index 2j in its low nibble, 2j+1 high
    w_gu_scale uint8  [E, 2W, d/32]   E8M0, one per 32 consecutive K
    b_gu       uint16 [E, 2W]         bf16 bits
    w_dn       uint8  [E, d, W/2]
    w_dn_scale uint8  [E, d, W/32]
    b_dn       uint16 [E, d]          bf16 bits
    """

    wl: Workload
    x: np.ndarray
    router_w: np.ndarray
    router_b: np.ndarray
    w_gu: np.ndarray
    w_gu_scale: np.ndarray
    b_gu: np.ndarray
    w_dn: np.ndarray
    w_dn_scale: np.ndarray
    b_dn: np.ndarray
    limit: float = 7.0
    alpha: float = 1.702
    # the step before the block (make_block_inputs): RMSNorm weight [d] and eps;
    # x is then the un-normalised residual stream
    norm_w: np.ndarray | None = None
    eps: float = 1e-5


def _router_bias(rng: np.random.Generator, wl: Workload) -> np.ndarray:
    if wl.router_bias == "zero":
        return np.zeros(wl.E, dtype=np.float32)
    if wl.router_bias == "normal":
        return rng.normal(0.0, wl.router_bias_std, size=wl.E).astype(np.float32)
    if wl.router_bias == "zipf":
        ranks = np.arange(1, wl.E + 1, dtype=np.float64)
        p = ranks ** (-wl.zipf_s)
        p /= p.sum()
        pi = rng.permutation(wl.E)
        b = np.empty(wl.E, dtype=np.float64)
        b[pi] = wl.zipf_c * np.log(p)
        return b.astype(np.float32)
    raise ValueError(f"unknown router_bias recipe {wl.router_bias!r}")


def make_inputs(wl: Workload, limit: float = 7.0, alpha: float = 1.702) -> MoEInputs:
    """Draw one workload's inputs (see the module docstring for the order)."""
    if wl.d % 32 or wl.W % 32:
        raise ValueError("d and W must be multiples of the 32-element MX block")
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    T, d, W, E = wl.T, wl.d, wl.W, wl.E
    x = f32_to_bf16_bits(rng.standard_normal((T, d), dtype=np.float32))
    router_w = (rng.standard_normal((E, d), dtype=np.float32)
                * np.float32(1.0 / math.sqrt(d))).astype(np.float32)
    router_b = _router_bias(rng, wl)
    w_gu = rng.integers(0, 256, size=(E, 2 * W, d // 2), dtype=np.uint8)
    w_gu_scale = (127 + rng.integers(wl.scale_lo, wl.scale_hi + 1,
                                     size=(E, 2 * W, d // 32))).astype(np.uint8)
    b_gu = f32_to_bf16_bits(rng.normal(0.0, 0.02, size=(E, 2 * W)).astype(np.float32))
    w_dn = rng.integers(0, 256, size=(E, d, W // 2), dtype=np.uint8)
    w_dn_scale = (127 + rng.integers(wl.scale_lo, wl.scale_hi + 1,
                                     size=(E, d, W // 32))).astype(np.uint8)
    b_dn = f32_to_bf16_bits(rng.normal(0.0, 0.02, size=(E, d)).astype(np.float32))
    return MoEInputs(wl, x, router_w, router_b, w_gu, w_gu_scale, b_gu,
                     w_dn, w_dn_scale, b_dn, limit=limit, alpha=alpha)


def mxfp4_bytes_per_expert(d: int, W: int) -> int:
    """Bytes of packed E2M1 codes plus E8M0 scales for one expert's three matrices."""
    n = 2 * W * d + d * W
    return n // 2 + n // 32


def make_router_inputs(wl: Workload):
    """Only the first three draws of make_inputs (x, router_w, router_b).

    Same stream prefix, so the values equal those of make_inputs(wl); used where
    only routing is needed and the expert weights would be wasted memory.
    """
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    T, d, E = wl.T, wl.d, wl.E
    x = f32_to_bf16_bits(rng.standard_normal((T, d), dtype=np.float32))
    router_w = (rng.standard_normal((E, d), dtype=np.float32)
                * np.float32(1.0 / math.sqrt(d))).astype(np.float32)
    router_b = _router_bias(rng, wl)
    return x, router_w, router_b


def make_block_inputs(wl: Workload, limit: float = 7.0, alpha: float = 1.702,
                      eps: float = 1e-5) -> MoEInputs:
    """Inputs of the pre-norm block (RMSNorm, the MoE, the residual add).

    The router and expert arguments are those of make_inputs(wl); a second
    stream, PCG64([seed, 1]), then draws the residual stream and the RMSNorm
    weight, in this order:
      s_t    per-token magnitude, exp(N(0, 0.5))  (tokens of unequal RMS)
      x      bf16 of s_t times N(0, 1)            [T, d], replaces make_inputs' x
      norm_w float32, 1 + N(0, 0.1)               [d]
    """
    inp = make_inputs(wl, limit=limit, alpha=alpha)
    rng = np.random.Generator(np.random.PCG64([wl.seed, 1]))
    s_t = np.exp(rng.normal(0.0, 0.5, size=(wl.T, 1))).astype(np.float32)
    z = rng.standard_normal((wl.T, wl.d), dtype=np.float32)
    inp.x = f32_to_bf16_bits((z * s_t).astype(np.float32))
    inp.norm_w = (1.0 + rng.normal(0.0, 0.1, size=wl.d)).astype(np.float32)
    inp.eps = float(np.float32(eps))       # the value a float32 argument carries
    return inp
