"""CPU oracle for the gpt-oss Mixture-of-Experts MLP block.

TEST INFRASTRUCTURE ONLY.  This is the plain, slow, fp64 definition of what the
CUDA library computes, used to check it.  Only the tests, the smoke entry point
and the benchmark's CPU-baseline leg may import it; the library itself never
does, and it shares no code, table or helper with the CUDA sources.

Sources (web pages about the gpt-oss architecture, cited by title and section):

* [P5] "OpenAI 最新开源模型 gpt-oss 架构与训练解析" (dtcms.com/a/486625)
  - section "模型架构", MoE bullet: 32 (20b) / 128 (120b) experts, top-4
    routing, softmax weighting of the selected experts, FFN = gated-SwiGLU
    variant with clamping and a residual term.
  - section "模型架构", weight-quantisation bullet: MoE weights in MXFP4,
    4.25 bits per parameter.
  - section "Swish/SwiGLU 替换 GELU": Swish(x) = x·σ(x).
  - section "更深对比更宽": d_model 2880, expert projection width 2880.
  - section "更少的大专家 vs 更多的小专家": 4 active experts per token, no
    shared expert.
* [P3] "【LLM】GPT-OSS架构变化详解" (dtcms.com/a/386406), section 2.4 (MoE
  replaces the single FFN; a router picks experts per token) and 1.2 (top-4 of
  the experts are activated per token).
* [P4] Xin Zhiyuan report (dreamgost.com .../564), GLU discussion around
  Figure 6: a gated FFN has three weight matrices instead of two; the
  parameter arithmetic FC1+FC2 = 8,388,608 vs 3 x 1,048,576 = 3,145,728.
* The step before the block (rms_norm, moe_block_forward): [P3] 2.7.1 and
  [P5] "RMSNorm 替换 LayerNorm" — RMSNorm divides the activations by their root
  mean square, with no mean subtraction and no bias term; [P5] "更深对比更宽"
  — residual connections around the sub-layers.

Facts the pages leave open, and the reading taken here:

* limit = 7.0 and alpha = 1.702; the gate is clamped from above only, the up
  branch on both sides; the "residual" is the +1 on the up branch:
  h = g·σ(alpha·g)·(u + 1) with g = min(z_g, limit), u = clamp(z_u, ±limit).
* MXFP4: each block of 32 consecutive K elements of a weight row holds 32 E2M1
  codes and one E8M0 scale byte; value = sign·{0,.5,1,1.5,2,3,4,6}[m]·2^(s-127);
  s = 255 is NaN.  Packed two codes per byte, the even K index in the low
  nibble.
* Router bias present (fp32); ties in the top-4 broken towards the lower expert
  index; the four slots of a token ordered by (logit descending, index
  ascending).
* W_gu rows [0, W) are the gate projection, rows [W, 2W) the up projection.
* Expert biases b_gu, b_dn are bf16 and sit inside each expert, so the down
  bias is scaled by the routing weight.
* Permuted ("expert-contiguous") row order: rows sorted by (expert, token,
  slot) ascending.
* RMSNorm keeps the usual learned per-feature scale g and a small eps inside
  the square root (the pages name neither): x / sqrt(mean(x²) + eps) · g.  The
  block is pre-norm: the MoE reads RMSNorm(x) and its output is added to the
  un-normalised x, out = x + MoE(RMSNorm(x)).  The MoE's input is bf16 (its x
  is a bf16 tensor), so RMSNorm's output enters it rounded to the nearest bf16,
  ties to even: the one rounding this oracle performs, because it is part of
  what the block computes.

Apart from that input rounding of the block, the oracle rounds nothing: every
intermediate stays fp64.
"""
from __future__ import annotations

import numpy as np

# E2M1 magnitudes indexed by the low three bits of a code (exponent bits 2..1,
# mantissa bit 0); bit 3 is the sign.  OCP MX element format.
E2M1_MAGNITUDE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
MX_BLOCK = 32


# ---------------------------------------------------------------- formats --

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """A bf16 bit pattern is the upper half of the float32 with the same value."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """E2M1 code (0..15) -> value, by the table above ([P5] 权重量化 bullet)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = np.asarray(E2M1_MAGNITUDE, dtype=np.float64)[c & 7]
    return np.where(c & 8, -mag, mag)


def decode_e8m0(scales: np.ndarray) -> np.ndarray:
    """E8M0 byte s -> 2^(s-127); s = 255 encodes NaN."""
    s = np.asarray(scales, dtype=np.int64)
    v = np.ldexp(1.0, s - 127)
    return np.where(s == 255, np.nan, v)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] codes; the even K index is the low nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0x0F
    out[..., 1::2] = p >> 4
    return out


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP4 matrix [rows, K/2] codes + [rows, K/32] scales -> fp64 [rows, K].

    Every value is an E2M1 magnitude times a power of two, so the fp64 result is
    exact.
    """
    vals = decode_e2m1(unpack_e2m1(packed))
    sc = np.repeat(decode_e8m0(scales), MX_BLOCK, axis=-1)
    return vals * sc


def mxfp4_storage_bytes(n_params: int) -> float:
    """Bytes to store n MXFP4 parameters: 4-bit codes plus one byte per 32."""
    return n_params * 4 / 8 + n_params / MX_BLOCK


# -------------------------------------------------------- parameter counts --

def ffn_params(d_model: int, hidden: int) -> int:
    """Plain two-layer FFN, no biases: FC1 (d x h) + FC2 (h x d)."""
    return 2 * d_model * hidden


def glu_params(d_model: int, hidden: int) -> int:
    """Gated FFN, no biases: gate, up and down, three d x h matrices ([P4] Fig. 6)."""
    return 3 * d_model * hidden


# ---------------------------------------------------------------- routing --

def router_logits(x: np.ndarray, router_w: np.ndarray, router_b: np.ndarray) -> np.ndarray:
    """logits[t, e] = x[t]·Wr[e] + br[e], fp64 ([P3] 2.4.1, [P5] MoE bullet)."""
    return np.asarray(x, np.float64) @ np.asarray(router_w, np.float64).T \
        + np.asarray(router_b, np.float64)


def select_topk(logits: np.ndarray, k: int):
    """Top-k experts per token, slots ordered by (logit desc, expert index asc).

    Returns (idx [T,k] int64, gap [T]) where gap is the k-th minus the (k+1)-th
    largest logit (inf when E == k); a small gap marks a near-tie.
    """
    l = np.asarray(logits, np.float64)
    order = np.argsort(-l, axis=1, kind="stable")  # stable: lower index first on ties
    idx = order[:, :k]
    srt = np.take_along_axis(l, order, axis=1)
    if l.shape[1] > k:
        gap = srt[:, k - 1] - srt[:, k]
    else:
        gap = np.full(l.shape[0], np.inf)
    return idx, gap


def selected_softmax(sel_logits: np.ndarray) -> np.ndarray:
    """Softmax over only the k selected logits of each token ([P5] MoE bullet)."""
    s = np.asarray(sel_logits, np.float64)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True)


def expert_permutation(topk_idx: np.ndarray, E: int):
    """Expert-contiguous order of the T·k routed rows.

    Rows are sorted by (expert, token, slot).  Returns
      counts  [E]      rows per expert
      offsets [E+1]    exclusive prefix sum of counts, offsets[E] = T·k
      perm    [T·k]    row -> t·k + j
      inv     [T, k]   (t, j) -> row
    """
    idx = np.asarray(topk_idx, np.int64)
    T, k = idx.shape
    expert = idx.reshape(-1)
    flat = np.arange(T * k)
    token, slot = flat // k, flat % k
    perm = np.lexsort((slot, token, expert))
    counts = np.bincount(expert, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    inv = np.empty(T * k, dtype=np.int64)
    inv[perm] = np.arange(T * k)
    return counts, offsets, perm, inv.reshape(T, k)


# ------------------------------------------------------------- expert FFN --

def sigmoid(v: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-v))


def clamped_swiglu(z_gate: np.ndarray, z_up: np.ndarray, limit: float, alpha: float) -> np.ndarray:
    """Gated-SwiGLU with clamping and the +1 on the up branch ([P5] MoE bullet).

    g = min(z_gate, limit); u = clamp(z_up, -limit, limit); h = g·σ(alpha·g)·(u+1).
    With limit = inf, alpha = 1 and the +1 absorbed into the up bias this is the
    textbook SwiGLU, Swish(g)·u ([P5] "Swish/SwiGLU 替换 GELU").
    """
    g = np.minimum(z_gate, limit)
    u = np.clip(z_up, -limit, limit)
    return g * sigmoid(alpha * g) * (u + 1.0)


def expert_ffn(x_rows, w_gu, b_gu, w_dn, b_dn, limit, alpha):
    """One expert on its rows: fp64 weights already dequantised.

    w_gu [2W, d] (gate rows then up rows), b_gu [2W], w_dn [d, W], b_dn [d].
    Returns (z [n, 2W], h [n, W], y [n, d]).
    """
    W = w_dn.shape[1]
    z = x_rows @ w_gu.T + b_gu
    h = clamped_swiglu(z[:, :W], z[:, W:], limit, alpha)
    y = h @ w_dn.T + b_dn
    return z, h, y


# ------------------------------------------------------------ whole block --

def moe_forward(x_bits, router_w, router_b, w_gu, w_gu_scale, b_gu_bits,
                w_dn, w_dn_scale, b_dn_bits, k=4, limit=7.0, alpha=1.702,
                tokens=None, keep_hidden=False, workers=1):
    """The MoE MLP block on fp64: router -> top-k -> selected softmax -> experts
    -> weighted sum ([P5] MoE bullet; [P3] 2.4.1).  No shared expert is added
    ([P5] "更少的大专家 vs 更多的小专家").

    Routing (logits, top-k, weights, permutation) is computed for all T tokens.
    The expert FFN runs for `tokens` only (default: all), so large layers can be
    checked on a sample.  Returns a dict; "out" has one row per entry of
    `tokens` in that order.  `workers` > 1 runs the experts on that many threads
    (numpy releases the interpreter lock inside its loops); each expert's rows
    are computed exactly as with one thread and added in expert order.
    """
    return moe_forward_f64(bf16_bits_to_f64(x_bits), router_w, router_b, w_gu, w_gu_scale,
                           b_gu_bits, w_dn, w_dn_scale, b_dn_bits, k=k, limit=limit,
                           alpha=alpha, tokens=tokens, keep_hidden=keep_hidden, workers=workers)


def moe_forward_f64(x, router_w, router_b, w_gu, w_gu_scale, b_gu_bits,
                    w_dn, w_dn_scale, b_dn_bits, k=4, limit=7.0, alpha=1.702,
                    tokens=None, keep_hidden=False, workers=1):
    """moe_forward on activations already in fp64 (the block's normalised x)."""
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    E = router_w.shape[0]
    logits = router_logits(x, router_w, router_b)
    idx, gap = select_topk(logits, k)
    w = selected_softmax(np.take_along_axis(logits, idx, axis=1))
    counts, offsets, perm, inv = expert_permutation(idx, E)

    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.zeros((tok.shape[0], x.shape[1]), dtype=np.float64)
    hidden = {} if keep_hidden else None
    b_gu = bf16_bits_to_f64(b_gu_bits)
    b_dn = bf16_bits_to_f64(b_dn_bits)
    sel = idx[tok]                               # [n, k]

    def one_expert(e):
        pos, slot = np.nonzero(sel == e)         # sampled position, slot
        wg = dequant_mxfp4(w_gu[e], w_gu_scale[e])
        wd = dequant_mxfp4(w_dn[e], w_dn_scale[e])
        return pos, slot, expert_ffn(x[tok[pos]], wg, b_gu[e], wd, b_dn[e], limit, alpha)

    experts = np.unique(sel)
    if workers > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=workers) as pool:
            results = list(pool.map(one_expert, experts))
    else:
        results = [one_expert(e) for e in experts]
    for pos, slot, (z, h, y) in results:         # expert order
        out[pos] += w[tok[pos], slot][:, None] * y   # each (pos, e) occurs once
        if keep_hidden:
            for r, (p, j) in enumerate(zip(pos, slot)):
                hidden[(int(tok[p]), int(j))] = (z[r], h[r], y[r])
    res = dict(out=out, logits=logits, topk_idx=idx, topk_w=w, gap=gap,
               counts=counts, offsets=offsets, perm=perm, inv=inv, tokens=tok)
    if keep_hidden:
        res["hidden"] = hidden
    return res


def moe_forward_inputs(inp, tokens=None, keep_hidden=False, workers=1):
    """moe_forward on a MoEInputs bundle."""
    return moe_forward(inp.x, inp.router_w, inp.router_b, inp.w_gu, inp.w_gu_scale,
                       inp.b_gu, inp.w_dn, inp.w_dn_scale, inp.b_dn, k=inp.wl.k,
                       limit=inp.limit, alpha=inp.alpha, tokens=tokens,
                       keep_hidden=keep_hidden, workers=workers)


# --------------------------------------------------------- the step before --

def rms_norm(x, weight, eps):
    """RMSNorm ([P3] 2.7.1; [P5] "RMSNorm 替换 LayerNorm"): each row divided by
    its root mean square, with no mean subtracted and no bias added, then
    scaled by the per-feature weight: x / sqrt(mean(x²) + eps) · weight."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)


def round_bf16(v):
    """Nearest bf16 value (8 significant bits), ties to even, for finite v in
    the normal range: v = m·2^e with 0.5 <= |m| < 1, m rounded to a multiple of
    2^-8 (numpy's rint rounds halves to even)."""
    m, e = np.frexp(np.asarray(v, np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def moe_block_forward(x_bits, norm_w, eps, router_w, router_b, w_gu, w_gu_scale, b_gu_bits,
                      w_dn, w_dn_scale, b_dn_bits, k=4, limit=7.0, alpha=1.702,
                      tokens=None, keep_hidden=False, workers=1):
    """The MoE sub-layer of a pre-norm block with its residual connection:
    out = x + MoE(bf16(RMSNorm(x))), x the un-normalised residual stream ([P5]
    "更深对比更宽": residual connections; "RMSNorm 替换 LayerNorm"); the MoE's
    input is bf16.  Returns the moe_forward dict with "out" replaced by the block
    output and "normed" holding the MoE input bf16(RMSNorm(x)) of every token.
    """
    x = bf16_bits_to_f64(x_bits)
    xn = round_bf16(rms_norm(x, norm_w, eps))
    res = moe_forward_f64(xn, router_w, router_b, w_gu, w_gu_scale, b_gu_bits, w_dn,
                          w_dn_scale, b_dn_bits, k=k, limit=limit, alpha=alpha, tokens=tokens,
                          keep_hidden=keep_hidden, workers=workers)
    res["out"] = x[res["tokens"]] + res["out"]
    res["normed"] = xn
    return res


def moe_block_forward_inputs(inp, tokens=None, keep_hidden=False, workers=1):
    """moe_block_forward on a MoEInputs bundle that carries norm_w and eps."""
    return moe_block_forward(inp.x, inp.norm_w, inp.eps, inp.router_w, inp.router_b, inp.w_gu,
                             inp.w_gu_scale, inp.b_gu, inp.w_dn, inp.w_dn_scale, inp.b_dn,
                             k=inp.wl.k, limit=inp.limit, alpha=inp.alpha, tokens=tokens,
                             keep_hidden=keep_hidden, workers=workers)
