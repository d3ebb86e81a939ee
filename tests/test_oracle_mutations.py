"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is built from the oracle's source text with one edit applied and
executed as a throw-away module on the CPU; the real oracle is untouched.  A
mutant survives if every pin in tests/oracle_pins.py still passes on it.
"""
import os
import types

import pytest

from . import oracle_pins

ORACLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "oracle", "moe_oracle.py")

MUTANTS = {
    "nibble_order": [("out[..., 0::2] = p & 0x0F", "out[..., 0::2] = p >> 4"),
                     ("out[..., 1::2] = p >> 4", "out[..., 1::2] = p & 0x0F")],
    "scale_bias": [("np.ldexp(1.0, s - 127)", "np.ldexp(1.0, s - 126)")],
    "e2m1_table": [("(0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)",
                    "(0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0)")],
    "sign_dropped": [("return np.where(c & 8, -mag, mag)", "return mag")],
    "block_16": [("MX_BLOCK = 32", "MX_BLOCK = 16")],
    "router_bias_dropped": [("+ np.asarray(router_b, np.float64)", "+ 0.0")],
    "tie_high_index": [('order = np.argsort(-l, axis=1, kind="stable")',
                        'order = l.shape[1] - 1 - np.argsort(-l[:, ::-1], axis=1, kind="stable")')],
    "softmax_all_experts": [("w = selected_softmax(np.take_along_axis(logits, idx, axis=1))",
                             "w = np.take_along_axis(selected_softmax(logits), idx, axis=1)")],
    "no_plus_one": [("* (u + 1.0)", "* u")],
    "gate_clamped_below": [("g = np.minimum(z_gate, limit)", "g = np.clip(z_gate, -limit, limit)")],
    "alpha_dropped": [("sigmoid(alpha * g)", "sigmoid(g)")],
    "gate_up_swapped": [("clamped_swiglu(z[:, :W], z[:, W:]", "clamped_swiglu(z[:, W:], z[:, :W]")],
    "down_bias_dropped": [("y = h @ w_dn.T + b_dn", "y = h @ w_dn.T")],
    "up_bias_dropped": [("z = x_rows @ w_gu.T + b_gu", "z = x_rows @ w_gu.T")],
    "down_transposed": [("y = h @ w_dn.T + b_dn", "y = h @ w_dn + b_dn")],
    "perm_slot_major": [("np.lexsort((slot, token, expert))", "np.lexsort((token, slot, expert))")],
    "offsets_shifted": [("offsets[1:] = np.cumsum(counts)", "offsets[:-1] = np.cumsum(counts)")],
    "unweighted_sum": [("out[pos] += w[tok[pos], slot][:, None] * y", "out[pos] += y")],
    "wrong_slot_weight": [("w[tok[pos], slot][:, None]", "w[tok[pos], 0][:, None]")],
    "bf16_shift": [("np.uint32) << 16", "np.uint32) << 15")],
    "gap_index": [("gap = srt[:, k - 1] - srt[:, k]", "gap = srt[:, k - 2] - srt[:, k]")],
    "mx_bits": [("n_params * 4 / 8 + n_params / MX_BLOCK", "n_params * 4 / 8 + n_params / 16")],
    "glu_two_matrices": [("return 3 * d_model * hidden", "return 2 * d_model * hidden")],
    "sigmoid_sign": [("1.0 / (1.0 + np.exp(-v))", "1.0 / (1.0 + np.exp(v))")],
    "rms_mean_subtracted": [("return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)",
                             "return (x - x.mean(axis=-1, keepdims=True)) / np.sqrt(ms + eps)"
                             " * np.asarray(weight, np.float64)")],
    "rms_weight_dropped": [("return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)",
                            "return x / np.sqrt(ms + eps)")],
    "rms_eps_outside": [("np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)")],
    "rms_sum_not_mean": [("ms = np.mean(x * x, axis=-1, keepdims=True)",
                          "ms = np.sum(x * x, axis=-1, keepdims=True)")],
    "rms_bias_added": [("return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)",
                        "return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64) + 0.01")],
    "residual_dropped": [('res["out"] = x[res["tokens"]] + res["out"]', 'res["out"] = res["out"] + 0.0')],
    "residual_of_normed": [('res["out"] = x[res["tokens"]] + res["out"]',
                            'res["out"] = xn[res["tokens"]] + res["out"]')],
    "moe_reads_raw_x": [("res = moe_forward_f64(xn, router_w", "res = moe_forward_f64(x, router_w")],
    "moe_input_not_rounded": [("xn = round_bf16(rms_norm(x, norm_w, eps))",
                               "xn = rms_norm(x, norm_w, eps)")],
    "bf16_round_truncates": [("np.rint(np.ldexp(m, 8))", "np.trunc(np.ldexp(m, 8))")],
    "bf16_round_7_bits": [("np.rint(np.ldexp(m, 8)), e - 8)", "np.rint(np.ldexp(m, 7)), e - 7)")],
}


def _mutant(edits):
    with open(ORACLE, encoding="utf-8") as f:
        src = f.read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation anchor not unique or missing: {old!r}"
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = ORACLE
    exec(compile(src, "<oracle mutant>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _mutant(MUTANTS[name])
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception as exc:  # an assertion or a crash both count as caught
            caught.append((check.__name__, type(exc).__name__))
    assert caught, f"mutant {name} passed every pin"
