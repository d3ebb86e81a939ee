"""Comparison rules between the CUDA path and the CPU oracle.

Tolerances (floating point), for the path that keeps activations in bf16
(W4A16): relative L2 error <= 5e-3 over the compared outputs and, per element,
|err| <= 3e-2 * max(1, |ref|).  Routing is integer work and is compared
bit-exactly, except at near-ties: a token whose k-th and (k+1)-th exact logits
differ by less than 1e-4 is flagged, and for it any selection that is a valid
top-k of the exact logits within that margin is accepted.

The routing weights are fp32 softmaxes of fp32 logits; their error against the
fp64 oracle is bounded by the logit error (a few 1e-6 for d = 2880), so they
are held to 2e-5 absolute.
"""
from __future__ import annotations

import numpy as np

REL_L2 = 5e-3
ELEM = 3e-2
GAP = 1e-4
W_ABS = 2e-5


def check_routing(ref, idx_gpu: np.ndarray, w_gpu: np.ndarray, k: int):
    """Compare top-k selections and weights.

    The selected SET is what is unique: it must equal the oracle's, except for
    a token whose k-th and (k+1)-th exact logits are within GAP (a flagged
    near-tie), where any valid top-k within that margin is accepted.  The slot
    ORDER is only unique up to near-equal logits, so it is checked for being
    non-increasing in the exact logits (within GAP).  Weights are compared per
    expert.  Returns the tokens whose selection legitimately differs.
    """
    idx_ref = ref["topk_idx"]
    logits = ref["logits"]
    T = idx_ref.shape[0]
    assert idx_gpu.shape == idx_ref.shape
    set_gpu = np.sort(idx_gpu, axis=1)
    set_ref = np.sort(idx_ref, axis=1)
    differ = np.nonzero(np.any(set_gpu != set_ref, axis=1))[0]
    excused = []
    for t in differ:
        assert ref["gap"][t] < GAP, (
            f"token {t}: gpu {idx_gpu[t].tolist()} vs oracle {idx_ref[t].tolist()}, "
            f"gap {ref['gap'][t]:.3g} is not a near-tie")
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < logits.shape[1]
        kth = np.sort(logits[t])[::-1][k - 1]
        assert np.all(logits[t, sel] >= kth - GAP), f"token {t}: invalid near-tie choice"
        excused.append(int(t))
    # slot order: non-increasing exact logits, up to near-ties
    lg = np.take_along_axis(logits, idx_gpu.astype(np.int64), axis=1)
    bad = np.nonzero(np.any(lg[:, 1:] > lg[:, :-1] + GAP, axis=1))[0]
    assert bad.size == 0, f"token {bad[0]}: slots not in descending logit order {idx_gpu[bad[0]]}"
    same = np.setdiff1d(np.arange(T), differ)
    if same.size:
        og = np.argsort(idx_gpu[same], axis=1)
        orf = np.argsort(idx_ref[same], axis=1)
        wg = np.take_along_axis(w_gpu[same], og, axis=1)
        wr = np.take_along_axis(ref["topk_w"][same], orf, axis=1)
        err = np.abs(wg - wr)
        assert err.max() <= W_ABS, f"routing weight error {err.max():.3g} > {W_ABS}"
    return excused


def check_output(out_gpu: np.ndarray, ref_out: np.ndarray, what: str = "out"):
    """The two floating-point criteria on matching rows; returns the metrics."""
    assert out_gpu.shape == ref_out.shape, (out_gpu.shape, ref_out.shape)
    assert np.all(np.isfinite(out_gpu)), f"{what}: non-finite values"
    err = out_gpu - ref_out
    rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(ref_out), 1e-300))
    elem = np.abs(err) / np.maximum(1.0, np.abs(ref_out))
    worst = np.unravel_index(np.argmax(elem), elem.shape)
    assert rel_l2 <= REL_L2, f"{what}: relative L2 error {rel_l2:.3g} > {REL_L2}"
    assert elem.max() <= ELEM, (
        f"{what}: element {worst} error {err[worst]:.4g} vs ref {ref_out[worst]:.4g} "
        f"exceeds {ELEM}*max(1,|ref|)")
    return rel_l2, float(elem.max())


def check_permutation(ref_perm_fn, idx_gpu: np.ndarray, E: int, off_gpu, perm_gpu, inv_gpu):
    """offsets / perm / inv must equal the oracle's permutation of the GPU's own
    selection (identical to the oracle's selection unless a near-tie differs)."""
    counts, offsets, perm, inv = ref_perm_fn(idx_gpu, E)
    assert np.array_equal(off_gpu, offsets), "offsets differ"
    assert np.array_equal(perm_gpu, perm), "perm differs"
    assert np.array_equal(inv_gpu, inv), "inv differs"
