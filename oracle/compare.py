"""Parity metrics between device logits and oracle logits.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: octlm "Proving it's the same model", sections "Every logit, every
position" (maximum absolute error as the gate, mean absolute error, argmax
agreement), "Pick the tolerance before looking" (the limit is fixed before
the first run) and "Both devices pass" (agreement must be counted in
integers: a float32 mean printed 0.99999994 for 188/188).  The near-tie
rule is this build's reading of the "near-tie rule" that tinyllm L10.1
section 4 names without defining: where the oracle's top-1/top-2 gap is at
most 2*tol, a device id whose oracle logit is within 2*tol of the oracle's
maximum counts as agreeing (it is a correct answer at that precision).
"""

from __future__ import annotations

import numpy as np

# Tolerances fixed before the first device run (max absolute logit error).
TOL_FP32 = 1e-3
TOL_BF16 = 5e-2


def compare(device_logits, oracle_logits, tol: float, device_ids=None) -> dict:
    """Compare [R, V] logits; returns integer counts and the error figures."""
    dev = np.asarray(device_logits, dtype=np.float64)
    ref = np.asarray(oracle_logits, dtype=np.float64)
    if dev.shape != ref.shape:
        raise ValueError(f"shape mismatch {dev.shape} vs {ref.shape}")
    finite = bool(np.isfinite(dev).all())
    delta = np.abs(dev - ref)
    rows = ref.shape[0]
    ref_id = np.argmax(ref, axis=-1)
    if device_ids is None:
        device_ids = np.argmax(dev, axis=-1)
    device_ids = np.asarray(device_ids, dtype=np.int64)
    top2 = np.sort(ref, axis=-1)[:, -2:] if ref.shape[1] > 1 else np.concatenate([ref, ref], axis=-1)
    gap = top2[:, 1] - top2[:, 0]
    near = gap <= 2 * tol
    exact = device_ids == ref_id
    ref_max = ref[np.arange(rows), ref_id]
    ok_near = ref[np.arange(rows), device_ids] >= ref_max - 2 * tol
    agree = np.where(near, ok_near, exact)
    return {
        "rows": int(rows),
        "finite": finite,
        "max_absolute_error": float(delta.max()) if delta.size else 0.0,
        "mean_absolute_error": float(delta.mean()) if delta.size else 0.0,
        "argmax_exact": int(exact.sum()),
        "argmax_agree": int(agree.sum()),
        "near_ties": int(near.sum()),
        "tolerance": tol,
        "passed": bool(finite and (delta.max() <= tol if delta.size else True) and agree.all()),
    }
