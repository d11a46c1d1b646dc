"""Shared pieces of the GPU parity tests: build a decoder and its oracle from
the same seeded weights, and run the pages' paths (full, cached, decode)."""

from __future__ import annotations

import json
import os

import numpy as np

from decoder_qwen3_step_gb300 import dec, inputs
from oracle.compare import TOL_BF16, TOL_FP32, compare
from oracle.model import DecoderConfig, Oracle

MODES = {"fp32": dec.DEC_FP32, "bf16": dec.DEC_BF16_F16KV, "int4": dec.DEC_INT4_F16KV}
TOLS = {"fp32": TOL_FP32, "bf16": TOL_BF16, "int4": TOL_BF16}


def make_pair(shape_name, mode, max_positions, max_tokens=4096, max_seqs=64, n_blocks=None, weights=None):
    import torch  # noqa: F401  (device memory for the decoder)
    from decoder_qwen3_step_gb300.runtime import Decoder

    shape = inputs.SHAPES[shape_name]
    w = weights if weights is not None else inputs.make_weights(shape)
    if n_blocks is None:
        n_blocks = max_seqs * ((max_positions + 15) // 16) + 8
    m = Decoder(shape, w, mode=MODES[mode], max_positions=max_positions, max_tokens=max_tokens, max_seqs=max_seqs,
                n_blocks=n_blocks)
    orc = Oracle(DecoderConfig(**shape, max_positions=max_positions), w, mode=mode)
    return m, orc, w


def check(dev_logits, dev_ids, ref_logits, mode, what="", case=None, path=None):
    """Compare device logits and ids with the oracle's under the mode's
    tolerance and the near-tie argmax rule.  With DEC_PARITY_ROWS set to a
    file path, the comparison is appended there as one JSON row per call that
    names its case and path (octlm "Proving it's the same model": one row per
    case and path, max and mean absolute error, argmax agreement as integer
    counts), extended with the mode, the near-tie count and the tolerance."""
    r = compare(dev_logits, ref_logits, TOLS[mode], dev_ids)
    out = os.environ.get("DEC_PARITY_ROWS")
    if out and case:
        row = {"case": case, "path": path or what, "mode": mode, **{k: (float(v) if isinstance(v, np.floating) else v)
                                                                    for k, v in r.items()}}
        with open(out, "a") as f:
            f.write(json.dumps(row, default=float) + "\n")
    assert r["passed"], f"{what}: {r}"
    assert r["argmax_agree"] == r["rows"], f"{what}: {r}"
    return r


def np_(t):
    return t.detach().cpu().numpy()
