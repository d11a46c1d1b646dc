"""Pins of the int4 oracle against what the pages and the mathematics fix.

The hand example (tests/golden/int4_hand_example.txt), the error bound
|W - q s| <= s/2, rounding half to even, numpy's own f32 -> f16 conversion for
the scales, a byte-by-byte loop for the packing, and the effective weights in
the oracle's int4 mode.  The mutant tests plant a mistake each (swapped
nibbles, the unrounded scale, ties away from zero) into a copy of the oracle's
source and show that a pin fails.
"""

import os
import sys
import types

import numpy as np
import pytest

from oracle import int4 as Q0
from oracle.numerics import f16_bits_to_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SOURCE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "int4.py")


def golden():
    out = {}
    with open(os.path.join(GOLDEN, "int4_hand_example.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, *v = ln.split()
                out[k] = v
    return out


def check_hand_example(Q):
    g = golden()
    W = np.array([[float(x) for x in g["weights"]]], dtype=np.float32)
    group = int(g["group"][0])
    q, s = Q.quantize(W, group)
    assert float(f16_bits_to_f32(s)[0, 0]) == float(g["scale"][0])
    assert q[0].tolist() == [int(x) for x in g["codes"]]
    codes = np.array([[int(x) for x in g["pack_codes"]]], dtype=np.int8)
    assert Q.pack(codes)[0].tolist() == [int(x, 16) for x in g["pack_bytes"]]
    assert Q.unpack(Q.pack(codes)).tolist() == codes.tolist()


def check_exact_scale_matters(Q):
    # the last weight over the stored scale is 1.5001 -> 2; over 0.2 it would be 1.49975 -> 1
    g = golden()
    W = np.array([[float(x) for x in g["weights"]]], dtype=np.float32)
    q, _ = Q.quantize(W, int(g["group"][0]))
    assert q[0, 3] == 2 and int(g["code_with_exact_scale"][0]) == 1


def check_ties_to_even(Q):
    # max |W| = 7 gives the scale f16(1) = 1 exactly, so W / s = W
    W = np.zeros((1, 32), dtype=np.float32)
    W[0, :6] = [7.0, 2.5, 3.5, -0.5, -2.5, 0.5]
    q, s = Q.quantize(W, 32)
    assert float(f16_bits_to_f32(s)[0, 0]) == 1.0
    assert q[0, :6].tolist() == [7, 2, 4, 0, -2, 0]


CHECKS = {"hand": check_hand_example, "exact_scale": check_exact_scale_matters, "ties": check_ties_to_even}


@pytest.mark.parametrize("name", sorted(CHECKS))
def test_oracle_passes(name):
    CHECKS[name](Q0)


def test_error_bound_and_scales_against_numpy_f16():
    g = np.random.default_rng(0)
    W = (g.standard_normal((64, 256)) * g.uniform(0.01, 3.0, (64, 1))).astype(np.float32)
    W[3, 32:64] = 0.0  # an all-zero group
    q, s_bits = Q0.quantize(W)
    s = f16_bits_to_f32(s_bits).astype(np.float64)
    amax = np.abs(W.reshape(64, 8, 32)).max(axis=2)
    assert np.array_equal(s.astype(np.float32), (amax / np.float32(7)).astype(np.float16).astype(np.float32))
    What = Q0.dequantize(q, s_bits)
    err = np.abs(W.astype(np.float64) - What).reshape(64, 8, 32)
    assert np.all(err <= s[:, :, None] / 2 * (1 + 1e-12))
    assert np.all(q[3, 32:64] == 0) and s[3, 1] == 0.0
    assert q.min() >= -8 and q.max() <= 7


def test_packing_against_a_byte_loop():
    g = np.random.default_rng(1)
    q = g.integers(-8, 8, (5, 64)).astype(np.int8)
    b = Q0.pack(q)
    for r in range(5):
        for j in range(32):
            want = (int(q[r, 2 * j]) & 0xF) | ((int(q[r, 2 * j + 1]) & 0xF) << 4)
            assert b[r, j] == want
    assert np.array_equal(Q0.unpack(b), q)


def test_oracle_int4_mode_uses_the_effective_weights():
    from decoder_qwen3_step_gb300 import inputs
    from oracle.model import DecoderConfig, Oracle
    from oracle.numerics import bf16_round

    shape = inputs.SHAPES["tiny"]
    w = inputs.make_weights(shape)
    orc = Oracle(DecoderConfig(**shape, max_positions=32), w, mode="int4")
    assert np.array_equal(orc.layers[0]["q"], Q0.effective(w["layers.0.q"]))
    assert np.array_equal(orc.layers[1]["down"], Q0.effective(w["layers.1.down"]))
    assert np.array_equal(orc.embed, bf16_round(w["embed"]).astype(np.float64))


MUTANTS = {
    "nibbles": ("return (lo | (hi << 4)).astype(np.uint8)", "return (hi | (lo << 4)).astype(np.uint8)", "hand"),
    "unrounded_scale": ("    s = f16_bits_to_f32(s_bits).astype(np.float32)         # the stored value\n",
                        "    s = (amax / np.float32(7.0)).astype(np.float32)\n", "exact_scale"),
    "ties_away": ("q = np.clip(np.rint(r), -8, 7)", "q = np.clip(np.trunc(r + np.copysign(0.5, r)), -8, 7)", "ties"),
}


def planted(old, new):
    src = open(SOURCE).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle.int4_mutant")
    mod.__package__ = "oracle"
    sys.modules["oracle.int4_mutant"] = mod
    try:
        exec(compile(src.replace(old, new), SOURCE, "exec"), mod.__dict__)
    finally:
        del sys.modules["oracle.int4_mutant"]
    return mod


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_each_planted_mistake_fails_a_pin(mutant):
    old, new, check = MUTANTS[mutant]
    with pytest.raises(AssertionError):
        CHECKS[check](planted(old, new))
