"""Planted mistakes in the oracle's number formats each fail a pin.

The f16 and bf16 conversions of oracle/numerics.py decide every cached key
and value and every serving-mode weight, so each plausible slip in them is
planted into a copy of the module's source (the pages' mutant s08 among
them: truncating instead of rounding to f16) and run through the pins: the
worked examples of tests/golden/f16_ties.txt and the library conversions
(numpy's float16, torch's bfloat16).
"""

import os
import sys
import types

import numpy as np
import pytest
import torch

from oracle import numerics as nm0

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "oracle", "numerics.py")
GOLDEN = os.path.join(ROOT, "tests", "golden", "f16_ties.txt")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")  # numpy warns when 1e6 overflows to f16 inf


def check_f16_golden(nm):
    with open(GOLDEN) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                expr, bits = ln.split()
                value = np.float32(eval(expr, {"__builtins__": {}}))
                assert int(nm.f32_to_f16_bits(value)) == int(bits, 16), expr


def check_f16_library(nm):
    base = nm0.f16_bits_to_f32(np.arange(0, 0x7C00, dtype=np.uint16)).astype(np.float64)
    nxt = nm0.f16_bits_to_f32(np.arange(1, 0x7C01, dtype=np.uint16)).astype(np.float64)
    ties = ((base + nxt) / 2).astype(np.float32)
    rng = np.random.default_rng(8)
    randoms = (rng.standard_normal(50000) * np.exp(rng.uniform(-20, 12, 50000))).astype(np.float32)
    vals = np.concatenate([ties, -ties, randoms, np.float32([65504, 65519, 65520, 1e6, 2.0 ** -25])])
    assert np.array_equal(nm.f32_to_f16_bits(vals), vals.astype(np.float16).view(np.uint16))


def check_bf16_library(nm):
    rng = np.random.default_rng(9)
    vals = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    vals = np.concatenate([vals, np.float32([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)])])
    lib = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(nm.bf16_round(vals), lib)


CHECKS = {"f16_golden": check_f16_golden, "f16_library": check_f16_library, "bf16_library": check_bf16_library}

MUTANTS = {
    # s08: truncating instead of rounding to f16
    "f16_truncate": ("    up = (rem > half) | ((rem == half) & ((kept & 1) == 1))\n",
                     "    up = rem < 0\n"),
    "f16_ties_away": ("    up = (rem > half) | ((rem == half) & ((kept & 1) == 1))\n",
                      "    up = rem >= half\n"),
    "f16_subnormal_ties_down": (
        "    up_s = (sh > 0) & ((rem_s > half_s) | ((rem_s == half_s) & ((k & 1) == 1)))\n",
        "    up_s = (sh > 0) & (rem_s > half_s)\n"),
    "f16_overflow_saturates": ("normal_bits = np.where(biased >= 31, 0x7C00, normal_bits)",
                               "normal_bits = np.where(biased >= 31, 0x7BFF, normal_bits)"),
    "bf16_truncate": ("rounded = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000))",
                      "rounded = (u & np.uint64(0xFFFF0000))"),
    "bf16_ties_away": ("rounded = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000))",
                       "rounded = ((u + np.uint64(0x8000)) & np.uint64(0xFFFF0000))"),
}


def planted(old, new):
    src = open(SOURCE).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle.numerics_mutant")
    mod.__package__ = "oracle"
    sys.modules["oracle.numerics_mutant"] = mod
    try:
        exec(compile(src.replace(old, new), SOURCE, "exec"), mod.__dict__)
    finally:
        del sys.modules["oracle.numerics_mutant"]
    return mod


@pytest.mark.parametrize("name", sorted(CHECKS))
def test_the_oracle_passes_every_check(name):
    CHECKS[name](nm0)


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_each_planted_mistake_fails_a_pin(mutant):
    mod = planted(*MUTANTS[mutant])
    failed = []
    for name, check in CHECKS.items():
        try:
            check(mod)
        except AssertionError:
            failed.append(name)
    assert failed, f"mutant {mutant} passed every pin"
