"""Pins of the float64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a
worked example printed on the pages (tests/golden), a closed form, an
invariant, a library conversion routine, or the scalar-loop oracle.  The
mutant tests plant each named mistake in the oracle and show that the parity
harness flags it far above the tolerance.
"""

import math
import os

import numpy as np
import pytest
import torch

from decoder_qwen3_step_gb300 import inputs
from oracle import compare as cmp
from oracle import numerics as nm
from oracle.brute import BruteDecoder
from oracle.model import DecoderConfig, Oracle, attention_one, param_count, rms_norm, rope, silu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def cfg_of(name, **kw):
    return DecoderConfig(**inputs.SHAPES[name], **kw)


@pytest.fixture(scope="module")
def tiny():
    cfg = cfg_of("tiny", max_positions=64)
    w = inputs.make_weights(inputs.SHAPES["tiny"])
    ids = inputs.make_ids(cfg.vocab, 16)
    return cfg, w, ids


# -- golden values from the pages ------------------------------------------------

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_param_count_matches_published_qwen3_0p6b():
    expected = int(_golden_lines("param_count.txt")[0][0])
    assert param_count(cfg_of("qwen3_0p6b")) == expected


def test_f16_worked_examples():
    for expr, bits in _golden_lines("f16_ties.txt"):
        value = np.float32(eval(expr, {"__builtins__": {}}))  # exact in float32
        assert int(nm.f32_to_f16_bits(value)) == int(bits, 16), expr


# -- number formats against their definition and against library routines ----------

def test_f16_every_pattern_round_trips():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = nm.f16_bits_to_f32(bits)
    keep = ~np.isnan(vals)
    back = nm.f32_to_f16_bits(vals[keep])
    assert np.array_equal(back, bits[keep])
    assert np.isnan(nm.f16_bits_to_f32(nm.f32_to_f16_bits(np.float32(np.nan))))


def test_f16_matches_numpy_conversion_on_ties_subnormals_and_overflow():
    rng = np.random.default_rng(3)
    base = nm.f16_bits_to_f32(np.arange(0, 0x7C00, dtype=np.uint16)).astype(np.float64)
    nxt = nm.f16_bits_to_f32(np.arange(1, 0x7C01, dtype=np.uint16)).astype(np.float64)
    ties = ((base + nxt) / 2).astype(np.float32)  # exactly halfway (representable in f32)
    quarter = (base + (nxt - base) * 0.25).astype(np.float32)
    randoms = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 12, 200000))).astype(np.float32)
    vals = np.concatenate([ties, -ties, quarter, randoms, np.float32([65504, 65519, 65520, 1e6, -1e6, 0.0, -0.0,
                                                                      2.0 ** -25, 2.0 ** -24 * 1.5, np.inf, -np.inf])])
    ours = nm.f32_to_f16_bits(vals)
    lib = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, lib)


def test_f16_overflow_goes_to_infinity():
    assert int(nm.f32_to_f16_bits(np.float32(65520.0))) == 0x7C00
    assert int(nm.f32_to_f16_bits(np.float32(65519.0))) == 0x7BFF


def test_bf16_ties_and_library_agreement():
    one = np.float32(1.0)
    assert nm.bf16_round(np.float32(1 + 2 ** -8)) == one  # halfway, even mantissa kept
    assert nm.bf16_round(np.float32(1 + 3 * 2 ** -8)) == np.float32(1 + 2 ** -6)
    rng = np.random.default_rng(5)
    vals = (rng.standard_normal(300000) * np.exp(rng.uniform(-30, 30, 300000))).astype(np.float32)
    lib = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(nm.bf16_round(vals), lib)


# -- closed forms and invariants of the pieces ----------------------------------------

def test_rmsnorm_unit_gain_has_closed_form_rms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64)) * 0.01
    y = rms_norm(x, np.ones(64), 1e-6)
    ms = np.mean(x * x, axis=-1)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + 1e-6)), rtol=1e-13)


def test_silu_values():
    assert silu(np.float64(0.0)) == 0.0
    assert math.isclose(silu(np.float64(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    assert math.isclose(silu(np.float64(-2.0)), -2.0 / (1.0 + math.exp(2.0)), rel_tol=1e-15)


def test_rope_basis_vector_rotates_into_its_split_half_partner():
    D, base = 128, 1e6
    for j in (0, 1, 5, 63):
        x = np.zeros((1, D))
        x[0, j] = 1.0
        for pos in (0, 1, 37, 4159):
            y = rope(x, np.array([pos]), base)[0]
            phi = pos * base ** (-2.0 * j / D)
            expect = np.zeros(D)
            expect[j] = math.cos(phi)
            expect[j + D // 2] = math.sin(phi)
            assert np.allclose(y, expect, atol=1e-12), (j, pos)


def test_rope_preserves_norm_and_is_identity_at_zero():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3, 64))
    pos = np.array([0, 1, 2, 100, 1000, 4000, 40959])
    y = rope(x, pos, 1e6)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    assert np.array_equal(rope(x[:1], np.array([0]), 1e6), x[:1])


def test_rope_score_depends_only_on_relative_position():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    for split in (True, False):
        def score(m, n):
            return float(rope(q, np.array([m]), 1e6, split)[0] @ rope(k, np.array([n]), 1e6, split)[0])
        assert math.isclose(score(10, 3), score(1007, 1000), rel_tol=1e-9, abs_tol=1e-9)
        assert math.isclose(score(5, 5), score(300, 300), rel_tol=1e-9, abs_tol=1e-9)
        assert not math.isclose(score(10, 3), score(10, 4), rel_tol=1e-6)


def test_split_half_differs_from_neighbour_pairing():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 128))
    pos = np.array([1, 17, 99])
    assert np.abs(rope(x, pos, 1e6, True) - rope(x, pos, 1e6, False)).max() > 0.1


def test_attention_special_cases():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, 32))
    assert np.array_equal(attention_one(rng.standard_normal(32), rng.standard_normal((1, 32)), v), v[0])
    keys = np.tile(rng.standard_normal(32), (9, 1))  # equal keys: uniform weights
    vals = rng.standard_normal((9, 32))
    assert np.allclose(attention_one(rng.standard_normal(32), keys, vals), vals.mean(axis=0), atol=1e-14)


# -- the whole decoder ----------------------------------------------------------------

def test_brute_force_equals_vectorised_oracle_full_cached_and_decode(tiny):
    cfg, w, ids = tiny
    orc = Oracle(cfg, w)
    full = orc.full(ids)
    brute = np.array(BruteDecoder(cfg, w).step(list(ids), 0))
    assert np.abs(brute - full).max() < 1e-12

    b2 = BruteDecoder(cfg, w)
    cached = np.array(b2.step(list(ids[:8]), 0) + b2.step(list(ids[8:]), 8))
    assert np.abs(cached - orc.cached(ids)).max() < 1e-12

    cache = orc.new_cache(64)
    orc.forward(cache, ids, 0)
    fed, rows = orc.greedy(cache, int(np.argmax(full[-1])), 16, 8)
    b3 = BruteDecoder(cfg, w)
    b3.step(list(ids), 0)
    for i, tok in enumerate(fed):
        assert np.abs(np.array(b3.step([tok], 16 + i)[0]) - rows[i]).max() < 1e-12


def test_brute_force_equals_oracle_in_bf16_mode(tiny):
    cfg, w, ids = tiny
    orc = Oracle(cfg, w, mode="bf16")
    brute = np.array(BruteDecoder(cfg, w, round_fn=nm.bf16_round).step(list(ids[:6]), 0))
    assert np.abs(brute - orc.full(ids[:6])).max() < 1e-12
    assert np.abs(orc.full(ids[:6]) - Oracle(cfg, w).full(ids[:6])).max() > 1e-4  # rounding is applied


def test_cached_and_decode_equal_full_prompt(tiny):
    cfg, w, ids = tiny
    orc = Oracle(cfg, w)
    full = orc.full(ids)
    assert np.abs(orc.cached(ids) - full).max() < 1e-12
    cache = orc.new_cache(64)
    orc.forward(cache, ids[:5], 0)
    for i in range(5, 16):
        row = orc.forward(cache, ids[i:i + 1], i)[0]
        assert np.abs(row - full[i]).max() < 1e-12


def test_gqa_with_repeated_kv_heads_equals_mha(tiny):
    cfg, w, ids = tiny
    G = cfg.n_heads // cfg.n_kv_heads
    D = cfg.head_dim
    mha_cfg = DecoderConfig(**{**inputs.SHAPES["tiny"], "n_kv_heads": cfg.n_heads}, max_positions=64)
    w2 = dict(w)
    for l in range(cfg.n_layers):
        for t in ("k", "v"):
            m = w[f"layers.{l}.{t}"].reshape(cfg.n_kv_heads, D, -1)
            w2[f"layers.{l}.{t}"] = np.repeat(m, G, axis=0).reshape(cfg.n_heads * D, -1)
    a = Oracle(cfg, w).full(ids)
    b = Oracle(mha_cfg, w2).full(ids)
    assert np.abs(a - b).max() < 1e-12


def test_layer_dump_has_embedding_and_every_layer(tiny):
    cfg, w, ids = tiny
    dump = []
    Oracle(cfg, w).forward(Oracle(cfg, w).new_cache(64), ids, 0, dump=dump)
    assert len(dump) == cfg.n_layers + 1
    assert np.array_equal(dump[0], w["embed"][ids].astype(np.float64))


@pytest.mark.parametrize("mutant", ["s13", "s14", "s15", "s16", "s20", "s22", "neighbour"])
def test_parity_harness_detects_every_planted_mistake(tiny, mutant):
    """Each pitfall, planted in the oracle, moves the logits far past the fp32 gate."""
    cfg, w, ids = tiny
    orc = Oracle(cfg, w)
    good_full = orc.full(ids)
    if mutant in ("s13", "s14"):  # only visible once a step starts past position 0
        bad = orc.cached(ids, mutant=mutant)
    else:
        bad = orc.full(ids, mutant=mutant)
    res = cmp.compare(bad, good_full, cmp.TOL_FP32)
    assert not res["passed"]
    assert res["max_absolute_error"] > 10 * cmp.TOL_FP32


def test_refuses_out_of_vocab_ids(tiny):
    cfg, w, ids = tiny
    orc = Oracle(cfg, w)
    with pytest.raises(ValueError):
        orc.forward(orc.new_cache(64), [cfg.vocab], 0)


# -- the comparison rule --------------------------------------------------------------

def test_compare_counts_near_ties_and_exact_agreement():
    ref = np.array([[0.0, 1.0, 0.9995, -1.0], [2.0, 0.0, 0.0, 0.0]])
    dev = ref + 1e-4
    r = cmp.compare(dev, ref, 1e-3, device_ids=np.array([2, 0]))
    assert r["near_ties"] == 1 and r["argmax_exact"] == 1 and r["argmax_agree"] == 2 and r["passed"]
    r2 = cmp.compare(dev, ref, 1e-3, device_ids=np.array([1, 1]))
    assert r2["argmax_agree"] == 1 and not r2["passed"]
    r3 = cmp.compare(ref + 2e-3, ref, 1e-3)
    assert not r3["passed"]
    nan = ref.copy()
    nan[0, 3] = np.nan
    assert not cmp.compare(nan, ref, 1e-3)["passed"]


def test_argmax_ties_go_to_lowest_id():
    ref = np.array([[1.0, 3.0, 2.0, 3.0, -1.0]])  # the sampler example's logits
    assert int(np.argmax(ref[0])) == 1


def test_serving_context_lengths_are_distinct_and_span_the_range():
    lens = inputs.serving_context_lengths()
    assert len(set(lens)) == 32 and min(lens) == 1024 and max(lens) == 2048
    assert sum(lens) == 49152
