"""Pins of the sampler oracle against what the pages and the mathematics fix.

The checks compare the oracle with the worked example printed on the pages
(tests/golden/sampling_hand_example.txt), with closed forms worked by hand
(penalties, a crossing nucleus, the CDF walk order, the logprob's
independence of the temperature), with library routines (numpy's lexsort for
the top-k order, math.fsum for the prefix sums), and with a chi-square fit of
its draws.  The mutant tests plant each mistake the pages list for this step
(tinyllm L10.1 section 5, mutants s01-s07) into a copy of the oracle's source
and show that one of these checks fails.
"""

import math
import os
import sys
import types

import numpy as np
import pytest

from oracle import sampler as S0

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SOURCE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "sampler.py")


def golden():
    out = {}
    with open(os.path.join(GOLDEN, "sampling_hand_example.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, *v = ln.split()
                out[k] = v
    return out


class FixedU:
    """A generator stand-in that returns one chosen uniform."""

    def __init__(self, u):
        self.u = u
        self.draws = 0

    def uniform_f64(self):
        self.draws += 1
        return self.u


# -- the checks (each takes the sampler module, so a mutant can be run through it) --

def check_hand_example(S):
    g = golden()
    logits = [float(x) for x in g["logits"]]
    p = S.SamplingParams(temperature=float(g["temperature"][0]), top_k=int(g["top_k"][0]), top_p=float(g["top_p"][0]))
    seed = int(g["seed"][0])
    assert S.child_seed(seed, S.PURPOSE_SAMPLE) == int(g["child_seed"][0], 16)
    assert round(S.stream(seed).uniform_f64(), 5) == float(g["first_uniform"][0])
    t = S.sample_trace(logits, p, [], [], S.stream(seed))
    assert round(math.exp(t["lse"]), 5) == float(g["log_partition"][0])
    assert t["topk"] == [int(x) for x in g["topk_order"]]
    for item in g["q_topk"]:
        i, v = item.split(":")
        assert round(t["q"][int(i)], 5) == float(v)
    assert t["nucleus"] == [int(x) for x in g["nucleus"]]
    assert t["token"] == int(g["token"][0])
    assert round(t["logprob"], 5) == float(g["logprob"][0])


def check_penalties(S):
    # hand-worked: prompt {0, 1}, output [2, 2, 4]; r = 2, presence 0.5, frequency 0.25
    #   id 0 (prompt, +2):  2 / 2                      =  1.0
    #   id 1 (prompt, -2): -2 * 2                      = -4.0
    #   id 2 (output x2, +1): 1 / 2 - (0.25*2 + 0.5)   = -0.5
    #   id 3 (untouched)                               =  0.5
    #   id 4 (output x1, -3): -3 * 2 - (0.25*1 + 0.5)  = -6.75
    p = S.SamplingParams(temperature=0.0, repetition_penalty=2.0, presence_penalty=0.5, frequency_penalty=0.25)
    logits = [2.0, -2.0, 1.0, 0.5, -3.0]
    assert S.penalized(logits, p, [0, 1, 1], [2, 2, 4]) == [1.0, -4.0, -0.5, 0.5, -6.75]
    tok, lp = S.sample(logits, p, [0, 1, 1], [2, 2, 4], FixedU(0.5))
    assert tok == 0
    want = -math.log(1 + math.exp(-5.0) + math.exp(-1.5) + math.exp(-0.5) + math.exp(-7.75))
    assert abs(lp - want) < 1e-15


def check_crossing_token(S):
    # four equal logits: q = 1/4 each, exactly; the running sums 0.25, 0.5, 0.75 are exact
    p = S.SamplingParams(temperature=1.0, top_p=0.5)
    assert S.sample_trace([0.0] * 4, p, [], [], FixedU(0.1))["nucleus"] == [0, 1]
    p.top_p = 0.25
    assert S.sample_trace([0.0] * 4, p, [], [], FixedU(0.1))["nucleus"] == [0]
    p.top_p = 0.75
    assert S.sample_trace([0.0] * 4, p, [], [], FixedU(0.1))["nucleus"] == [0, 1, 2]


def check_walk_order(S):
    # logits [0, 1, 0.5]: probabilities 1, e, e^0.5 over Z = 1 + e + e^0.5 = 5.36700...
    #   ascending ids: cumulative 0.18632, 0.69281, 1   -> u = 0.6 lands on id 1
    #   by probability (1, 2, 0): 0.50650, 0.81368, 1   -> would land on id 2
    tok, _ = S.sample([0.0, 1.0, 0.5], S.SamplingParams(temperature=1.0), [], [], FixedU(0.6))
    assert tok == 1
    tok, _ = S.sample([0.0, 1.0, 0.5], S.SamplingParams(temperature=1.0), [], [], FixedU(0.1))
    assert tok == 0
    tok, _ = S.sample([0.0, 1.0, 0.5], S.SamplingParams(temperature=1.0), [], [], FixedU(0.95))
    assert tok == 2


def check_logprob_before_temperature(S):
    # top_k = 1 keeps id 1 whatever T is; its logprob is -ln(e^-1 + 1 + e^-0.5) at every T
    want = -math.log(math.exp(-1.0) + 1.0 + math.exp(-0.5))
    for T in (0.25, 0.5, 1.0, 2.0, 7.0):
        tok, lp = S.sample([0.0, 1.0, 0.5], S.SamplingParams(temperature=T, top_k=1), [], [], FixedU(0.3))
        assert tok == 1
        assert abs(lp - want) < 1e-15, T


def check_generator_shape(S):
    r = S.stream(7)
    for _ in range(1000):
        u = r.uniform_f64()
        assert 0.0 <= u < 1.0
        assert float(u * 2.0**53).is_integer()  # on the 2^-53 grid
    # the uniform is built from two consecutive outputs: a's top 27 bits over b's top 26
    a, b = S.stream(11), S.stream(11)
    x, y = a.next_u32(), a.next_u32()
    assert b.uniform_f64() == ((x >> 5) * 2**26 + (y >> 6)) / 2**53


CHECKS = {
    "hand": check_hand_example,
    "penalties": check_penalties,
    "crossing": check_crossing_token,
    "walk": check_walk_order,
    "temperature": check_logprob_before_temperature,
    "generator": check_generator_shape,
}


@pytest.mark.parametrize("name", sorted(CHECKS))
def test_oracle_passes(name):
    CHECKS[name](S0)


# -- properties --------------------------------------------------------------------

def test_greedy_takes_no_draw_and_sampling_takes_one():
    logits = [0.5, 2.0, 2.0, -1.0]
    r = S0.stream(3)
    before = r.snapshot()
    tok, lp = S0.sample(logits, S0.SamplingParams(temperature=0.0), [], [], r)
    assert tok == 1 and r.snapshot() == before  # ties to the lowest id; untouched generator
    ref = S0.stream(3)
    ref.next_u32()
    ref.next_u32()
    S0.sample(logits, S0.SamplingParams(temperature=0.8, top_p=0.9), [], [], r)
    assert r.snapshot() == ref.snapshot()  # exactly one uniform: two outputs


def test_seeded_sampling_matches_the_distribution():
    probs = [0.4, 0.3, 0.2, 0.1]
    logits = [float(np.float32(math.log(x))) for x in probs]
    p = S0.SamplingParams(temperature=1.0)

    def draws(seed, n):
        r = S0.stream(seed)
        return [S0.sample(logits, p, [], [], r)[0] for _ in range(n)]

    d = draws(2024, 4000)
    counts = np.bincount(d, minlength=4)
    chi2 = sum((counts[i] - 4000 * probs[i]) ** 2 / (4000 * probs[i]) for i in range(4))
    assert chi2 < 16.27, (counts, chi2)  # 3 degrees of freedom, p = 0.001
    assert draws(2024, 200) == d[:200]  # a seed repeats
    assert draws(2025, 200) != d[:200]


def random_case(rng, V):
    logits = np.float32(rng.normal(0, 2, V))
    logits[rng.integers(0, V, 3)] = logits[0]  # equal logits: the id order decides
    p = S0.SamplingParams(
        temperature=float(rng.choice([0.3, 0.7, 1.0, 1.6])),
        top_k=int(rng.choice([0, 1, 3, V - 1, V + 2])),
        top_p=float(rng.choice([1.0, 0.9, 0.5, 0.2])),
        min_p=float(rng.choice([0.0, 0.05, 0.3])),
        repetition_penalty=float(rng.choice([1.0, 1.3])),
        presence_penalty=float(rng.choice([0.0, 0.4])),
        frequency_penalty=float(rng.choice([0.0, 0.2])),
    )
    prompt = list(rng.integers(0, V, 4))
    output = list(rng.integers(0, V, 3))
    return [float(x) for x in logits], p, prompt, output


def test_filters_against_library_order_and_exact_sums():
    """Each kept set is what its rule asks, checked with other tools: numpy's
    lexsort for the (logit desc, id asc) order, math.fsum (an exactly rounded
    sum) for the nucleus and CDF decisions, away from rounding-level ties."""
    rng = np.random.default_rng(5)
    for case in range(300):
        V = int(rng.integers(2, 13))
        logits, p, prompt, output = random_case(rng, V)
        t = S0.sample_trace(logits, p, prompt, output, S0.stream(case))
        lt = np.array(t["scaled"])
        order = list(np.lexsort((np.arange(V), -lt)))
        k = p.top_k if 0 < p.top_k < V else V
        assert t["topk"] == order[:k]
        q = t["q"]
        nuc = t["nucleus"]
        assert nuc == order[: len(nuc)]
        if p.top_p < 1:
            before = math.fsum(q[i] for i in nuc[:-1])
            upto = math.fsum(q[i] for i in nuc)
            if min(abs(before - p.top_p), abs(upto - p.top_p)) > 1e-12:
                assert before < p.top_p
                assert upto >= p.top_p or len(nuc) == k
        else:
            assert len(nuc) == k
        bound = p.min_p * q[nuc[0]]
        assert t["kept"] == [i for i in nuc if q[i] >= bound]
        ids = sorted(t["kept"])
        w = [math.exp(lt[i] - lt[ids[0]]) for i in ids]
        w = [x / math.fsum(w) for x in w]
        cum = [math.fsum(w[: j + 1]) for j in range(len(ids))]
        if min(abs(c - t["u"]) for c in cum) > 1e-12:
            first = next((ids[j] for j in range(len(ids)) if t["u"] < cum[j]), ids[-1])
            assert t["token"] == first
        lse = math.log(math.fsum(math.exp(x - max(t["penalized"])) for x in t["penalized"]))
        assert abs(t["logprob"] - (t["penalized"][t["token"]] - max(t["penalized"]) - lse)) < 1e-13


# -- planted mistakes ------------------------------------------------------------------

MUTANTS = {
    # s01 swapped shifts of the two draws
    "s01": ("((a >> 5) * 67108864 + (b >> 6))", "((a >> 6) * 67108864 + (b >> 5))", "hand"),
    # s02 the sample stream seeded on sequence 54 instead of its purpose
    "s02": ("return Pcg32(child_seed(seed, purpose), purpose)", "return Pcg32(child_seed(seed, purpose), 54)", "hand"),
    # s03 the logprob taken after the temperature
    "s03": ("out.update(token=tok, logprob=logprob(tok), drew=True",
            "out.update(token=tok, logprob=(lt[tok] - max(lt)) - math.log(sum(math.exp(x - max(lt)) for x in lt)), drew=True",
            "temperature"),
    # s04 > instead of >= in the nucleus walk
    "s04": ("if cum >= p.top_p:", "if cum > p.top_p:", "crossing"),
    # s05 the CDF walked in probability order
    "s05": ("ids = sorted(kept)", "ids = sorted(kept, key=lambda i: (-lt[i], i))", "walk"),
    # s06 presence and frequency over the prompt too
    "s06": ("for i in output:\n        counts[i]", "for i in list(prompt) + list(output):\n        counts[i]", "penalties"),
    # s07 negative logits divided by the repetition penalty
    "s07": ("l[i] / r if l[i] > 0 else l[i] * r", "l[i] / r", "penalties"),
}


def planted(old, new):
    src = open(SOURCE).read()
    assert src.count(old) == 1, old  # the mistake is really planted
    mod = types.ModuleType("sampler_mutant")
    sys.modules["sampler_mutant"] = mod  # dataclasses look their module up by name
    try:
        exec(compile(src.replace(old, new), SOURCE, "exec"), mod.__dict__)
    finally:
        del sys.modules["sampler_mutant"]
    return mod


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_each_planted_mistake_fails_a_pin(mutant):
    old, new, check = MUTANTS[mutant]
    with pytest.raises(AssertionError):
        CHECKS[check](planted(old, new))
