"""The sampler and its random generator, written out from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain Python floats
(IEEE binary64) in plain loops: every sum runs left to right, in the order the
pages give, so a reader can check each step against them by eye.

Sources
-------
* tinyllm L10.1 "Candle model runner (Llama + bigram, int4), Rust KV cache,
  sampler and PCG32", section 2.6 "The sampler and PCG32": the order of the
  steps (widen to f64; repetition penalty over the distinct ids of prompt and
  output, dividing positive logits and multiplying the others; presence and
  frequency penalties over the output only; the logprob is the log-softmax at
  that point; greedy is the argmax with ties to the lowest id and takes no
  draw; otherwise divide by T, keep the top k by (logit desc, id asc), keep
  the nucleus up to and including the id that reaches p, keep ids whose
  probability is at least min_p times the largest, softmax over the kept ids
  in ascending id order, draw one uniform and walk the cumulative sum in
  ascending id order to the first id with u < c); the per-request stream
  child_seed(s, 4) = mix64(s + 4 * 0x9E3779B97F4A7C15) seeding PCG32 on
  sequence 4; the uniform made of two 32-bit outputs a, b:
  ((a >> 5) * 2^26 + (b >> 6)) * 2^-53.
* same page, section 3 "Worked example by hand", the sampled token.
* PCG32 is O'Neill's XSH RR 64/32 generator (M. E. O'Neill, "PCG: A Family of
  Simple Fast Space-Efficient Statistically Good Algorithms for Random Number
  Generation", 2014): a 64-bit LCG with multiplier 6364136223846793005 and an
  odd increment; each output is the xorshifted old state (bits 18 up, xored
  into itself, then shifted down 27) rotated right by its top five bits.
  Seeding with (initstate, initseq): state 0, increment 2 * initseq + 1, one
  step, add initstate, one step.
* mix64 is used on the pages but not defined there.  Reading: the 64-bit
  finaliser of SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014; it is named mix64
  in that work's Java generator): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
  z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31.  The worked example
  pins this reading: child_seed(0, 4) comes out as the printed
  0xF88BB8A8724C81EC and the first uniform as 0.80209.

Readings where the pages leave a step open
------------------------------------------
* top_k = 0, or top_k >= vocab, keeps every id (the field is a count; zero is
  the conventional "off").
* top_p >= 1 skips the nucleus; the walk runs in (logit desc, id asc) order
  over the probabilities of the ids top-k kept (the worked example
  renormalises over the top-k set before walking); if rounding keeps the sum
  below p to the end, every id stays.
* min_p = 0 skips the step; the probabilities compared are those of the
  nucleus step (softmax over the top-k set); "max q" is the largest of them.
* Presence and frequency touch only ids that occur in the output: such an id
  loses frequency * count + presence; an id absent from the output is left
  alone.  The repetition penalty touches each distinct id once.
* The softmax sums (the log-partition, the top-k set, the final kept set)
  run over ids in ascending order, as the worked example writes them.
* If rounding leaves the last cumulative sum at or below u, the last kept id
  is the token.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

MASK64 = (1 << 64) - 1
PURPOSE_SAMPLE = 4
GOLDEN_GAMMA = 0x9E3779B97F4A7C15  # the stream spacing of child_seed
PCG_MULT = 6364136223846793005


def mix64(z: int) -> int:
    """SplitMix64's finaliser (the reading of mix64; see the module docstring)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def child_seed(seed: int, purpose: int) -> int:
    """child_seed(s, purpose) = mix64(s + purpose * 0x9E3779B97F4A7C15) (mod 2^64)."""
    return mix64((seed + purpose * GOLDEN_GAMMA) & MASK64)


class Pcg32:
    """PCG32 (XSH RR 64/32).  Pcg32(initstate, initseq) is pcg32_srandom_r."""

    def __init__(self, initstate: int, initseq: int):
        self.state = 0
        self.inc = ((initseq << 1) | 1) & MASK64
        self.next_u32()
        self.state = (self.state + initstate) & MASK64
        self.next_u32()

    def next_u32(self) -> int:
        old = self.state
        self.state = (old * PCG_MULT + self.inc) & MASK64
        xorshifted = (((old >> 18) ^ old) >> 27) & 0xFFFFFFFF
        rot = old >> 59
        return ((xorshifted >> rot) | (xorshifted << ((32 - rot) & 31))) & 0xFFFFFFFF

    def uniform_f64(self) -> float:
        """u = ((a >> 5) * 2^26 + (b >> 6)) * 2^-53 from two consecutive outputs a, b."""
        a = self.next_u32()
        b = self.next_u32()
        return ((a >> 5) * 67108864 + (b >> 6)) * (1.0 / 9007199254740992.0)

    def snapshot(self):
        return (self.state, self.inc)


def stream(seed: int, purpose: int = PURPOSE_SAMPLE) -> Pcg32:
    """The generator of one request and purpose: PCG32 seeded with child_seed on sequence `purpose`."""
    return Pcg32(child_seed(seed, purpose), purpose)


@dataclass
class SamplingParams:
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    min_p: float = 0.0
    repetition_penalty: float = 1.0
    presence_penalty: float = 0.0
    frequency_penalty: float = 0.0


def penalized(logits, p: SamplingParams, prompt, output):
    """Widen to f64, then the repetition penalty over the distinct ids of prompt
    and output, then presence and frequency over the output only."""
    l = [float(x) for x in logits]
    r = float(p.repetition_penalty)
    for i in sorted(set(prompt) | set(output)):
        l[i] = l[i] / r if l[i] > 0 else l[i] * r
    counts = {}
    for i in output:
        counts[i] = counts.get(i, 0) + 1
    for i in sorted(counts):
        l[i] = l[i] - (float(p.frequency_penalty) * counts[i] + float(p.presence_penalty))
    return l


def log_partition(l):
    """(M, ln Z): M the largest logit, Z = sum_i exp(l_i - M) over ids in order."""
    M = max(l)
    Z = 0.0
    for x in l:
        Z += math.exp(x - M)
    return M, math.log(Z)


def sample_trace(logits, p: SamplingParams, prompt, output, rng: Pcg32) -> dict:
    """Every intermediate of one sampling step, in the pages' order.

    Returns a dict with the token, its logprob, the kept sets after each
    filter, and the cumulative sums each decision compared (the parity tests
    read the margins of those comparisons).
    """
    l = penalized(logits, p, prompt, output)
    V = len(l)
    M, lse = log_partition(l)

    def logprob(i):
        return (l[i] - M) - lse

    out = {"penalized": l, "M": M, "lse": lse}
    if p.temperature == 0:
        tok = min(i for i in range(V) if l[i] == M)  # ties to the lowest id; no draw
        out.update(token=tok, logprob=logprob(tok), drew=False)
        return out

    T = float(p.temperature)
    lt = [x / T for x in l]
    order = sorted(range(V), key=lambda i: (-lt[i], i))
    k = int(p.top_k)
    kept = order[:k] if 0 < k < V else order
    out["topk"] = list(kept)

    Mk = lt[kept[0]]
    Zk = 0.0
    for i in sorted(kept):
        Zk += math.exp(lt[i] - Mk)
    q = {i: math.exp(lt[i] - Mk) / Zk for i in kept}
    out["q"] = q

    nucleus_cums = []
    if p.top_p < 1:
        nucleus, cum = [], 0.0
        for i in kept:
            nucleus.append(i)
            cum += q[i]
            nucleus_cums.append(cum)
            if cum >= p.top_p:
                break
        kept = nucleus
    out["nucleus"] = list(kept)
    out["nucleus_cums"] = nucleus_cums

    if p.min_p > 0:
        bound = p.min_p * q[kept[0]]
        out["minp_bound"] = bound
        kept = [i for i in kept if q[i] >= bound]
    out["kept"] = list(kept)

    ids = sorted(kept)
    Mf = max(lt[i] for i in ids)
    Zf = 0.0
    for i in ids:
        Zf += math.exp(lt[i] - Mf)
    u = rng.uniform_f64()
    c, tok, cums = 0.0, ids[-1], []
    for i in ids:
        c += math.exp(lt[i] - Mf) / Zf
        cums.append(c)
        if u < c:
            tok = i
            break
    out.update(token=tok, logprob=logprob(tok), drew=True, u=u, ids=ids, cdf=cums, scaled=lt)
    return out


def sample(logits, p: SamplingParams, prompt, output, rng: Pcg32):
    """(token id, f64 logprob) of one sampling step; advances `rng` by one
    uniform unless the step is greedy."""
    t = sample_trace(logits, p, prompt, output, rng)
    return t["token"], t["logprob"]


def decision_margin(t: dict, p: SamplingParams) -> float:
    """The smallest distance between a compared quantity and its threshold in
    one sampling step: how far u sat from the cumulative sums around the
    token, the nucleus sum from p, and the probabilities at the min-p edge
    from their bound.  Inf for a greedy step.  A device that adds in another
    order can decide differently only where this is within its rounding."""
    if not t["drew"]:
        return math.inf
    m = math.inf
    cdf, u = t["cdf"], t["u"]
    for c in cdf[-2:]:
        m = min(m, abs(u - c))
    if p.top_p < 1:
        for c in t["nucleus_cums"][-2:]:
            m = min(m, abs(c - p.top_p))
    if p.min_p > 0:
        b = t["minp_bound"]
        for i in t["nucleus"]:
            m = min(m, abs(t["q"][i] - b))
    return m
