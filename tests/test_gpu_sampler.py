"""The device sampler (dec_sample) against the f64 oracle, sequence by sequence.

Each case runs the C-ABI sampler on seeded logits and histories and the
oracle on the same float32 logits, the same prompt/output ids and the same
PCG32 stream; it compares the token (exactly), the f64 logprob (within
1e-10: both are ln of a sum of at most 151,936 positive terms, rounded in two
different orders, about 2 * 151,936 * 2^-53 = 3.4e-11 relative, plus a
last-place difference in exp), and the generator state afterwards (exactly:
no draw when greedy, one uniform otherwise).  Where a decision of the oracle
sat within 1e-8 of its threshold (u against a cumulative sum, a nucleus sum
against p, a probability against the min-p bound) the device may decide the
other way; such cases only have to return a kept id, and must stay rare.
"""

import ctypes as C
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402
from decoder_qwen3_step_gb300.runtime import Sampler, sampling_params  # noqa: E402
from oracle import sampler as S  # noqa: E402

pytestmark = pytest.mark.gpu

NEAR = 1e-8
LP_TOL = 1e-10


def oracle_params(p):
    return S.SamplingParams(temperature=p.temperature, top_k=p.top_k, top_p=p.top_p, min_p=p.min_p,
                            repetition_penalty=p.repetition_penalty, presence_penalty=p.presence_penalty,
                            frequency_penalty=p.frequency_penalty)


def run_and_compare(sampler, logits, params, histories, seeds, label, exact=False):
    """Sample on the device and with the oracle; returns the number of near
    ties (exact=True: every sum is exact here, so no tie is excused)."""
    n = logits.shape[0]
    x = torch.from_numpy(logits).cuda()
    rng = sampler.streams(seeds)
    tok, lp = sampler.sample(x, params, histories, rng)
    torch.cuda.synchronize()
    tok, lp = tok.cpu().numpy(), lp.cpu().numpy()
    rng_after = rng.cpu().numpy().view(np.uint64)
    near = 0
    for i in range(n):
        pr, ou = histories[i] if histories else ([], [])
        op = oracle_params(params[i])
        r = S.stream(seeds[i])
        t = S.sample_trace([float(v) for v in logits[i]], op, list(pr), list(ou), r)
        where = f"{label} seq {i} params {params[i].temperature, params[i].top_k, params[i].top_p, params[i].min_p}"
        assert (int(rng_after[i][0]), int(rng_after[i][1])) == r.snapshot(), where + ": generator state"
        if not exact and S.decision_margin(t, op) < NEAR:
            near += 1
            assert int(tok[i]) in t.get("kept", [t["token"]]), where
            continue
        assert int(tok[i]) == t["token"], where + f": device {tok[i]} oracle {t['token']}"
        assert abs(lp[i] - t["logprob"]) <= LP_TOL, where + f": logprob {lp[i]} vs {t['logprob']}"
    assert sampler.status() == 0
    return near


def test_double_f32_exponential_against_f64():
    """The sampler's exponential (double-f32, table-driven) against the f64
    one: relative error at most 2^-44 down to e^-60 (the double-f32 tail is a
    normal float there), 2^-30 down to e^-80, 0 below e^-87."""
    g = np.random.default_rng(1)
    # arguments that are exact as a float head plus a float tail, as the sampler's l - M is
    hi = np.concatenate([-g.exponential(3.0, 200000), -g.uniform(0, 87, 200000), -g.uniform(0, 1e-3, 20000)])
    hi = hi.astype(np.float32)
    lo = (g.uniform(-0.5, 0.5, hi.size) * np.spacing(np.abs(hi))).astype(np.float32)
    x = np.concatenate([hi.astype(np.float64) + lo.astype(np.float64),
                        np.array([0.0, -0.0, -1e-30, -1e-8, -1.0, -60.0, -86.9, -87.5, -700.0, -np.inf])])
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    dec.check(dec.lib().dec_debug_df_exp(C.c_void_p(xd.data_ptr()), C.c_void_p(yd.data_ptr()), len(x), None),
              "dec_debug_df_exp")
    torch.cuda.synchronize()
    y = yd.cpu().numpy()
    ref = np.exp(x)
    rel = np.abs(y - ref) / np.maximum(ref, 1e-300)
    assert np.all(y[x == 0.0] == 1.0)  # exp(0) is exactly one: the top id's weight
    assert rel[x >= -60].max() <= 2.0**-44, rel[x >= -60].max()
    assert rel[(x < -60) & (x >= -80)].max() <= 2.0**-30
    assert np.all(y[x < -87] == 0.0)


def test_worked_example_on_the_device():
    s = Sampler(5, 1)
    x = np.array([[1, 3, 2, 3, -1]], dtype=np.float32)
    p = [sampling_params(temperature=1.0, top_k=3, top_p=0.8)]
    rng = s.streams([0])
    tok, lp = s.sample(torch.from_numpy(x).cuda(), p, None, rng)
    assert int(tok.item()) == 3
    assert round(float(lp.item()), 5) == -0.92487
    run_and_compare(s, x, p, None, [0], "worked example")
    s.close()


def param_grid(rng, V):
    grid = []
    for T in (0.0, 0.6, 1.0, 1.7):
        for k in (0, 1, 7, 50, 1000, V - 1, 5000):
            for p_ in (1.0, 0.9, 0.5):
                for m in (0.0, 0.05):
                    grid.append(sampling_params(temperature=T, top_k=k if k < V else 0, top_p=p_, min_p=m,
                                                repetition_penalty=float(rng.choice([1.0, 1.2])),
                                                presence_penalty=float(rng.choice([0.0, 0.3])),
                                                frequency_penalty=float(rng.choice([0.0, 0.1]))))
    return grid


def random_logits(rng, n, V, scale=3.0):
    x = rng.normal(0.0, scale, (n, V)).astype(np.float32)
    for i in range(n):  # a few dominant ids, and a run of equal logits
        x[i, rng.integers(0, V, 5)] += np.float32(rng.uniform(5, 12))
        j = int(rng.integers(0, V - 8))
        x[i, j:j + 8] = x[i, j]
    return x


@pytest.mark.parametrize("V", [1000, 6000])
def test_parameter_grid_matches_the_oracle(V):
    """Greedy, temperature, top-k (1 to beyond the shared-memory list),
    top-p and min-p, alone and together, with penalised histories."""
    rng = np.random.default_rng(V)
    grid = param_grid(rng, V)
    s = Sampler(V, 32)
    near = 0
    for c in range(0, len(grid), 32):
        ps = grid[c:c + 32]
        x = random_logits(rng, len(ps), V)
        hist = [(list(rng.integers(0, V, 20)), list(rng.integers(0, V, 12))) for _ in ps]
        near += run_and_compare(s, x, ps, hist, list(range(c, c + len(ps))), f"V={V} batch {c // 32}")
    assert near <= 2
    s.close()


@pytest.mark.parametrize("V", [7, 1025, 2049])
def test_ragged_vocabularies(V):
    """Vocabularies one past the scan kernels' chunk sizes (1,024 and 2,048
    ids) and below the 8-id padding: the chunk and padding tails."""
    rng = np.random.default_rng(50 + V)
    grid = param_grid(rng, V)
    ps = [grid[i] for i in rng.choice(len(grid), 32, replace=False)]
    x = random_logits(rng, len(ps), V) if V > 8 else rng.normal(0, 2, (len(ps), V)).astype(np.float32)
    hist = [(list(rng.integers(0, V, 6)), list(rng.integers(0, V, 4))) for _ in ps]
    s = Sampler(V, 32)
    assert run_and_compare(s, x, ps, hist, [700 + i for i in range(len(ps))], f"V={V}") <= 1
    s.close()


def test_full_qwen3_vocabulary():
    """151,936 ids: the bucket histogram, candidate gathering and the
    multi-chunk final walk at the model's own vocabulary."""
    V = inputs.SHAPES["qwen3_0p6b"]["vocab"]
    rng = np.random.default_rng(7)
    ps = [
        sampling_params(temperature=0.0, repetition_penalty=1.3, presence_penalty=0.5),
        sampling_params(temperature=0.7, top_k=40, top_p=0.9),
        sampling_params(temperature=1.0, top_p=0.95),          # nucleus without top-k
        sampling_params(temperature=0.8),                        # every id kept
        sampling_params(temperature=1.2, min_p=0.02),            # min-p alone
        sampling_params(temperature=1.0, top_k=20000, top_p=0.99),  # top-k beyond the list
        sampling_params(temperature=2.5, top_p=0.999),           # a nucleus of many thousand ids
        sampling_params(temperature=0.3, top_k=1),
    ]
    x = random_logits(rng, len(ps), V, scale=2.5)
    hist = [(list(rng.integers(0, V, 64)), list(rng.integers(0, V, 32))) for _ in ps]
    s = Sampler(V, 8)
    assert run_and_compare(s, x, ps, hist, [101 + i for i in range(len(ps))], "V=151936") == 0
    s.close()


def test_equal_logits_are_ordered_by_id():
    """All logits equal: every cut falls inside one run of ties, which the
    order breaks by id; the probabilities are exact dyadic numbers here, so
    the device must match the oracle exactly."""
    V = 8192
    x = np.zeros((4, V), dtype=np.float32)
    ps = [sampling_params(temperature=1.0, top_p=0.5), sampling_params(temperature=1.0, top_k=100),
          sampling_params(temperature=1.0, top_k=5000, top_p=0.25), sampling_params(temperature=0.0)]
    s = Sampler(V, 4)
    run_and_compare(s, x, ps, None, [3, 4, 5, 6], "equal logits", exact=True)
    s.close()


def test_top_p_keeps_the_crossing_token_on_the_device():
    x = np.zeros((3, 4), dtype=np.float32)
    ps = [sampling_params(temperature=1.0, top_p=v) for v in (0.25, 0.5, 0.75)]
    s = Sampler(4, 3)
    rng = s.streams([0, 0, 0])
    # u of stream 0 is 0.80209: with the nucleus {0}, {0,1}, {0,1,2} the token is 0, 1, 2
    tok, _ = s.sample(torch.from_numpy(x).cuda(), ps, None, rng)
    assert tok.cpu().tolist() == [0, 1, 2]
    s.close()


def test_greedy_takes_no_draw_and_penalties_apply():
    V = 64
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (2, V)).astype(np.float32)
    x[:, 10] = 9.0  # the argmax, then penalised away by the repetition penalty
    ps = [sampling_params(temperature=0.0, repetition_penalty=8.0), sampling_params(temperature=0.0)]
    s = Sampler(V, 2)
    gen = s.streams([5, 6])
    before = gen.clone()
    tok, _ = s.sample(torch.from_numpy(x).cuda(), ps, [([10], []), ([10], [])], gen)
    assert torch.equal(gen, before)
    assert tok.cpu().tolist()[1] == 10
    run_and_compare(s, x, ps, [([10], []), ([10], [])], [5, 6], "greedy")
    s.close()


def test_seeded_draws_follow_the_distribution():
    probs = [0.4, 0.3, 0.2, 0.1]
    x = np.tile(np.array([[math.log(p) for p in probs]], dtype=np.float32), (1000, 1))
    ps = [sampling_params(temperature=1.0)] * 1000
    s = Sampler(4, 1000)
    gen = s.streams(list(range(1000)))
    toks = []
    for _ in range(4):
        t, _ = s.sample(torch.from_numpy(x).cuda(), ps, None, gen)
        toks.append(t.cpu().numpy())
    toks = np.stack(toks)  # [draw, stream]
    for i in (0, 1, 517, 999):  # the device streams are the oracle's
        r = S.stream(i)
        want = [S.sample([float(v) for v in x[0]], S.SamplingParams(temperature=1.0), [], [], r)[0] for _ in range(4)]
        assert toks[:, i].tolist() == want
    counts = np.bincount(toks.reshape(-1), minlength=4)
    chi2 = sum((counts[i] - 4000 * probs[i]) ** 2 / (4000 * probs[i]) for i in range(4))
    assert chi2 < 16.27, counts
    s.close()


def test_batch_invariance():
    V = 5000
    rng = np.random.default_rng(11)
    x = random_logits(rng, 6, V)
    ps = [sampling_params(temperature=0.9, top_k=k, top_p=p_) for k, p_ in
          [(0, 0.9), (40, 1.0), (0, 1.0), (4500, 0.95), (10, 0.5), (0, 0.2)]]
    hist = [(list(rng.integers(0, V, 8)), list(rng.integers(0, V, 8))) for _ in ps]
    s = Sampler(V, 6)
    gen = s.streams(range(6))
    tb, lb = s.sample(torch.from_numpy(x).cuda(), ps, hist, gen)
    for i in range(6):
        g1 = s.streams([i])
        t1, l1 = s.sample(torch.from_numpy(x[i:i + 1]).cuda(), [ps[i]], [hist[i]], g1)
        assert int(t1.item()) == int(tb[i].item())
        assert float(l1.item()) == float(lb[i].item())
    s.close()


def test_bad_history_ids_raise_the_device_flag_only():
    s = Sampler(16, 1)
    x = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    tok, _ = s.sample(x, [sampling_params(temperature=0.0)], [([3, 99], [])], s.streams([0]))
    torch.cuda.synchronize()
    assert s.status() & dec.DEC_SAMPLE_BAD_ID
    assert int(tok.item()) == 0
    s.close()


def test_host_checks_refuse_bad_parameters():
    s = Sampler(16, 2)
    x = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    for bad in (dict(temperature=-1.0), dict(top_p=1.5), dict(min_p=-0.1), dict(repetition_penalty=0.0),
                dict(top_k=-3), dict(temperature=float("nan"))):
        with pytest.raises(dec.DecError):
            s.sample(x, [sampling_params(**bad)], None, s.streams([0]))
    s.close()


def test_sampling_the_decoders_logits():
    """The step after the LM head: the decoder's own device logits go straight
    into the sampler (no host round trip) and the oracle samples the same rows."""
    from .helpers import make_pair

    m, orc, w = make_pair("small", "bf16", max_positions=128, max_tokens=256, max_seqs=4)
    V = inputs.SHAPES["small"]["vocab"]
    prompts = [inputs.make_ids(V, n, seed=300 + i) for i, n in enumerate([17, 40, 65])]
    tables = [m.blocks_for(80) for _ in prompts]
    logits, _ = m.prefill([(p, 0, t) for p, t in zip(prompts, tables)], rows=dec.DEC_ROWS_LAST)
    ps = [sampling_params(temperature=0.8, top_k=50, top_p=0.9, repetition_penalty=1.1),
          sampling_params(temperature=1.0, min_p=0.1), sampling_params(temperature=0.0)]
    s = Sampler(V, 4)
    x = logits.float().contiguous()
    hist = [(list(p), []) for p in prompts]
    run_and_compare(s, x.cpu().numpy(), ps, hist, [9, 10, 11], "decoder logits")
    gen = s.streams([9, 10, 11])
    tok, _ = s.sample(x, ps, hist, gen)
    assert tok.dtype == torch.int32 and tok.is_cuda
    for t in tables:
        m.release(t)
    m.close()
    s.close()
