"""bench.py's reference arm on CPU: the line it prints and the step count it times.

The arm's oracle setup is swapped for the tiny shape so that the test runs in
seconds; the loop, the timing and the JSON line are bench.py's own."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from decoder_qwen3_step_gb300 import inputs  # noqa: E402
from oracle.model import DecoderConfig, Oracle  # noqa: E402

CONTRACT_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                 "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e")


def test_reference_arm_times_k_steps_after_w_and_prints_the_contract_line(monkeypatch):
    calls = []
    shape = inputs.SHAPES["tiny"]

    def tiny_sample(n_sample, horizon):
        cfg = DecoderConfig(**shape, max_positions=20 + horizon + 1)
        orc = Oracle(cfg, inputs.make_weights(shape), mode="bf16")
        rng = np.random.default_rng(1)
        caches = []
        for _ in range(n_sample):
            c = orc.new_cache(20 + horizon + 1)
            for l in range(cfg.n_layers):
                c.k[l][:20] = rng.standard_normal((20, cfg.n_kv_heads, cfg.head_dim))
                c.v[l][:20] = rng.standard_normal((20, cfg.n_kv_heads, cfg.head_dim))
                c.written[l][:20] = True
            caches.append(c)
        return orc, cfg, caches, [20] * n_sample

    real_step = bench._oracle_step

    def counting_step(orc, cfg, caches, pick, step):
        calls.append(step)
        real_step(orc, cfg, caches, pick, step)

    monkeypatch.setattr(bench, "_oracle_sample", tiny_sample)
    monkeypatch.setattr(bench, "_oracle_step", counting_step)

    class Args:
        steps, warmup = 5, 3

    line = bench.reference_arm(Args, 0, 1)
    assert calls == list(range(8))  # W untimed steps, then K timed ones, each at the next position
    for k in CONTRACT_KEYS:
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["steps"] == 5 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["e2e"]["value"] == line["value"] == line["cpu_baseline"]["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["sampled_sequences"] == 4


def test_reference_arm_samples_fewer_sequences_for_long_runs(monkeypatch):
    seen = {}

    def fake_sample(n_sample, horizon):
        seen["n"], seen["horizon"] = n_sample, horizon
        return None, None, [], []

    monkeypatch.setattr(bench, "_oracle_sample", fake_sample)
    monkeypatch.setattr(bench, "_oracle_step", lambda *a: None)

    class Args:
        steps, warmup = 1000, 5

    bench.reference_arm(Args, 0, 1)
    assert seen == {"n": 1, "horizon": 1005}
    assert bench.reference_arm(Args, 1, 2) is None  # only rank 0 runs the oracle
