"""Parity at the Qwen3-0.6B shape (596,049,920 parameters), through the C ABI.

* fp32 parity mode: one 188-token prompt, full prefill and 94 + 94 cached
  prefill with logits at every position, then 256 greedy decode tokens
  (octlm "Proving it's the same model": full vs cached path, max abs error
  <= 1e-3, argmax at every position).
* serving mode (bf16 weights, f16 KV, block 16): 32 sequences preloaded with
  contexts of distinct lengths 1024..2048 and 128 decode steps at batch 32;
  sampled sequences (the shortest and the longest) against the oracle run on
  the same bf16-rounded weights, tolerance 5e-2.
* serving mode chunked prefill: 4 x 4096 tokens in 512-token chunks
  interleaved across sequences, against each sequence's single 4096-token
  prefill run alone (chunk and batch invariance, tinyllm L10.1 section 2.4),
  the first sequence also against the oracle, then 64 decode steps at batch 4.

The oracle's decode is fed its own greedy ids; the device is fed the same
ids (teacher forcing), so both see identical inputs at every step.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402

from .helpers import TOLS, check, make_pair, np_  # noqa: E402

pytestmark = pytest.mark.gpu
SHAPE = inputs.SHAPES["qwen3_0p6b"]
V = SHAPE["vocab"]


@pytest.fixture(scope="module")
def weights():
    return inputs.make_weights(SHAPE)


def test_qwen3_fp32_full_cached_and_256_decode_tokens(weights):
    m, orc, _ = make_pair("qwen3_0p6b", "fp32", max_positions=512, max_tokens=512, max_seqs=4, n_blocks=96,
                          weights=weights)
    ids = inputs.make_ids(V, 188)
    ref_full = orc.full(ids)
    t1 = m.blocks_for(188)
    lg, am = m.prefill([(ids, 0, t1)])
    check(np_(lg), np_(am), ref_full, "fp32", "full", case="C3 qwen3-0.6B fp32", path="full prefill")
    del lg
    t2 = m.blocks_for(188 + 256)
    a1, i1 = m.prefill([(ids[:94], 0, t2)])
    a2, i2 = m.prefill([(ids[94:], 94, t2)])
    check(np.concatenate([np_(a1), np_(a2)]), np.concatenate([np_(i1), np_(i2)]), orc.cached(ids), "fp32", "cached",
          case="C3 qwen3-0.6B fp32", path="94+94 cached prefill")
    del a1, a2
    cache = orc.new_cache(188 + 257)
    orc.forward(cache, ids, 0, rows="last")
    tok = int(np.argmax(ref_full[-1]))
    worst = 0.0
    for i in range(256):
        ref = orc.forward(cache, [tok], 188 + i)
        lg, am = m.decode([([tok], 188 + i, t2)])
        r = check(np_(lg), np_(am), ref, "fp32", f"decode {i}", case="C3 qwen3-0.6B fp32" if i in (0, 255) else None,
                  path=f"decode step {i} (context {189 + i})")
        worst = max(worst, r["max_absolute_error"])
        tok = int(np.argmax(ref[0]))
    assert m.device_status() == 0
    print(f"fp32 0.6B: worst decode max abs error {worst:.3e}")
    m.close()


def test_qwen3_bf16_serving_batch32_decode(weights):
    lens = inputs.serving_context_lengths(32)
    steps = 128
    n_blocks = sum((L + steps + 16) // 16 + 1 for L in lens) + 16
    m, orc, _ = make_pair("qwen3_0p6b", "bf16", max_positions=2048 + steps + 16, max_tokens=8192, max_seqs=32,
                          n_blocks=n_blocks, weights=weights)
    ctx = [inputs.make_ids(V, 2048, seed=100 + s)[:lens[s]] for s in range(32)]
    tables = [m.blocks_for(L + steps + 1) for L in lens]
    last_lg, last_id = [], []
    for g in range(0, 32, 4):
        lg, am = m.prefill([(ctx[s], 0, tables[s]) for s in range(g, g + 4)], rows=dec.DEC_ROWS_LAST)
        last_lg.append(np_(lg))
        last_id.append(np_(am))
    last_lg = np.concatenate(last_lg)
    last_id = np.concatenate(last_id)
    sampled = [0, 15, 31]
    caches, feed = {}, [int(i) for i in last_id]
    for s in sampled:
        caches[s] = orc.new_cache(lens[s] + steps + 1)
        ref = orc.forward(caches[s], ctx[s], 0, rows="last")
        check(last_lg[s:s + 1], last_id[s:s + 1], ref, "bf16", f"preload seq {s}", case="C4 qwen3-0.6B serving",
              path=f"preload prefill, sequence {s} (context {lens[s]})")
        feed[s] = int(np.argmax(ref[0]))
    worst = 0.0
    tol = TOLS["bf16"]
    for i in range(steps):
        lg, am = m.decode([([feed[s]], lens[s] + i, tables[s]) for s in range(32)])
        lg, am = np_(lg), np_(am)
        assert np.isfinite(lg).all(), f"decode step {i}: non-finite logits"
        nxt = [int(x) for x in am]
        for s in sampled:
            ref = orc.forward(caches[s], [feed[s]], lens[s] + i)
            r = check(lg[s:s + 1], am[s:s + 1], ref, "bf16", f"decode step {i} seq {s}",
                      case="C4 qwen3-0.6B serving" if i in (0, steps - 1) else None,
                      path=f"batch-32 decode step {i}, sequence {s}")
            worst = max(worst, r["max_absolute_error"])
            nxt[s] = int(np.argmax(ref[0]))
        if i in (0, steps - 1):
            # every sequence once more on its own (the batch-1 path rewrites the same new key
            # and value): the same logits within the serving tolerance, the same id unless
            # the batch-32 row's top two are within 2 * tol (a near tie)
            for s in range(32):
                lg1, am1 = m.decode([([feed[s]], lens[s] + i, tables[s])])
                lg1, am1 = np_(lg1)[0], int(np_(am1)[0])
                assert np.abs(lg1 - lg[s]).max() <= tol, f"step {i} seq {s}: batch 1 vs batch 32"
                top2 = np.sort(lg[s])[-2:]
                assert am1 == int(am[s]) or top2[1] - top2[0] <= 2 * tol, f"step {i} seq {s}: ids differ"
        feed = nxt
    assert m.device_status() == 0
    print(f"bf16 0.6B batch 32: worst decode max abs error {worst:.3e}")
    m.close()


def test_qwen3_bf16_chunked_prefill_matches_single_prefill_and_oracle(weights):
    m, orc, _ = make_pair("qwen3_0p6b", "bf16", max_positions=4096 + 64 + 16, max_tokens=4096, max_seqs=4,
                          n_blocks=4 * 2 * 262 + 16, weights=weights)
    seqs = [inputs.make_ids(V, 4096, seed=200 + s) for s in range(4)]
    tabs = [m.blocks_for(4096 + 65) for _ in range(4)]
    chunk_lg, chunk_id = [], []
    for k in range(8):
        lg, am = m.prefill([(seqs[s][512 * k:512 * (k + 1)], 512 * k, tabs[s]) for s in range(4)],
                           rows=dec.DEC_ROWS_LAST)
        chunk_lg.append(np_(lg))
        chunk_id.append(np_(am))
    chunk_lg = np.stack(chunk_lg)  # [8 chunks, 4 seqs, V]
    chunk_id = np.stack(chunk_id)
    rows = np.arange(511, 4096, 512)
    bitwise = True
    for s in range(4):
        single = m.blocks_for(4096)
        lg, am = m.prefill([(seqs[s], 0, single)])
        idx = torch.from_numpy(rows).to(lg.device)
        lg_s = np_(lg.index_select(0, idx))
        del lg, am
        m.release(single)
        diff = np.abs(lg_s - chunk_lg[:, s]).max()
        bitwise &= bool(np.array_equal(lg_s, chunk_lg[:, s]))
        assert diff <= 5e-2, f"seq {s}: chunked vs single {diff}"
    print(f"chunked vs single prefill bitwise equal: {bitwise}")
    # the first sequence against the oracle, chunk by chunk (the oracle's chunked
    # path equals its full path to rounding, a pinned invariant)
    cache = orc.new_cache(4096 + 65)
    for k in range(8):
        ref = orc.forward(cache, seqs[0][512 * k:512 * (k + 1)], 512 * k, rows="last")
        check(chunk_lg[k, 0:1], chunk_id[k, 0:1], ref, "bf16", f"chunk {k}", case="C5 qwen3-0.6B chunked prefill",
              path=f"chunk {k} of sequence 0 (positions {512 * k}..{512 * k + 511})")
    # 64 decode steps at batch 4
    feed = [int(chunk_id[-1, s]) for s in range(4)]
    feed[0] = int(np.argmax(ref[0]))
    for i in range(64):
        lg, am = m.decode([([feed[s]], 4096 + i, tabs[s]) for s in range(4)])
        lg, am = np_(lg), np_(am)
        r = orc.forward(cache, [feed[0]], 4096 + i)
        check(lg[0:1], am[0:1], r, "bf16", f"decode {i}", case="C5 qwen3-0.6B chunked prefill" if i in (0, 63) else None,
              path=f"batch-4 decode step {i}, sequence 0")
        feed = [int(x) for x in am]
        feed[0] = int(np.argmax(r[0]))
    assert m.device_status() == 0
    m.close()
