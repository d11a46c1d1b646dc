"""The serving-mode decode step as one persistent kernel (dec_set_megakernel).

Its logits are checked against the float64 oracle on the bf16-rounded
weights (the serving tolerance and argmax rule), against the per-operation
kernels, for batch invariance (a sequence's logits are the same bits alone or
in a batch: every reduction has one fixed order), on contexts that cross
16-key blocks and 64-key attention chunks, and at the Qwen3-0.6B shape.  The
kernel-class counter proves the one-kernel path is the one that ran."""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402
from .helpers import check, make_pair, np_  # noqa: E402

pytestmark = pytest.mark.gpu

STEP = dec.KERNEL_CLASSES.index("step")


def step_launches(m):
    ms, n = C.c_double(), C.c_int64()
    dec.check(m.L.dec_profile_read(m.handle, STEP, C.byref(ms), C.byref(n)), "dec_profile_read")
    return n.value


def decode_run(m, orc, prompts, steps, start_tok=None):
    """Prefill every prompt, then `steps` greedy decode steps at batch
    len(prompts), teacher-forced on the oracle's ids; returns the device
    logits and ids of every step and the oracle's rows."""
    S = len(prompts)
    tables = [m.blocks_for(len(p) + steps + 1) for p in prompts]
    m.prefill([(p, 0, t) for p, t in zip(prompts, tables)], rows=dec.DEC_ROWS_LAST)
    caches, toks = [], []
    for p in prompts:
        c = orc.new_cache(len(p) + steps + 1)
        ref = orc.forward(c, p, 0, rows="last")
        caches.append(c)
        toks.append(int(np.argmax(ref[-1])))
    got, ids, want = [], [], []
    for i in range(steps):
        refs = [orc.forward(caches[s], [toks[s]], len(prompts[s]) + i)[0] for s in range(S)]
        lg, am = m.decode([([toks[s]], len(prompts[s]) + i, tables[s]) for s in range(S)])
        got.append(np_(lg))
        ids.append(np_(am))
        want.append(np.stack(refs))
        toks = [int(np.argmax(r)) for r in refs]
    for t in tables:
        m.release(t)
    return got, ids, want


@pytest.mark.parametrize("shape", ["tiny", "small"])
def test_one_kernel_step_matches_the_oracle_and_the_layered_kernels(shape):
    m, orc, w = make_pair(shape, "bf16", max_positions=256, max_tokens=512, max_seqs=8)
    if not m.megakernel_available():
        pytest.skip("the one-kernel step is not available for this shape on this device")
    V = inputs.SHAPES[shape]["vocab"]
    # contexts that end inside, and just past, 16-key blocks and 64-key chunks
    lens = [13, 63, 64, 100] if shape == "tiny" else [60, 64, 128, 129]
    prompts = [inputs.make_ids(V, n, seed=40 + s) for s, n in enumerate(lens)]
    m.L.dec_profile_enable(m.handle, STEP, 1)
    step_launches(m)
    got, ids, want = decode_run(m, orc, prompts, steps=6)
    assert step_launches(m) == 6  # every decode step was one launch of the persistent kernel
    m.L.dec_profile_enable(m.handle, STEP, 0)
    for i in range(6):
        check(got[i], ids[i], want[i], "bf16", f"{shape} one-kernel decode step {i}")
    # the same steps on the per-operation kernels
    m.set_megakernel(False)
    got2, ids2, want2 = decode_run(m, orc, prompts, steps=6)
    for i in range(6):
        check(got2[i], ids2[i], want2[i], "bf16", f"{shape} layered decode step {i}")
        assert np.abs(got[i] - got2[i]).max() < 5e-2
    assert m.device_status() == 0
    m.close()


def test_one_kernel_step_is_batch_invariant():
    m, orc, w = make_pair("small", "bf16", max_positions=256, max_tokens=512, max_seqs=8)
    if not m.megakernel_available():
        pytest.skip("the one-kernel step is not available on this device")
    prompts = [inputs.make_ids(8192, n, seed=70 + s) for s, n in enumerate([90, 33, 150])]
    tables = [m.blocks_for(200) for _ in prompts]
    alone = [m.blocks_for(200) for _ in prompts]
    for p, t, u in zip(prompts, tables, alone):  # identical caches for both copies
        m.prefill([(p, 0, t)], rows=dec.DEC_ROWS_LAST)
        m.prefill([(p, 0, u)], rows=dec.DEC_ROWS_LAST)
    tok = [5, 77, 4000]
    for i in range(3):
        lg_b, _ = m.decode([([tok[s]], len(prompts[s]) + i, tables[s]) for s in range(3)])
        lg_b = np_(lg_b)
        for s in range(3):
            lg_1, _ = m.decode([([tok[s]], len(prompts[s]) + i, alone[s])])
            assert np.array_equal(np_(lg_1)[0].view(np.uint32), lg_b[s].view(np.uint32)), (i, s)
    assert m.device_status() == 0
    m.close()


def test_one_kernel_step_reads_ids_from_the_device():
    """The ids of a step may come from the previous step's argmax buffer."""
    m, orc, w = make_pair("tiny", "bf16", max_positions=128, max_tokens=128, max_seqs=4)
    if not m.megakernel_available():
        pytest.skip("the one-kernel step is not available on this device")
    prompts = [inputs.make_ids(512, n, seed=90 + s) for s, n in enumerate([20, 47])]
    tables = [m.blocks_for(80) for _ in prompts]
    host = [m.blocks_for(80) for _ in prompts]
    _, am = m.prefill([(p, 0, t) for p, t in zip(prompts, tables)], rows=dec.DEC_ROWS_LAST)
    _, am_h = m.prefill([(p, 0, t) for p, t in zip(prompts, host)], rows=dec.DEC_ROWS_LAST)
    ids_dev = am.to(torch.int32).clone()
    ids_host = np_(am_h).astype(np.int64)
    logits = torch.empty((2, 512), dtype=torch.float32, device=m.device)
    out_ids = torch.empty((2,), dtype=torch.int32, device=m.device)
    for i in range(5):
        pos = [len(p) + i for p in prompts]
        m.decode([([0], pos[s], tables[s]) for s in range(2)], device_ids=ids_dev, out=(logits, out_ids))
        lg_h, am_h = m.decode([([int(ids_host[s])], pos[s], host[s]) for s in range(2)])
        assert np.array_equal(np_(logits).view(np.uint32), np_(lg_h).view(np.uint32))
        assert np.array_equal(np_(out_ids), np_(am_h))
        ids_dev.copy_(out_ids)
        ids_host = np_(am_h).astype(np.int64)
    assert m.device_status() == 0
    m.close()


def test_one_kernel_step_at_the_qwen3_shape():
    m, orc, w = make_pair("qwen3_0p6b", "bf16", max_positions=512, max_tokens=512, max_seqs=4, n_blocks=160)
    if not m.megakernel_available():
        pytest.skip("the one-kernel step is not available on this device")
    prompts = [inputs.make_ids(151936, n, seed=120 + s) for s, n in enumerate([61, 190])]
    got, ids, want = decode_run(m, orc, prompts, steps=4)
    for i in range(4):
        check(got[i], ids[i], want[i], "bf16", f"0.6B one-kernel decode step {i}")
    assert m.device_status() == 0
    m.close()


def test_one_kernel_step_at_the_bench_batch1_case():
    """The bench's batch-1 decode case exactly: the Qwen3-0.6B shape in the
    serving mode, one sequence whose 2,048-token context is the bench's
    longest (ids seed 131), decode steps on the one-kernel path, each checked
    against the oracle on the same bf16-rounded weights."""
    shape = inputs.SHAPES["qwen3_0p6b"]
    V = shape["vocab"]
    m, orc, w = make_pair("qwen3_0p6b", "bf16", max_positions=2048 + 64, max_tokens=2048, max_seqs=1, n_blocks=140)
    if not m.megakernel_available():
        pytest.skip("the one-kernel step is not available on this device")
    ctx = inputs.make_ids(V, 2048, seed=100 + 31)
    table = m.blocks_for(2048 + 8)
    m.prefill([(ctx, 0, table)], rows=dec.DEC_ROWS_LAST)
    cache = orc.new_cache(2048 + 8)
    tok = int(np.argmax(orc.forward(cache, ctx, 0, rows="last")[-1]))
    m.L.dec_profile_enable(m.handle, STEP, 1)
    step_launches(m)
    for i in range(4):
        ref = orc.forward(cache, [tok], 2048 + i)
        lg, am = m.decode([([tok], 2048 + i, table)])
        check(np_(lg), np_(am), ref, "bf16", f"batch-1 decode step {i}", case="decode_b1 bench case",
              path=f"one-kernel decode step {i} (context {2049 + i})")
        tok = int(np.argmax(ref[0]))
    assert step_launches(m) == 4
    m.L.dec_profile_enable(m.handle, STEP, 0)
    assert m.device_status() == 0
    m.close()


def test_one_kernel_step_wait_gives_up_and_the_gpu_stays_usable():
    """A bounded wait of the one-kernel step runs out on purpose (the test
    hook makes every hand-off expect one arrival too many, with a 2 ms
    limit): the step ends with DEC_DEV_TIMEOUT in the device error word, no
    fault; then the same step with the normal waits matches the oracle."""
    m, orc, w = make_pair("tiny", "bf16", max_positions=128, max_tokens=128, max_seqs=2)
    if not m.megakernel_available():
        pytest.skip("the one-kernel step is not available on this device")
    prompt = inputs.make_ids(512, 37, seed=140)
    table = m.blocks_for(48)
    m.prefill([(prompt, 0, table)], rows=dec.DEC_ROWS_LAST)
    cache = orc.new_cache(48)
    tok = int(np.argmax(orc.forward(cache, prompt, 0, rows="last")[-1]))
    assert m.device_status() == 0
    with pytest.raises(dec.DecError):  # the limit is bounded on both sides
        dec.check(m.L.dec_debug_wait_timeout(m.handle, 1, 10), "dec_debug_wait_timeout")
    dec.check(m.L.dec_debug_wait_timeout(m.handle, 1, 2_000_000), "dec_debug_wait_timeout")
    m.decode([([tok], 37, table)])
    assert m.device_status() & dec.DEC_DEV_TIMEOUT
    dec.check(m.L.dec_debug_wait_timeout(m.handle, 0, 0), "dec_debug_wait_timeout")
    ref = orc.forward(cache, [tok], 37)
    lg, am = m.decode([([tok], 37, table)])
    check(np_(lg), np_(am), ref, "bf16", "decode after a timed-out step")
    assert m.device_status() == 0
    m.close()


def test_long_context_decode_merges_records_without_staging():
    """Contexts long enough that a (sequence, KV head)'s chunk records no longer
    fit the decode attention kernel's shared-memory staging (more than 52
    64-key chunks at head_dim 64): the merge then reads the records from
    global memory.  Two sequences of about 3,500 tokens at the small shape,
    decoded on the per-operation kernels (the one-kernel step off), against
    the oracle."""
    lens = [3400, 3530]
    m, orc, w = make_pair("small", "bf16", max_positions=3600, max_tokens=10496, max_seqs=4,
                          n_blocks=sum((n + 16) // 16 + 1 for n in lens) + 8)
    m.set_megakernel(False)
    V = inputs.SHAPES["small"]["vocab"]
    prompts = [inputs.make_ids(V, n, seed=160 + s) for s, n in enumerate(lens)]
    got, ids, want = decode_run(m, orc, prompts, steps=2)
    for i in range(2):
        check(got[i], ids[i], want[i], "bf16", f"long-context decode step {i}", case="long-context decode",
              path=f"per-operation decode step {i}, contexts {[n + 1 + i for n in lens]}")
    assert m.device_status() == 0
    m.close()


def test_decode_above_32_sequences_matches_the_oracle():
    """A decode step of 40 sequences: more token rows than the skinny
    products take, so the projections run on the many-token tcgen05 kernel,
    and the decode attention's items span 40 x 4 (sequence, KV head) pairs of
    different lengths (small shape, serving mode), against the oracle."""
    S = 40
    m, orc, w = make_pair("small", "bf16", max_positions=256, max_tokens=8192, max_seqs=S)
    V = inputs.SHAPES["small"]["vocab"]
    prompts = [inputs.make_ids(V, 20 + 5 * s, seed=200 + s) for s in range(S)]
    got, ids, want = decode_run(m, orc, prompts, steps=2)
    for i in range(2):
        check(got[i], ids[i], want[i], "bf16", f"40-sequence decode step {i}", case="decode above 32 sequences",
              path=f"per-operation decode step {i}, 40 sequences")
    assert m.device_status() == 0
    m.close()
