"""GPU parity of the whole decoder step against the float64 oracle, through
the C ABI, on the tiny and small shapes (several tiles and ragged tails),
plus the boundary's refusals and the bit-exact pieces.

Paths (octlm "Proving it's the same model"): full prompt, cached (first half,
then the second half on top of its cache), and greedy decode one token at a
time, teacher-forced on the oracle's greedy ids.  Gates fixed before any run:
max abs logit error <= 1e-3 (fp32) / 5e-2 (bf16 weights, f16 KV) and argmax
agreement on every row under the near-tie rule."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402
from oracle import numerics as nm  # noqa: E402

from .helpers import check, make_pair, np_  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=["fp32", "bf16"])
def tiny(request):
    m, orc, w = make_pair("tiny", request.param, max_positions=64, max_tokens=256, max_seqs=8)
    yield request.param, m, orc, w
    m.close()


def test_tiny_full_cached_and_greedy_decode(tiny):
    mode, m, orc, w = tiny
    ids = inputs.make_ids(512, 16)
    ref_full = orc.full(ids)
    table = m.blocks_for(25)
    lg, am = m.prefill([(ids, 0, table)])
    check(np_(lg), np_(am), ref_full, mode, "full", case="C1 tiny", path="full prefill (16 tokens)")
    # cached: 8 + 8 on top of the first half's cache
    t2 = m.blocks_for(25)
    a1, i1 = m.prefill([(ids[:8], 0, t2)])
    a2, i2 = m.prefill([(ids[8:], 8, t2)])
    check(np.concatenate([np_(a1), np_(a2)]), np.concatenate([np_(i1), np_(i2)]), orc.cached(ids), mode, "cached",
          case="C1 tiny", path="8+8 cached prefill")
    # 8 greedy decode steps on the cached sequence
    cache = orc.new_cache(64)
    orc.forward(cache, ids, 0)
    fed, rows = orc.greedy(cache, int(np.argmax(ref_full[-1])), 16, 8)
    for i, tok in enumerate(fed):
        lg, am = m.decode([([tok], 16 + i, t2)])
        check(np_(lg), np_(am), rows[i:i + 1], mode, f"decode {i}", case="C1 tiny", path=f"greedy decode step {i}")
    assert m.device_status() == 0
    m.release(table)
    m.release(t2)


def test_tiny_context_filled_to_the_last_position(tiny):
    """The largest context the model was made for: a 60-token prompt, then
    greedy decode at positions 60..63, the last row of the RoPE table and the
    last slot of the fourth (last) 16-token block."""
    mode, m, orc, w = tiny
    ids = inputs.make_ids(512, 60, seed=11)
    table = m.blocks_for(64)
    assert len(table) == 4
    lg, am = m.prefill([(ids, 0, table)], rows=dec.DEC_ROWS_LAST)
    cache = orc.new_cache(64)
    ref = orc.forward(cache, ids, 0, rows="last")
    check(np_(lg), np_(am), ref, mode, "prompt of 60")
    fed, rows = orc.greedy(cache, int(np.argmax(ref[-1])), 60, 4)
    for i, tok in enumerate(fed):
        lg, am = m.decode([([tok], 60 + i, table)])
        check(np_(lg), np_(am), rows[i:i + 1], mode, f"decode at position {60 + i}")
    assert m.device_status() == 0
    m.release(table)


def test_tiny_embedding_rows_are_bit_exact(tiny):
    mode, m, orc, w = tiny
    ids = inputs.make_ids(512, 16, seed=7)
    dump = torch.zeros((3, 16, 64), dtype=torch.float32, device=m.device)
    m.set_dump(dump)
    table = m.blocks_for(16)
    m.prefill([(ids, 0, table)])
    torch.cuda.synchronize()
    m.set_dump(None)
    rows = w["embed"][ids]
    expect = nm.bf16_round(rows) if mode == "bf16" else rows
    assert np.array_equal(np_(dump[0]).view(np.uint32), expect.view(np.uint32))
    # layer-by-layer residuals stay close to the oracle's
    ref = []
    orc.forward(orc.new_cache(64), ids, 0, dump=ref)
    for i in range(1, 3):
        assert np.abs(np_(dump[i]) - ref[i]).max() < (1e-4 if mode == "fp32" else 2e-2)
    m.release(table)


def test_small_batched_full_cached_and_decode():
    for mode in ("fp32", "bf16"):
        m, orc, w = make_pair("small", mode, max_positions=256, max_tokens=1024, max_seqs=8)
        prompts = [inputs.make_ids(8192, 128, seed=10 + s) for s in range(4)]
        tables = [m.blocks_for(128 + 64) for _ in range(4)]
        # full: the 4 prompts in one step (512 tokens), logits at every position
        lg, am = m.prefill([(p, 0, t) for p, t in zip(prompts, tables)])
        lg, am = np_(lg), np_(am)
        caches = []
        for s, p in enumerate(prompts):
            cache = orc.new_cache(256)
            ref = orc.forward(cache, p, 0)
            caches.append(cache)
            check(lg[128 * s:128 * (s + 1)], am[128 * s:128 * (s + 1)], ref, mode, f"{mode} full seq {s}",
                  case="C2 small", path=f"full prefill, batch 4, sequence {s}")
        # cached: 64 + 64, both halves batched over the 4 sequences
        t2 = [m.blocks_for(128 + 64) for _ in range(4)]
        a1, i1 = m.prefill([(p[:64], 0, t) for p, t in zip(prompts, t2)])
        a2, i2 = m.prefill([(p[64:], 64, t) for p, t in zip(prompts, t2)])
        a1, i1, a2, i2 = np_(a1), np_(i1), np_(a2), np_(i2)
        for s, p in enumerate(prompts):
            got = np.concatenate([a1[64 * s:64 * (s + 1)], a2[64 * s:64 * (s + 1)]])
            gid = np.concatenate([i1[64 * s:64 * (s + 1)], i2[64 * s:64 * (s + 1)]])
            check(got, gid, orc.cached(p), mode, f"{mode} cached seq {s}", case="C2 small",
                  path=f"64+64 cached prefill, sequence {s}")
        # 64 greedy decode steps at batch 4, teacher-forced on the oracle's ids
        steps = 64
        toks = [int(np.argmax(orc.forward(orc.new_cache(256), p, 0)[-1])) for p in prompts]
        for i in range(steps):
            refs = [orc.forward(caches[s], [toks[s]], 128 + i)[0] for s in range(4)]
            lg, am = m.decode([([toks[s]], 128 + i, t2[s]) for s in range(4)])
            check(np_(lg), np_(am), np.stack(refs), mode, f"{mode} decode step {i}",
                  case="C2 small" if i in (0, steps - 1) else None, path=f"batch-4 decode step {i}")
            toks = [int(np.argmax(r)) for r in refs]
        assert m.device_status() == 0
        m.close()


def test_tensor_core_products_match_cuda_core_products():
    """Serving mode, 300-token prefill of the small shape: the tcgen05 products
    and the CUDA-core products add the same bf16 products in another order.
    After the first layer the residual streams agree to within the bf16
    rounding of the attention output (a summation-order difference in k can
    flip an f16 key, which moves many bf16 roundings downstream); both end
    results are held to the oracle.  The products alone are pinned exactly in
    test_gpu_products.py."""
    m, orc, w = make_pair("small", "bf16", max_positions=512, max_tokens=512, max_seqs=4)
    ids = inputs.make_ids(8192, 300, seed=77)
    out, dumps = {}, {}
    for tc in (True, False):
        m.set_tensor_cores(tc)
        dump = torch.zeros((9, 300, 512), dtype=torch.float32, device=m.device)
        m.set_dump(dump)
        t = m.blocks_for(300)
        lg, am = m.prefill([(ids, 0, t)])
        torch.cuda.synchronize()
        m.set_dump(None)
        out[tc] = (np_(lg), np_(am))
        dumps[tc] = np_(dump)
        m.release(t)
    assert m.device_status() == 0
    x1_tc, x1_cc = dumps[True][1], dumps[False][1]
    scale = np.abs(x1_cc).max()
    assert np.abs(x1_tc - x1_cc).max() <= 5e-3 * scale, (np.abs(x1_tc - x1_cc).max(), scale)
    ref = orc.full(ids)
    check(out[True][0], out[True][1], ref, "bf16", "tensor cores vs oracle")
    check(out[False][0], out[False][1], ref, "bf16", "CUDA cores vs oracle")
    print("tc vs cuda-core: layer-1 residual max diff", float(np.abs(x1_tc - x1_cc).max()), "scale", float(scale),
          "logits max diff", float(np.abs(out[True][0] - out[False][0]).max()))
    m.close()


def test_batched_forward_equals_single(tiny):
    mode, m, orc, w = tiny
    a = inputs.make_ids(512, 13, seed=3)
    b = inputs.make_ids(512, 7, seed=4)
    ta, tb = m.blocks_for(13), m.blocks_for(7)
    la, _ = m.prefill([(a, 0, ta)])
    lb, _ = m.prefill([(b, 0, tb)])
    tc, td = m.blocks_for(13), m.blocks_for(7)
    lab, _ = m.prefill([(a, 0, tc), (b, 0, td)])
    both = np_(lab)
    tol = 1e-5 if mode == "fp32" else 1e-3
    assert np.abs(both[:13] - np_(la)).max() <= tol
    assert np.abs(both[13:] - np_(lb)).max() <= tol
    for t in (ta, tb, tc, td):
        m.release(t)


def test_step_refuses_bad_batches_and_leaves_the_cache_untouched(tiny):
    mode, m, orc, w = tiny
    ids = inputs.make_ids(512, 8)
    table = m.blocks_for(16)
    extra = m.blocks_for(1)
    freed = m.blocks_for(16)
    m.release(freed)
    m.prefill([(ids, 0, table)])
    torch.cuda.synchronize()
    before = m.slabs.clone()
    free_before = m.free_blocks()

    def refused(code, seqs, decode=False):
        with pytest.raises(dec.DecError) as e:
            (m.decode if decode else m.prefill)(seqs)
        assert e.value.code == code, str(e.value)

    refused(dec.DEC_EVOCAB, [([5, 512], 8, table)])
    refused(dec.DEC_EVOCAB, [([-1], 8, table)])
    refused(dec.DEC_ERANGE, [([1, 2], 63, table + extra + extra + extra)])  # position 64 is past the context
    refused(dec.DEC_ERANGE, [([1] * 9, 8, table[:1])])  # table too short for position 16
    refused(dec.DEC_EBLOCK, [([1], 8, [m.n_blocks + 3])])
    refused(dec.DEC_EBLOCK, [([1], 8, freed)])  # block not allocated
    refused(dec.DEC_EINVAL, [([1, 2], 8, table)], decode=True)  # decode takes one token per sequence
    with pytest.raises(dec.DecError):
        m.prefill([])
    torch.cuda.synchronize()
    assert torch.equal(before, m.slabs)
    assert m.free_blocks() == free_before
    m.release(table)
    m.release(extra)


def test_device_ids_out_of_vocab_raise_the_device_flag(tiny):
    mode, m, orc, w = tiny
    table = m.blocks_for(4)
    bad = torch.tensor([600], dtype=torch.int32, device=m.device)
    m.decode([([0], 0, table)], device_ids=bad)
    assert m.device_status() & dec.DEC_DEV_BAD_ID
    assert m.device_status() == 0  # the read cleared it
    m.release(table)


def test_run_once_returns_its_blocks(tiny):
    mode, m, orc, w = tiny
    free = m.free_blocks()
    for i in range(5):
        t = m.blocks_for(10)
        m.prefill([(inputs.make_ids(512, 10, seed=i), 0, t)], rows=dec.DEC_ROWS_LAST)
        m.release(t)
    assert m.free_blocks() == free


def test_graph_replay_matches_eager_decode_bitwise(tiny):
    mode, m, orc, w = tiny
    prompts = [inputs.make_ids(512, n, seed=20 + n) for n in (5, 9, 16)]
    outs = {}
    for graphs in (False, True):
        m.set_graphs(graphs)
        tabs = [m.blocks_for(40) for _ in prompts]
        m.prefill([(p, 0, t) for p, t in zip(prompts, tabs)], rows=dec.DEC_ROWS_LAST)
        lg = torch.empty((3, 512), dtype=torch.float32, device=m.device)
        ids = [torch.empty((3,), dtype=torch.int32, device=m.device) for _ in range(2)]
        ids[0].fill_(7)
        rows = []
        for i in range(6):  # eager, capture, then replays; ids fed back on the device
            m.decode([([0], len(p) + i, t) for p, t in zip(prompts, tabs)], device_ids=ids[i & 1],
                     out=(lg, ids[(i + 1) & 1]))
            rows.append(np_(lg).copy())
        outs[graphs] = np.stack(rows)
        for t in tabs:
            m.release(t)
    m.set_graphs(True)
    assert np.array_equal(outs[False], outs[True])
    assert m.device_status() == 0


def test_profiled_classes_stay_timed_inside_graph_replays(tiny):
    """Attention and the LM head profiled while decode steps replay a graph:
    the logits equal the eager ones bit for bit, and every step (eager,
    captured or replayed) contributes one timed launch per layer (attention)
    and one per step (LM head)."""
    import ctypes as C

    mode, m, orc, w = tiny
    n_layers = inputs.SHAPES["tiny"]["n_layers"]
    classes = (dec.KERNEL_CLASSES.index("attn"), dec.KERNEL_CLASSES.index("lmhead"))
    prompts = [inputs.make_ids(512, n, seed=40 + n) for n in (6, 11)]
    m.set_megakernel(False)
    outs, counts = {}, {}
    for graphs in (False, True):
        m.set_graphs(graphs)
        tabs = [m.blocks_for(40) for _ in prompts]
        m.prefill([(p, 0, t) for p, t in zip(prompts, tabs)], rows=dec.DEC_ROWS_LAST)
        lg = torch.empty((2, 512), dtype=torch.float32, device=m.device)
        ids = [torch.empty((2,), dtype=torch.int32, device=m.device) for _ in range(2)]
        ids[0].fill_(3)
        for c in classes:
            dec.check(m.L.dec_profile_enable(m.handle, c, 1), "dec_profile_enable")
        rows = []
        for i in range(6):
            m.decode([([0], len(p) + i, t) for p, t in zip(prompts, tabs)], device_ids=ids[i & 1],
                     out=(lg, ids[(i + 1) & 1]))
            rows.append(np_(lg).copy())
        got = []
        for c in classes:
            ms, n = C.c_double(), C.c_int64()
            dec.check(m.L.dec_profile_read(m.handle, c, C.byref(ms), C.byref(n)), "dec_profile_read")
            dec.check(m.L.dec_profile_enable(m.handle, c, 0), "dec_profile_enable")
            assert ms.value > 0.0
            got.append(n.value)
        outs[graphs], counts[graphs] = np.stack(rows), got
        for t in tabs:
            m.release(t)
    m.set_graphs(True)
    m.set_megakernel(True)
    assert np.array_equal(outs[False], outs[True])
    assert counts[False] == counts[True] == [6 * n_layers, 6]
    assert m.device_status() == 0


def test_f16_kv_store_rounds_to_nearest_even_bit_exact():
    import ctypes as C

    L = dec.lib()
    base = nm.f16_bits_to_f32(np.arange(0, 0x7C00, dtype=np.uint16)).astype(np.float64)
    nxt = nm.f16_bits_to_f32(np.arange(1, 0x7C01, dtype=np.uint16)).astype(np.float64)
    rng = np.random.default_rng(9)
    vals = np.concatenate([((base + nxt) / 2).astype(np.float32), np.float32([1 + 2 ** -11, 1 + 3 * 2 ** -11,
                                                                              65519, 65520, -65520, 2 ** -25]),
                           (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 12, 100000))).astype(np.float32)])
    x = torch.from_numpy(vals).cuda()
    out = torch.empty(x.numel(), dtype=torch.int16, device="cuda")
    s = torch.cuda.current_stream()
    dec.check(L.dec_f32_to_f16(C.c_void_p(x.data_ptr()), C.c_void_p(out.data_ptr()), x.numel(),
                               C.c_void_p(s.cuda_stream)), "dec_f32_to_f16")
    got = np_(out).view(np.uint16)
    assert np.array_equal(got, nm.f32_to_f16_bits(vals))
    assert int(got[vals.size - 100000 - 6]) == 0x3C00 and int(got[vals.size - 100000 - 5]) == 0x3C02
