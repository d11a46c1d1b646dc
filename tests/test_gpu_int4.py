"""Int4 weights on the GPU (DEC_INT4_F16KV) against the int4 oracle.

The quantizer is compared bit for bit with the oracle's (codes and f16
scales, including an all-zero group and rounding ties); the int4 product
against X times the oracle's effective weights in float64; the whole decoder
(full prompt, cached halves, batched ragged prefill, greedy decode) against
the oracle's int4 mode at the serving tolerance (5e-2, argmax under the
near-tie rule): the effective weights are exact on both sides, so the error
budget is the bf16 activations and f16 cache of the serving mode."""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402
from oracle import int4 as Q  # noqa: E402
from oracle import numerics as nm  # noqa: E402

from .helpers import check, make_pair, np_  # noqa: E402

pytestmark = pytest.mark.gpu


def test_quantizer_is_bit_exact():
    g = np.random.default_rng(0)
    W = (g.standard_normal((96, 320)) * g.uniform(0.001, 4.0, (96, 1))).astype(np.float32)
    W[5, 64:96] = 0.0                                  # an all-zero group
    W[7, :32] = 0.0
    W[7, :5] = [7.0, 2.5, 3.5, -0.5, -2.5]             # scale exactly 1: ties to even
    W[9, :4] = [0.7, -1.4, 0.0, 0.29995]               # the pages' hand example inside a group of 32
    q, s = Q.quantize(W)
    Wd = torch.from_numpy(W).cuda()
    codes = torch.zeros((96, 160), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((96, 10), dtype=torch.int16, device="cuda")
    dec.check(dec.lib().dec_quantize_int4(C.c_void_p(Wd.data_ptr()), 96, 320, C.c_void_p(codes.data_ptr()),
                                          C.c_void_p(scales.data_ptr()), None), "dec_quantize_int4")
    torch.cuda.synchronize()
    assert np.array_equal(np_(codes), Q.pack(q))
    assert np.array_equal(np_(scales).view(np.uint16), s)


@pytest.mark.parametrize("which", [0, 1, 2, 3])
def test_int4_products_match_the_effective_weights(which):
    m, orc, w = make_pair("small", "int4", max_positions=64, max_tokens=64, max_seqs=4)
    shape = inputs.SHAPES["small"]
    d, HD, F = shape["d_model"], shape["n_heads"] * shape["head_dim"], shape["ff_hidden"]
    L = orc.layers[1]
    mats = {0: np.concatenate([L["q"], L["k"], L["v"]]), 1: L["o"], 3: L["down"]}
    if which == 2:  # gate and up rows interleave in groups of 8
        G, U = L["gate"], L["up"]
        mats[2] = np.concatenate([np.concatenate([G[i:i + 8], U[i:i + 8]]) for i in range(0, F, 8)])
    Wm = mats[which]
    K = Wm.shape[1]
    for T in (1, 5, 8, 13, 40):
        x = np.random.default_rng(T).standard_normal((T, K)).astype(np.float32)
        xb = nm.bf16_round(x)
        X = torch.from_numpy(xb).cuda().to(torch.bfloat16)
        Y = torch.empty((T, Wm.shape[0]), dtype=torch.float32, device="cuda")
        dec.check(m.L.dec_debug_product(m.handle, which, 1, C.c_void_p(X.data_ptr()), T, C.c_void_p(Y.data_ptr()), 0,
                                        None), "dec_debug_product")
        torch.cuda.synchronize()
        ref = xb.astype(np.float64) @ Wm.T
        scale = np.abs(xb).astype(np.float64) @ np.abs(Wm).T + 1e-30
        assert np.max(np.abs(np_(Y) - ref) / scale) < 1e-5, (which, T)
    m.close()


def test_tiny_full_cached_and_greedy_decode_int4():
    m, orc, w = make_pair("tiny", "int4", max_positions=64, max_tokens=256, max_seqs=8)
    ids = inputs.make_ids(512, 16)
    ref_full = orc.full(ids)
    table = m.blocks_for(25)
    lg, am = m.prefill([(ids, 0, table)])
    check(np_(lg), np_(am), ref_full, "int4", "full")
    t2 = m.blocks_for(25)
    a1, i1 = m.prefill([(ids[:8], 0, t2)])
    a2, i2 = m.prefill([(ids[8:], 8, t2)])
    check(np.concatenate([np_(a1), np_(a2)]), np.concatenate([np_(i1), np_(i2)]), orc.cached(ids), "int4", "cached")
    cache = orc.new_cache(64)
    orc.forward(cache, ids, 0)
    fed, rows = orc.greedy(cache, int(np.argmax(ref_full[-1])), 16, 8)
    for i, tok in enumerate(fed):
        lg, am = m.decode([([tok], 16 + i, t2)])
        check(np_(lg), np_(am), rows[i:i + 1], "int4", f"decode {i}")
    assert m.device_status() == 0
    m.close()


def test_small_batched_ragged_prefill_and_decode_int4():
    m, orc, w = make_pair("small", "int4", max_positions=256, max_tokens=1024, max_seqs=8)
    lens = [37, 128, 64, 100]
    prompts = [inputs.make_ids(8192, n, seed=20 + s) for s, n in enumerate(lens)]
    tables = [m.blocks_for(n + 8) for n in lens]
    lg, am = m.prefill([(p, 0, t) for p, t in zip(prompts, tables)], rows=dec.DEC_ROWS_LAST)
    caches, toks = [], []
    want = []
    for p in prompts:
        c = orc.new_cache(256)
        want.append(orc.forward(c, p, 0, rows="last")[-1])
        caches.append(c)
    want = np.stack(want)
    check(np_(lg), np_(am), want, "int4", "ragged prefill")
    toks = [int(np.argmax(r)) for r in want]
    for i in range(4):
        refs = np.stack([orc.forward(caches[s], [toks[s]], lens[s] + i)[0] for s in range(4)])
        lg, am = m.decode([([toks[s]], lens[s] + i, tables[s]) for s in range(4)])
        check(np_(lg), np_(am), refs, "int4", f"batched decode {i}")
        toks = [int(np.argmax(r)) for r in refs]
    assert m.device_status() == 0
    m.close()


def test_int4_at_the_qwen3_shape():
    m, orc, w = make_pair("qwen3_0p6b", "int4", max_positions=256, max_tokens=256, max_seqs=2, n_blocks=40)
    prompts = [inputs.make_ids(151936, n, seed=130 + s) for s, n in enumerate([45, 120])]
    tables = [m.blocks_for(n + 4) for n in (45, 120)]
    lg, am = m.prefill([(p, 0, t) for p, t in zip(prompts, tables)], rows=dec.DEC_ROWS_LAST)
    caches, want = [], []
    for p in prompts:
        c = orc.new_cache(256)
        want.append(orc.forward(c, p, 0, rows="last")[-1])
        caches.append(c)
    check(np_(lg), np_(am), np.stack(want), "int4", "0.6B int4 prefill")
    toks = [int(np.argmax(r)) for r in want]
    for i in range(2):
        refs = np.stack([orc.forward(caches[s], [toks[s]], (45, 120)[s] + i)[0] for s in range(2)])
        lg, am = m.decode([([toks[s]], (45, 120)[s] + i, tables[s]) for s in range(2)])
        check(np_(lg), np_(am), refs, "int4", f"0.6B int4 decode {i}")
        toks = [int(np.argmax(r)) for r in refs]
    assert m.device_status() == 0
    m.close()
