"""dec_attend: the split-K decode attention alone, through the C ABI, against
float64 attention over the very same cached keys and values (written into the
pool's slabs by the test, at the addresses dec_kv_offset gives)."""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402
from oracle.model import attention_one  # noqa: E402

from .helpers import make_pair  # noqa: E402

pytestmark = pytest.mark.gpu


def fill_cache(m, tables, ctxs, layer, rng):
    """Random K/V for positions 0..ctx-1 of each sequence; returns float64 copies."""
    s = m.shape
    Hkv, D = s["n_kv_heads"], s["head_dim"]
    kt = torch.float16 if m.mode == dec.DEC_BF16_F16KV else torch.float32
    slab = m.slabs.view(kt)
    ks, vs = [], []
    for tab, n in zip(tables, ctxs):
        k = rng.standard_normal((n, Hkv, D)).astype(np.float32)
        v = rng.standard_normal((n, Hkv, D)).astype(np.float32)
        kk = torch.from_numpy(k).to(kt)
        vv = torch.from_numpy(v).to(kt)
        tarr = (C.c_int32 * len(tab))(*tab)
        off = C.c_int64()
        for p in range(n):
            for h in range(Hkv):
                for is_v, src in ((0, kk), (1, vv)):
                    dec.check(m.L.dec_kv_offset(m.pool, tarr, len(tab), p, layer, h, is_v, C.byref(off)), "offset")
                    slab[off.value:off.value + D] = src[p, h].to(m.device)
        ks.append(kk.double().numpy())
        vs.append(vv.double().numpy())
    return ks, vs


def run_attend(m, layer, q, ctxs, tables, out, scratch=None):
    S = len(ctxs)
    max_blocks = max(len(t) for t in tables)
    tab = np.zeros((S, max_blocks), dtype=np.int32)
    for i, t in enumerate(tables):
        tab[i, :len(t)] = t
    ctx = np.asarray(ctxs, dtype=np.int32)
    if scratch is None:
        sz = C.c_size_t()
        dec.check(m.L.dec_attend_scratch_bytes(C.byref(m.cfg), S, int(ctx.max()), max_blocks, C.byref(sz)), "bytes")
        scratch = torch.empty(sz.value, dtype=torch.uint8, device=m.device)
    s = torch.cuda.current_stream()
    dec.check(m.L.dec_attend(m.pool, layer, S, C.c_void_p(q.data_ptr()), ctx.ctypes.data_as(C.POINTER(C.c_int32)),
                             tab.ctypes.data_as(C.POINTER(C.c_int32)), max_blocks, C.c_void_p(out.data_ptr()),
                             C.c_void_p(scratch.data_ptr()), scratch.numel(), C.c_void_p(s.cuda_stream)),
              "dec_attend")
    torch.cuda.synchronize()
    return scratch


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_attend_matches_float64_attention(mode):
    m, _, _ = make_pair("small", mode, max_positions=1024, max_tokens=64, max_seqs=8, n_blocks=300)
    s = m.shape
    H, Hkv, D = s["n_heads"], s["n_kv_heads"], s["head_dim"]
    rng = np.random.default_rng(21)
    ctxs = [1, 17, 128, 129, 300, 777]  # one key, ragged blocks, exact chunk, chunk + 1, several chunks
    tables = [m.blocks_for(n) for n in ctxs]
    layer = 3
    ks, vs = fill_cache(m, tables, ctxs, layer, rng)
    q = rng.standard_normal((len(ctxs), H, D)).astype(np.float32)
    qt = torch.from_numpy(q).to(m.device)
    ot = torch.float32 if mode == "fp32" else torch.bfloat16
    out = torch.full((len(ctxs), H * D), float("nan"), dtype=ot, device=m.device)
    scratch = run_attend(m, layer, qt, ctxs, tables, out)
    got = out.float().cpu().numpy().reshape(len(ctxs), H, D).astype(np.float64)
    tol = 1e-5 if mode == "fp32" else 1e-2
    for i, n in enumerate(ctxs):
        for h in range(H):
            g = h * Hkv // H
            ref = attention_one(q[i, h].astype(np.float64), ks[i][:, g], vs[i][:, g])
            assert np.abs(got[i, h] - ref).max() <= tol * max(1.0, np.abs(ref).max()), (i, h)
    err = np.frombuffer(scratch[:4].cpu().numpy().tobytes(), dtype=np.uint32)[0]
    assert err == 0
    # refusals: a block not allocated, a context past the table
    with pytest.raises(dec.DecError):
        run_attend(m, layer, qt, [40], [[m.n_blocks + 5, 0, 0]], out)
    with pytest.raises(dec.DecError):
        run_attend(m, layer, qt, [40], [tables[0][:1]], out)
    m.close()
