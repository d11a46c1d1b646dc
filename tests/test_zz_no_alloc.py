"""dec_attend_noalloc: decode attention for callers that cannot allocate
device memory when they need it (code inside a framework that owns every
device allocation, plug-ins with a fixed memory budget, latency-critical
loops that must not touch the allocator).  Its scratch is an array inside
the library, so the only buffers a caller passes are inputs and outputs.

Checked through the C ABI against dec_attend (the same kernel with caller
scratch) on two calls in a row, within the tolerance of test_gpu_attend;
the second call also shows that what the first left in the shared array does
not leak into the result.  A repeated call leaves the device's free memory
and torch's allocation count unchanged (it allocates nothing), and the
array's error word reads 0 after good calls.  This file is named to be
collected last."""

import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec  # noqa: E402

from .helpers import make_pair  # noqa: E402
from .test_gpu_attend import fill_cache, run_attend  # noqa: E402

pytestmark = pytest.mark.gpu


def noalloc_status(m):
    v = C.c_uint32(0xFFFFFFFF)
    s = torch.cuda.current_stream()
    dec.check(m.L.dec_attend_noalloc_status(C.c_void_p(s.cuda_stream), C.byref(v)), "dec_attend_noalloc_status")
    return v.value


def run_noalloc(m, layer, q, ctxs, tables, out):
    S = len(ctxs)
    max_blocks = max(len(t) for t in tables)
    tab = np.zeros((S, max_blocks), dtype=np.int32)
    for i, t in enumerate(tables):
        tab[i, :len(t)] = t
    ctx = np.asarray(ctxs, dtype=np.int32)
    s = torch.cuda.current_stream()
    dec.check(m.L.dec_attend_noalloc(m.pool, layer, S, C.c_void_p(q.data_ptr()),
                                     ctx.ctypes.data_as(C.POINTER(C.c_int32)),
                                     tab.ctypes.data_as(C.POINTER(C.c_int32)), max_blocks,
                                     C.c_void_p(out.data_ptr()), C.c_void_p(s.cuda_stream)), "dec_attend_noalloc")
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_noalloc_attention_matches_dec_attend_twice(mode):
    m, _, _ = make_pair("small", mode, max_positions=1024, max_tokens=64, max_seqs=8, n_blocks=300)
    s = m.shape
    H, D = s["n_heads"], s["head_dim"]
    rng = np.random.default_rng(31)
    ot = torch.float32 if mode == "fp32" else torch.bfloat16
    tol = 1e-5 if mode == "fp32" else 1e-2
    layer = 2
    calls = [([5, 130, 600], layer), ([1, 256, 33, 900], layer + 1)]  # different shapes: stale scratch is ignored
    for ctxs, lay in calls:
        tables = [m.blocks_for(n) for n in ctxs]
        fill_cache(m, tables, ctxs, lay, rng)
        q = torch.from_numpy(rng.standard_normal((len(ctxs), H, D)).astype(np.float32)).to(m.device)
        want = torch.empty((len(ctxs), H * D), dtype=ot, device=m.device)
        got = torch.full((len(ctxs), H * D), float("nan"), dtype=ot, device=m.device)
        run_attend(m, lay, q, ctxs, tables, want)
        run_noalloc(m, lay, q, ctxs, tables, got)
        w, g = want.float().cpu().numpy(), got.float().cpu().numpy()
        assert np.isfinite(g).all()
        assert np.abs(g - w).max() <= tol * max(1.0, np.abs(w).max())
        assert noalloc_status(m) == 0
        # the same call again: no device memory taken, by the driver's count or torch's
        torch.cuda.synchronize()
        free0, allocated0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        run_noalloc(m, lay, q, ctxs, tables, got)
        free1, allocated1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        assert (free1, allocated1) == (free0, allocated0)
        assert np.array_equal(got.float().cpu().numpy(), g)
        for t in tables:
            m.release(t)
    # beyond the fixed scratch (256 sequences x 1,024 keys: 8.7 MB): refused with a message,
    # nothing launched; the sequences share one allocated table
    big = [1024] * 256
    shared = m.blocks_for(1024)
    tables = [shared] * len(big)
    q = torch.zeros((len(big), H, D), dtype=torch.float32, device=m.device)
    out = torch.empty((len(big), H * D), dtype=ot, device=m.device)
    with pytest.raises(dec.DecError) as e:
        run_noalloc(m, layer, q, big, tables, out)
    assert e.value.code == dec.DEC_ERANGE and "scratch" in str(e.value)
    m.release(shared)
    m.close()
