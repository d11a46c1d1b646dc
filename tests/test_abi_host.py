"""The C ABI without a GPU: the library loads, exports every declared symbol,
and its host-side logic (config checks, sizes, the block pool, KV addressing)
behaves as the pages specify.  No call here launches device work."""

import ctypes as C
import os
import re

import pytest

from decoder_qwen3_step_gb300 import dec, inputs
from decoder_qwen3_step_gb300.runtime import make_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(dec.LIB_PATH):
        from decoder_qwen3_step_gb300 import build

        build.build()
    return dec.lib()


def cfg(name="qwen3_0p6b", mode=dec.DEC_BF16_F16KV, max_positions=4224):
    return make_config(inputs.SHAPES[name], mode, max_positions)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(names) == set(dec.EXPORTS)
    for n in names:
        assert hasattr(L, n), n
    assert b"sm_103a" in L.dec_version()


def test_config_accepts_the_qwen3_shape_and_refuses_what_it_cannot_run(L):
    c = cfg()
    assert L.dec_config_check(C.byref(c)) == dec.DEC_OK
    for field, val in [("rope_scaling", 1), ("sliding_window", 4096), ("attention_bias", 1), ("qk_norm", 0),
                       ("rope_split", 0), ("tied", 0), ("n_kv_heads", 3), ("head_dim", 96), ("block_tokens", 8),
                       ("vocab", 0), ("mode", 7), ("rms_eps", 0.0)]:
        bad = cfg()
        setattr(bad, field, val)
        assert L.dec_config_check(C.byref(bad)) == dec.DEC_EINVAL, field
        assert L.dec_last_error()


def test_packed_weight_and_workspace_sizes(L):
    sz = C.c_size_t()
    c = cfg()
    assert L.dec_weights_bytes(C.byref(c), C.byref(sz)) == 0
    # 596,049,920 parameters: matrices in bf16, gains in fp32, plus the fp32 RoPE table
    matrices = 596049920 - 28 * (2 * 1024 + 2 * 128) - 1024
    rope = 4224 * 64 * 2 * 4
    assert matrices * 2 + rope <= sz.value <= matrices * 2 + rope + 28 * 12 * 256 + 4 * 256 + 2 ** 20
    assert L.dec_workspace_bytes(C.byref(c), 4096, 32, C.byref(sz)) == 0
    assert L.dec_workspace_bytes(C.byref(c), 0, 1, C.byref(sz)) == dec.DEC_EINVAL


def _pool(L, n_blocks, name="tiny"):
    c = cfg(name, dec.DEC_FP32, 64)
    sz = C.c_size_t()
    assert L.dec_pool_bytes(C.byref(c), n_blocks, C.byref(sz)) == 0
    p = C.c_void_p()
    # Host-only bookkeeping: the slab address is never dereferenced on the host.
    fake = C.c_void_p(1 << 40)
    assert L.dec_pool_create(C.byref(c), n_blocks, fake, sz.value, C.byref(p)) == 0
    return c, p, sz.value


def test_pool_rejects_zero_capacity(L):
    c = cfg("tiny", dec.DEC_FP32, 64)
    sz = C.c_size_t()
    assert L.dec_pool_bytes(C.byref(c), 0, C.byref(sz)) == dec.DEC_EINVAL
    p = C.c_void_p()
    assert L.dec_pool_create(C.byref(c), 0, C.c_void_p(1 << 40), 1 << 20, C.byref(p)) == dec.DEC_EINVAL


def test_pool_bytes_match_the_slab_layout(L):
    c, p, size = _pool(L, 10)
    s = inputs.SHAPES["tiny"]
    assert size == 10 * s["n_layers"] * 2 * s["n_kv_heads"] * 16 * s["head_dim"] * 4
    L.dec_pool_destroy(p)


def test_pool_lifecycle_all_or_nothing_and_refcounts(L):
    c, p, _ = _pool(L, 6)
    n = C.c_int32()
    ids = (C.c_int32 * 8)()
    assert L.dec_pool_alloc(p, 4, ids) == 0
    got = list(ids[:4])
    assert len(set(got)) == 4 and all(0 <= i < 6 for i in got)
    L.dec_pool_free_blocks(p, C.byref(n))
    assert n.value == 2
    assert L.dec_pool_alloc(p, 3, ids) == dec.DEC_ECAPACITY  # all or nothing
    L.dec_pool_free_blocks(p, C.byref(n))
    assert n.value == 2
    assert L.dec_pool_retain(p, got[0]) == 0
    r = C.c_int32()
    L.dec_pool_refcount(p, got[0], C.byref(r))
    assert r.value == 2
    assert L.dec_pool_release(p, got[0]) == 0
    assert L.dec_pool_release(p, got[0]) == 0
    L.dec_pool_free_blocks(p, C.byref(n))
    assert n.value == 3
    assert L.dec_pool_release(p, got[0]) == dec.DEC_EBLOCK  # already free
    assert L.dec_pool_retain(p, 99) == dec.DEC_EBLOCK
    assert L.dec_pool_release(p, -1) == dec.DEC_EBLOCK
    for i in got[1:]:
        assert L.dec_pool_release(p, i) == 0
    L.dec_pool_free_blocks(p, C.byref(n))
    assert n.value == 6
    L.dec_pool_destroy(p)


def test_kv_offset_follows_the_worked_block_address_example(L):
    g = {}
    with open(os.path.join(GOLDEN, "block_address.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, *v = ln.split()
                g[k] = [int(x) for x in v]
    assert g["block_tokens"] == [16]
    c, p, _ = _pool(L, 12)
    s = inputs.SHAPES["tiny"]
    D, Hkv, nl = s["head_dim"], s["n_kv_heads"], s["n_layers"]
    table = (C.c_int32 * 3)(*g["table"])
    pos = g["position"][0]
    blk, slot = g["pool_block"][0], g["slot"][0]
    assert table[g["table_index"][0]] == blk and pos % 16 == slot
    off = C.c_int64()
    for layer in range(nl):
        for h in range(Hkv):
            for is_v in (0, 1):
                assert L.dec_kv_offset(p, table, 3, pos, layer, h, is_v, C.byref(off)) == 0
                slab = ((layer * 12 + blk) * 2 + is_v) * Hkv * 16 * D
                assert off.value == slab + (h * 16 + slot) * D
    assert L.dec_kv_offset(p, table, 3, 48, 0, 0, 0, C.byref(off)) == dec.DEC_ERANGE  # table too short
    bad = (C.c_int32 * 3)(7, 2, 12)
    assert L.dec_kv_offset(p, bad, 3, 37, 0, 0, 0, C.byref(off)) == dec.DEC_EBLOCK
    L.dec_pool_destroy(p)


def test_release_build_has_no_debug_hooks(L):
    """The release library reports no build options and refuses the debug
    build's table-poisoning hook; the DEC_DEBUG build adds -DDEC_DEBUG to every
    translation unit and links libdec_debug.so beside libdec.so."""
    from decoder_qwen3_step_gb300 import build

    if os.environ.get("DEC_DEBUG") != "1":
        assert L.dec_build_flags() == 0
    assert L.dec_debug_poison_table(None, 0, 0, 0) == dec.DEC_EINVAL
    assert "-DDEC_DEBUG" in build._flags(debug=True) and "-DDEC_DEBUG" not in build._flags()
    assert build.LIB_DEBUG != build.LIB and build.BUILD_DEBUG != build.BUILD


def test_debug_build_compiles_and_reports_its_flag():
    """The DEC_DEBUG build (device bounds checks behind #ifdef) compiles for
    sm_103a and exports the same symbols; loaded in a child process it reports
    DEC_BUILD_DEBUG.  No device work runs."""
    import subprocess
    import sys

    from decoder_qwen3_step_gb300 import build

    lib = build.build(debug=True)
    assert os.path.exists(lib) and lib.endswith("libdec_debug.so")
    code = ("from decoder_qwen3_step_gb300 import dec; L = dec.lib(); "
            "assert dec.LIB_PATH.endswith('libdec_debug.so'); "
            "assert L.dec_build_flags() == dec.DEC_BUILD_DEBUG; "
            "assert all(hasattr(L, n) for n in dec.EXPORTS); print('ok')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env={**os.environ, "DEC_DEBUG": "1"},
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stderr[-2000:]
