"""The DEC_DEBUG build: device bounds checks on every block-table read.

The test builds libdec_debug.so and runs a child process that loads it
(DEC_DEBUG=1).  Valid steps match the oracle with a clean error word (the
checks have no false positives); then a table entry past the pool, planted in
the device copy only after the host validated the real table, reaches the
prefill kernels, the one-kernel decode step and the per-operation decode
kernels: each step ends with DEC_DEV_BOUNDS set, no fault, and the context
stays usable (a fresh decoder in the same process matches the oracle)."""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import numpy as np
    from decoder_qwen3_step_gb300 import dec, inputs
    from tests.helpers import check, make_pair, np_

    L = dec.lib()
    assert dec.LIB_PATH.endswith("libdec_debug.so") and L.dec_build_flags() & dec.DEC_BUILD_DEBUG

    def run(m, orc, prompts, steps, poison=None):
        tables = [m.blocks_for(len(p) + steps + 1) for p in prompts]
        caches = [orc.new_cache(len(p) + steps + 1) for p in prompts]
        if poison == "prefill":
            dec.check(L.dec_debug_poison_table(m.handle, 1, 1, m.n_blocks + 3), "poison")
        m.prefill([(p, 0, t) for p, t in zip(prompts, tables)], rows=dec.DEC_ROWS_LAST)
        if poison == "prefill":
            assert m.device_status() & dec.DEC_DEV_BOUNDS
            return
        toks = [int(np.argmax(orc.forward(c, p, 0, rows="last")[-1])) for c, p in zip(caches, prompts)]
        for i in range(steps):
            pos = [len(p) + i for p in prompts]
            if poison == "decode":  # the block this step writes, for sequence 0
                dec.check(L.dec_debug_poison_table(m.handle, 0, pos[0] // 16, m.n_blocks + 3), "poison")
            lg, am = m.decode([([toks[s]], pos[s], tables[s]) for s in range(len(prompts))])
            if poison == "decode":
                assert m.device_status() & dec.DEC_DEV_BOUNDS
                continue
            refs = np.stack([orc.forward(caches[s], [toks[s]], pos[s])[0] for s in range(len(prompts))])
            check(np_(lg), np_(am), refs, "bf16", f"debug build step {i}")
            assert m.device_status() == 0
            toks = [int(np.argmax(r)) for r in refs]

    for shape, lens in (("tiny", [21, 40]), ("small", [70, 129])):
        V = inputs.SHAPES[shape]["vocab"]
        prompts = [inputs.make_ids(V, n, seed=150 + s) for s, n in enumerate(lens)]
        m, orc, w = make_pair(shape, "bf16", max_positions=256, max_tokens=512, max_seqs=4, n_blocks=64)
        run(m, orc, prompts, 3)                       # clean: parity, no bounds bit
        run(m, orc, prompts, 1, poison="prefill")
        for mega in (True, False):
            m.set_megakernel(mega)
            run(m, orc, prompts, 2, poison="decode")
        m.close()
        m, orc, w = make_pair(shape, "bf16", max_positions=256, max_tokens=512, max_seqs=4, n_blocks=64, weights=w)
        run(m, orc, prompts, 2)                       # the context is still good
        m.close()
    print("debug build ok")
""")


def test_debug_build_bounds_checks_fire_without_a_fault():
    from decoder_qwen3_step_gb300 import build

    build.build(debug=True)
    env = {**os.environ, "DEC_DEBUG": "1"}
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "debug build ok" in r.stdout, (r.stdout[-3000:], r.stderr[-3000:])
