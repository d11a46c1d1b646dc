"""The prefix cache end to end: a prompt that starts with a registered prefix
reuses its cached blocks and prefills only its new tokens; its logits match
the oracle and a full prefill of the whole prompt in fresh blocks."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from decoder_qwen3_step_gb300 import dec, inputs  # noqa: E402

from .helpers import TOLS, check, make_pair, np_  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["bf16", "fp32"])
def test_cached_prefix_is_reused(mode):
    m, orc, w = make_pair("small", mode, max_positions=256, max_tokens=512, max_seqs=4, n_blocks=40)
    a = inputs.make_ids(8192, 80, seed=61)                              # 5 full blocks
    b = np.concatenate([a[:64], inputs.make_ids(8192, 30, seed=62)])    # shares a's first 4 blocks
    ta = m.blocks_for(81)
    m.prefill([(a, 0, ta)], rows=dec.DEC_ROWS_LAST)
    torch.cuda.synchronize()
    assert m.register_prefix(ta, a) == 5
    m.release(ta)
    assert m.cached_blocks() == 5
    hit = m.lookup_prefix(b)
    assert hit == ta[:4]                                                # whole blocks, up to the first miss
    assert m.cached_blocks() == 1
    tb = hit + m.alloc(2)
    lg, am = m.prefill([(b[64:], 64, tb)])                              # only the new tokens
    ref = orc.forward(orc.new_cache(128), b, 0)[64:]
    check(np_(lg), np_(am), ref, mode, "prefill on a cached prefix")
    # the whole prompt in fresh blocks: the 30 new tokens alone run on the
    # few-token product kernels, the 94 tokens on the many-token ones, so in the
    # serving mode the two agree to the serving tolerance (bf16/f16 roundings of
    # another summation order), in the parity mode to fp32 rounding
    tf = m.blocks_for(95)
    lf, _ = m.prefill([(b, 0, tf)])
    tol = 1e-4 if mode == "fp32" else TOLS[mode]
    assert np.abs(np_(lf)[64:] - np_(lg)).max() <= tol
    for t in (tb, tf):
        m.release(t)
    assert m.device_status() == 0
    m.close()
