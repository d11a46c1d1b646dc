"""Host marshalling of a step (runtime.Batch) without a GPU: the decode fast
path (one token per sequence) and the general path give the same arrays, and
block tables given as Python lists or int32 arrays give the same table."""

import numpy as np
import pytest

pytest.importorskip("torch")

from decoder_qwen3_step_gb300.runtime import Batch  # noqa: E402


def _general(seqs):
    """The step's arrays built the plain way, element by element."""
    ids, pos, start, rows = [], [], [0], []
    mb = max(1, max(len(t) for _, _, t in seqs))
    for toks, p0, table in seqs:
        ids += [int(x) for x in toks]
        pos += list(range(p0, p0 + len(toks)))
        start.append(len(ids))
        rows.append([int(x) for x in table] + [0] * (mb - len(table)))
    return ids, pos, start, rows, mb


@pytest.mark.parametrize("as_array", [False, True])
def test_decode_fast_path_matches_the_plain_arrays(as_array):
    rng = np.random.default_rng(5)
    seqs = []
    for s in range(32):
        n = int(rng.integers(1, 150))
        table = rng.integers(0, 5000, n).astype(np.int32)
        seqs.append(([int(rng.integers(0, 151936))], int(rng.integers(0, 2400)), table if as_array else table.tolist()))
    b = Batch(seqs)
    ids, pos, start, rows, mb = _general(seqs)
    assert b.n_seqs == 32 and b.n_tokens == 32 and b.max_blocks == mb
    assert b.ids.dtype == np.int32 and b.ids.tolist() == ids
    assert b.positions.tolist() == pos and b.seq_start.tolist() == start
    assert b.tables.dtype == np.int32 and b.tables.tolist() == rows and b.tables.flags["C_CONTIGUOUS"]
    assert b.struct.n_seqs == 32 and b.struct.n_tokens == 32 and b.struct.max_blocks == mb


def test_multi_token_steps_keep_the_general_path():
    seqs = [([1, 2, 3], 10, [7, 8]), ([4], 0, np.array([9], dtype=np.int32)), ([5, 6], 3, [])]
    b = Batch(seqs)
    ids, pos, start, rows, mb = _general(seqs)
    assert b.ids.tolist() == ids and b.positions.tolist() == pos and b.seq_start.tolist() == start
    assert b.tables.tolist() == rows and b.n_tokens == 6 and b.max_blocks == mb
