"""The library's host side of the sampler, without a GPU: its PCG32 stream
helpers against the oracle's generator (same states, same outputs, the
pages' worked value), and the symbols of the sampler boundary."""

import ctypes as C

import pytest

from decoder_qwen3_step_gb300 import dec
from oracle import sampler as S


@pytest.fixture(scope="module")
def L():
    return dec.lib()


def test_child_seed_and_streams_match_the_oracle(L):
    assert L.dec_child_seed(C.c_uint64(0), C.c_uint64(4)) == 0xF88BB8A8724C81EC  # the pages' worked value
    for seed in (0, 1, 42, 2**63 + 5, 2**64 - 1):
        for purpose in (0, 4, 9):
            assert L.dec_child_seed(C.c_uint64(seed), C.c_uint64(purpose)) == S.child_seed(seed, purpose)
            r = dec.dec_rng()
            L.dec_rng_stream(C.c_uint64(seed), C.c_uint64(purpose), C.byref(r))
            o = S.stream(seed, purpose)
            assert (r.state, r.inc) == o.snapshot()
            for _ in range(5):
                assert L.dec_rng_next_u32(C.byref(r)) == o.next_u32()
            for _ in range(5):
                assert L.dec_rng_uniform(C.byref(r)) == o.uniform_f64()
            assert (r.state, r.inc) == o.snapshot()


def test_first_uniform_of_the_worked_example(L):
    r = dec.dec_rng()
    L.dec_rng_stream(C.c_uint64(0), C.c_uint64(dec.DEC_PURPOSE_SAMPLE), C.byref(r))
    assert round(L.dec_rng_uniform(C.byref(r)), 5) == 0.80209


def test_workspace_sizes_and_refusals(L):
    n = C.c_size_t()
    assert L.dec_sampler_workspace_bytes(151936, 32, C.byref(n)) == dec.DEC_OK
    assert n.value >= 151936 * 32 * 22  # marks 4, key 8, e' 8, bucket 2 bytes per id and row
    assert L.dec_sampler_workspace_bytes(0, 1, C.byref(n)) == dec.DEC_EINVAL
    assert L.dec_sampler_workspace_bytes(2**20 + 1, 1, C.byref(n)) == dec.DEC_EINVAL
    assert L.dec_sampler_workspace_bytes(1000, 0, C.byref(n)) == dec.DEC_EINVAL
    h = C.c_void_p()
    assert L.dec_sampler_create(1000, 1, None, 0, C.byref(h)) == dec.DEC_EINVAL  # refused before any device call
