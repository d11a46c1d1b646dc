"""The prefix cache of the paged KV pool, host side (no GPU): full blocks
register under a key, release caches a registered block, lookup reacquires
it, allocation stays all-or-nothing and evicts the oldest cached block first,
and references balance (the KvPool boundary tests of tinyllm L10.1: pool
bounds and cache lifecycle, eviction of the oldest cached block)."""

import ctypes as C

import pytest

from decoder_qwen3_step_gb300 import dec

from .test_abi_host import L, _pool  # noqa: F401  (fixture)

B = 16


def key_of(L, prev, toks):  # noqa: F811
    arr = (C.c_int32 * max(len(toks), 1))(*toks)
    return L.dec_prefix_key(C.c_uint64(prev), arr, len(toks))


def fnv1a(prev, toks):
    """The documented definition, written out: FNV-1a 64 over prev's 8 bytes, then each token's 4 bytes (LE)."""
    h = 0xCBF29CE484222325
    data = prev.to_bytes(8, "little") + b"".join((t & 0xFFFFFFFF).to_bytes(4, "little") for t in toks)
    for byte in data:
        h = ((h ^ byte) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def counts(L, p):  # noqa: F811
    n, c = C.c_int32(), C.c_int32()
    L.dec_pool_free_blocks(p, C.byref(n))
    L.dec_pool_cached_blocks(p, C.byref(c))
    return n.value, c.value


def refs(L, p, i):  # noqa: F811
    r = C.c_int32()
    L.dec_pool_refcount(p, i, C.byref(r))
    return r.value


def alloc(L, p, n):  # noqa: F811
    ids = (C.c_int32 * max(n, 1))()
    rc = L.dec_pool_alloc(p, n, ids)
    return rc, list(ids[:n])


def register(L, p, i, key):  # noqa: F811
    ok = C.c_int32()
    rc = L.dec_pool_register(p, i, C.c_uint64(key), C.byref(ok))
    return rc, ok.value


def lookup(L, p, key):  # noqa: F811
    i = C.c_int32()
    assert L.dec_pool_lookup(p, C.c_uint64(key), C.byref(i)) == 0
    return i.value


def test_prefix_key_is_the_documented_chain(L):  # noqa: F811
    toks = [1, 2, 70000, -1, 151935]
    assert key_of(L, 0, toks) == fnv1a(0, toks)
    k1 = key_of(L, 0, list(range(B)))
    k2 = key_of(L, k1, list(range(B, 2 * B)))
    assert k2 == fnv1a(k1, list(range(B, 2 * B)))
    assert key_of(L, 0, list(range(B))) != key_of(L, 1, list(range(B)))  # the chain matters
    assert key_of(L, 0, [5, 6]) != key_of(L, 0, [6, 5])


def test_full_blocks_register_release_caches_lookup_reacquires(L):  # noqa: F811
    c, p, _ = _pool(L, 4)
    rc, (a, b) = alloc(L, p, 2)
    assert rc == 0
    assert register(L, p, a, 111)[0] == dec.DEC_EINVAL  # not full yet
    assert L.dec_pool_set_fill(p, a, B + 1) == dec.DEC_EINVAL
    assert L.dec_pool_set_fill(p, a, B) == 0
    assert register(L, p, a, 111) == (0, 1)
    assert L.dec_pool_set_fill(p, b, B) == 0
    assert register(L, p, b, 111) == (0, 0)  # the key keeps its first block
    assert L.dec_pool_release(p, a) == 0
    assert refs(L, p, a) == 0 and counts(L, p) == (2, 1)  # cached, not free
    assert L.dec_pool_retain(p, a) == dec.DEC_EBLOCK  # a cached block is reacquired by lookup only
    assert lookup(L, p, 111) == a and refs(L, p, a) == 1 and counts(L, p) == (2, 0)
    assert lookup(L, p, 111) == a and refs(L, p, a) == 2  # a block in use is shared
    assert lookup(L, p, 222) == -1
    for i in (a, a, b):
        assert L.dec_pool_release(p, i) == 0
    assert counts(L, p) == (3, 1)  # b was never registered: free; a cached
    assert L.dec_pool_release(p, b) == dec.DEC_EBLOCK  # refs never go negative
    L.dec_pool_destroy(p)


def test_allocation_is_all_or_nothing_and_evicts_the_oldest_cached_block(L):  # noqa: F811
    c, p, _ = _pool(L, 4)
    rc, ids = alloc(L, p, 4)
    keys = [1000 + i for i in range(4)]
    for i, k in zip(ids, keys):
        assert L.dec_pool_set_fill(p, i, B) == 0 and register(L, p, i, k) == (0, 1)
    order = [ids[2], ids[0], ids[3]]  # release order: oldest first
    for i in order:
        assert L.dec_pool_release(p, i) == 0
    assert counts(L, p) == (0, 3)
    assert alloc(L, p, 4)[0] == dec.DEC_ECAPACITY  # 3 available: nothing taken, nothing evicted
    assert counts(L, p) == (0, 3)
    rc, got = alloc(L, p, 2)
    assert rc == 0 and sorted(got) == sorted(order[:2])  # the two oldest releases
    assert lookup(L, p, keys[2]) == -1 and lookup(L, p, keys[0]) == -1  # their keys are gone
    assert lookup(L, p, keys[3]) == ids[3]  # the newest stays cached and comes back
    assert counts(L, p) == (0, 0)
    for i in got + [ids[3], ids[1]]:
        assert L.dec_pool_release(p, i) == 0
    # ids[3] and ids[1] are still registered: back to the cache; the reused two are free
    assert counts(L, p) == (2, 2)
    L.dec_pool_destroy(p)


def test_reregistering_a_block_moves_its_key(L):  # noqa: F811
    c, p, _ = _pool(L, 2)
    rc, (a,) = alloc(L, p, 1)
    assert L.dec_pool_set_fill(p, a, B) == 0
    assert register(L, p, a, 7) == (0, 1)
    assert register(L, p, a, 8) == (0, 1)
    assert lookup(L, p, 7) == -1 and lookup(L, p, 8) == a
    L.dec_pool_destroy(p)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_lifecycles_keep_the_pool_invariants(L, seed):  # noqa: F811
    """Random alloc / register / retain / lookup / release sequences against a
    plain Python model of the pool: same answers, refs never negative, every
    block exactly one of in use, cached or free."""
    import random

    rng = random.Random(seed)
    N = 8
    c, p, _ = _pool(L, N)
    ref = [0] * N
    key = {}        # block -> key it is registered under
    index = {}      # key -> block
    lru = []        # cached blocks, oldest first
    free = [N - 1 - i for i in range(N)]  # stack: top is the next id
    for _ in range(400):
        op = rng.randrange(5)
        live = [i for i in range(N) if ref[i] > 0]
        if op == 0:
            n = rng.randrange(0, 4)
            rc, got = alloc(L, p, n)
            if n > len(free) + len(lru):
                assert rc == dec.DEC_ECAPACITY
                continue
            assert rc == 0
            while len(free) < n:
                b = lru.pop(0)
                del index[key.pop(b)]
                free.insert(0, b)
            want = [free.pop() for _ in range(n)]
            assert got == want
            for b in got:
                ref[b] = 1
        elif op == 1 and live:
            b = rng.choice(live)
            k = rng.randrange(6)
            assert L.dec_pool_set_fill(p, b, B) == 0
            rc, ok = register(L, p, b, k)
            assert rc == 0
            if k in index:
                assert ok == (index[k] == b)
            else:
                if b in key:
                    del index[key[b]]
                index[k] = b
                key[b] = k
                assert ok == 1
        elif op == 2 and live:
            b = rng.choice(live)
            assert L.dec_pool_retain(p, b) == 0
            ref[b] += 1
        elif op == 3:
            k = rng.randrange(6)
            got = lookup(L, p, k)
            if k in index:
                b = index[k]
                assert got == b
                if ref[b] == 0:
                    lru.remove(b)
                ref[b] += 1
            else:
                assert got == -1
        elif op == 4 and live:
            b = rng.choice(live)
            assert L.dec_pool_release(p, b) == 0
            ref[b] -= 1
            if ref[b] == 0:
                (lru if b in key else free).append(b)
        for b in range(N):
            assert refs(L, p, b) == ref[b] >= 0
        assert counts(L, p) == (len(free), len(lru))
        assert sorted(free + lru + [b for b in range(N) if ref[b] > 0]) == list(range(N))
    L.dec_pool_destroy(p)


def batch(seqs, vocab_ok=True):  # noqa: F811
    """A dec_batch (and the host arrays it points at) from [(ids, first position, table)]."""
    ids, pos, start, tab = [], [], [0], []
    mb = max(len(t) for _, _, t in seqs)
    for toks, p0, table in seqs:
        ids += list(toks)
        pos += list(range(p0, p0 + len(toks)))
        start.append(len(ids))
        tab += list(table) + [0] * (mb - len(table))
    arr = lambda v: (C.c_int32 * len(v))(*v)  # noqa: E731
    keep = (arr(ids), arr(pos), arr(start), arr(tab))
    b = dec.dec_batch(len(seqs), len(ids), keep[0], None, keep[1], keep[2], keep[3], mb)
    return b, keep


def check(L, p, seqs, decode=0):  # noqa: F811
    b, _keep = batch(seqs)
    return L.dec_batch_check(p, C.byref(b), decode)


def test_step_check_refuses_writes_into_shared_or_cached_blocks(L):  # noqa: F811
    """A step writes K/V only into blocks its sequence owns alone: a block
    shared after retain or lookup, or indexed in the prefix cache, is refused
    (DEC_EBLOCK) before anything runs, so a scheduler's mistake cannot
    overwrite another sequence's cache or a cached prefix."""
    _c, p, _ = _pool(L, 16)
    rc, blk = alloc(L, p, 3)
    assert rc == 0
    toks = list(range(1, 17))
    # a clean prefill of 20 tokens into blocks 0 and 1 of the table passes
    assert check(L, p, [(list(range(20)), 0, blk[:2])]) == 0
    # sharing the block the step writes (refcount 2) is refused ...
    assert L.dec_pool_retain(p, blk[1]) == 0
    assert check(L, p, [([7], 20, blk[:2])]) == dec.DEC_EBLOCK
    assert "shared" in L.dec_last_error().decode()
    # ... while reading a shared block is fine: the step writes only block 2
    assert check(L, p, [([7], 32, [blk[0], blk[1], blk[2]])]) == 0
    assert L.dec_pool_release(p, blk[1]) == 0
    # a full block registered in the prefix index may be read, never written
    assert L.dec_pool_set_fill(p, blk[0], B) == 0
    assert register(L, p, blk[0], key_of(L, 0, toks)) == (0, 1)
    assert check(L, p, [(toks, 0, blk[:1])]) == dec.DEC_EBLOCK
    assert check(L, p, [([3], 16, blk[:2])]) == 0
    # two sequences (or two positions) that would write the same block are refused
    assert check(L, p, [([3], 17, blk[:2]), ([4], 20, [blk[2], blk[1]])]) == dec.DEC_EBLOCK
    assert "two positions" in L.dec_last_error().decode()
    assert check(L, p, [(list(range(20)), 16, [blk[0], blk[1], blk[1]])]) == dec.DEC_EBLOCK
    # the remaining checks still hold: unallocated block, short table, decode shape
    assert check(L, p, [([3], 16, [blk[0], 15])]) == dec.DEC_EBLOCK
    assert check(L, p, [([3], 40, blk[:2])]) == dec.DEC_ERANGE
    assert check(L, p, [([3, 4], 16, blk[:2])], decode=1) == dec.DEC_EINVAL
    L.dec_pool_destroy(p)
