"""The library's radix-tree prefix cache (C++) against the oracle model
(Python): bit-exact trees (runs, blocks, locks, last-use stamps), match
results, block tables, refcounts and eviction outcomes over seeded agentic
traffic (a shared system prompt, per-session suffixes, branching), plus the
C ABI's error behaviour.  Host only."""
import random

import numpy as np
import pytest

import oracle
import paged_prefix_shared_decode_gb300 as kvp


def make(nb, bs, seqs=64, mb=64, seed=3):
    m = oracle.PoolModel(nb, bs, seqs, mb, alloc_seed=seed)
    p = kvp.kv_pool_create(kvp.PoolDesc(1, nb, bs, 1, 64, seqs, mb, seed))
    return m, oracle.RadixModel(m), p, kvp.kvp_radix_create(p)


def same_state(m, r, p, c, live):
    assert kvp.kvp_radix_dump(c) == r.dump()
    assert kvp.kvp_free_block_count(p) == m.free_count()
    for b in range(m.NB):
        assert kvp.block_refcount(p, b) == m.refcount(b)
    for sm, sl in live.values():
        assert list(kvp.seq_block_table(p, sl)) == m.table(sm)
        assert kvp.seq_len(p, sl) == m.length(sm)


@pytest.mark.parametrize("bs,seed,steps", [(16, 1, 600), (1, 2, 400), (4, 3, 400), (32, 4, 300)])
def test_agentic_traffic_bit_exact(bs, seed, steps):
    rng = random.Random(seed)
    nb = 4096
    m, r, p, c = make(nb, bs)
    system = [rng.randrange(1000) for _ in range(rng.randrange(4, 12) * bs + rng.randrange(bs))]
    branches = [system + [rng.randrange(1000) for _ in range(rng.randrange(1, 5) * bs)] for _ in range(4)]
    live, locks = {}, []          # name -> (model seq, lib seq), [(model lock, lib lock)]
    name = 0
    for step in range(steps):
        op = rng.random()
        if op < 0.4 and len(live) < 48:
            base = rng.choice([system, *branches, []])
            q = base[:rng.randrange(0, len(base) + 1)] + [rng.randrange(1000) for _ in range(rng.randrange(1, 4 * bs))]
            got_m, lock_m = r.match(q)
            got_l, lock_l = kvp.kvp_radix_match(c, q)
            assert list(got_l) == got_m
            assert (lock_m is None) == (lock_l == -1)
            locks.append((lock_m, lock_l))
            sm = m.alloc_prefix(got_m)
            sl = kvp.seq_alloc_prefix(p, got_l)
            assert sm == sl
            extra = len(q) - len(got_m) * bs
            try:
                m.append(sm, extra)
            except oracle.PoolError:
                with pytest.raises(kvp.KvpError):
                    kvp.seq_reserve(p, sl, extra)
                m.free_seq(sm)
                kvp.seq_free(p, sl)
                continue
            kvp.seq_reserve(p, sl, extra)
            live[name] = (sm, sl, q)
            name += 1
        elif op < 0.55 and live:
            # a session continues: append a few tokens
            k = rng.choice(sorted(live))
            sm, sl, q = live[k]
            n = rng.randrange(1, 2 * bs + 1)
            try:
                m.append(sm, n)
            except oracle.PoolError:
                continue
            kvp.seq_reserve(p, sl, n)
            live[k] = (sm, sl, q + [rng.randrange(1000) for _ in range(n)])
        elif op < 0.75 and live:
            # a session ends: cache it, then free it
            k = rng.choice(sorted(live))
            sm, sl, q = live.pop(k)
            r.insert(q, m.table(sm))
            kvp.kvp_radix_insert(c, q, kvp.seq_block_table(p, sl))
            m.free_seq(sm)
            kvp.seq_free(p, sl)
        elif op < 0.9 and locks:
            lm, ll = locks.pop(rng.randrange(len(locks)))
            if lm is not None:
                r.unlock(lm)
            kvp.kvp_radix_unlock(c, ll)
        else:
            need = rng.randrange(m.free_count(), nb + 1)
            assert kvp.kvp_radix_evict(c, need) == r.evict(need)
        if step % 25 == 0:
            same_state(m, r, p, c, {k: v[:2] for k, v in live.items()})
    same_state(m, r, p, c, {k: v[:2] for k, v in live.items()})
    kvp.kvp_radix_destroy(c)
    for sm, sl, _ in live.values():
        kvp.seq_free(p, sl)
    assert kvp.kvp_free_block_count(p) == nb
    kvp.kv_pool_destroy(p)


def test_page_split_example_through_the_library():
    A, B, C, D, E, F = 1, 2, 3, 4, 5, 6
    m, r, p, c = make(64, 1)
    for t in ([A, B, C, D], [A, B, E, F]):
        s = kvp.seq_alloc(p)
        kvp.seq_reserve(p, s, len(t))
        sm = m.alloc()
        m.append(sm, len(t))
        kvp.kvp_radix_insert(c, t, kvp.seq_block_table(p, s))
        r.insert(t, m.table(sm))
    d = kvp.kvp_radix_dump(c)
    assert [x[1] for x in d] == [(A, B), (C, D), (E, F)] and [x[0] for x in d] == [0, 1, 1]
    assert d == r.dump()
    kvp.kvp_radix_destroy(c)
    kvp.kv_pool_destroy(p)


def test_errors_change_nothing():
    m, r, p, c = make(32, 4)
    s = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s, 12)
    blocks = kvp.seq_block_table(p, s)
    kvp.kvp_radix_insert(c, list(range(12)), blocks)
    before = kvp.kvp_radix_dump(c)
    free_blk = next(b for b in range(32) if kvp.block_refcount(p, b) == 0)
    # a block that is not in use cannot be cached or start a sequence
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_radix_insert(c, list(range(100, 108)), [blocks[0], free_blk])
    assert e.value.code == kvp.KVP_ERR_INVALID
    with pytest.raises(kvp.KvpError):
        kvp.seq_alloc_prefix(p, [free_blk])
    assert kvp.kvp_radix_dump(c) == before
    # unlocking a path that is not locked
    _, lock = kvp.kvp_radix_match(c, list(range(8)))
    kvp.kvp_radix_unlock(c, lock)
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_radix_unlock(c, lock)
    assert e.value.code == kvp.KVP_ERR_STATE
    kvp.kvp_radix_unlock(c, -1)
    # everything locked: eviction reports that it could not free enough
    _, lock = kvp.kvp_radix_match(c, list(range(12)))
    kvp.seq_free(p, s)
    assert kvp.kvp_radix_evict(c, 32) == (False, 0)
    kvp.kvp_radix_unlock(c, lock)
    assert kvp.kvp_radix_evict(c, 32) == (True, 3)
    kvp.kvp_radix_destroy(c)
    kvp.kv_pool_destroy(p)


def test_match_and_insert_take_microseconds():
    # host cost of the cache on a 4096-token system prompt shared by 256
    # sessions, bs 16 (an agentic setting, synthetic tokens)
    rng = np.random.default_rng(0)
    bs, nb = 16, 8192
    p = kvp.kv_pool_create(kvp.PoolDesc(1, nb, bs, 1, 64, 300, 512, 1))
    c = kvp.kvp_radix_create(p)
    system = rng.integers(0, 32000, 4096).tolist()
    s = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s, len(system))
    kvp.kvp_radix_insert(c, system, kvp.seq_block_table(p, s))
    kvp.seq_free(p, s)
    import time
    t0 = time.perf_counter()
    for i in range(256):
        q = system + rng.integers(0, 32000, 64).tolist()
        got, lock = kvp.kvp_radix_match(c, q)
        assert len(got) == 4096 // bs
        kvp.kvp_radix_unlock(c, lock)
    dt = (time.perf_counter() - t0) / 256
    assert dt < 2e-3, dt
    kvp.kvp_radix_destroy(c)
    kvp.kv_pool_destroy(p)
