"""Speculative accept after tree verify: the library's bookkeeping (C++,
`seq_accept_draft` on a pool without K/V storage) against the oracle pool
model, bit-exact on kept paths, tables, lengths, refcounts, free lists and
copy-on-write counts, over random draft trees with forked siblings; and the
argument checks.  Host only (the device moves are compared in
tests/test_gpu_accept.py)."""
import numpy as np
import pytest

import oracle
import paged_prefix_shared_decode_gb300 as kvp


def make(nb, bs, seqs=32, mb=64, seed=5):
    m = oracle.PoolModel(nb, bs, seqs, mb, alloc_seed=seed)
    p = kvp.kv_pool_create(kvp.PoolDesc(1, nb, bs, 1, 64, seqs, mb, seed))
    return m, p


def same(m, p, ids):
    assert kvp.kvp_free_block_count(p) == m.free_count()
    assert kvp.kvp_cow_count(p) == m.cow_copies
    for s in ids:
        assert list(kvp.seq_block_table(p, s)) == m.table(s)
        assert kvp.seq_len(p, s) == m.length(s)
    for b in range(m.NB):
        assert kvp.block_refcount(p, b) == m.refcount(b)


@pytest.mark.parametrize("bs,seed", [(16, 1), (4, 2), (1, 3), (32, 4)])
def test_random_accepts_bit_exact(bs, seed):
    rng = np.random.default_rng(seed)
    m, p = make(2048, bs, mb=264 // bs + 2)
    live = []
    for trial in range(60):
        # a sequence with a context and a draft; sometimes a forked sibling
        # shares every block
        ctx, n = int(rng.integers(0, 200)), int(rng.integers(1, 65))
        s = m.alloc()
        assert kvp.seq_alloc(p) == s
        m.append(s, ctx + n)
        kvp.seq_reserve(p, s, ctx + n)
        live.append(s)
        if rng.random() < 0.4:
            c = m.fork(s)
            assert kvp.seq_fork(p, s) == c
            live.append(c)
        parent = [-1] + [int(rng.integers(-1, i)) for i in range(1, n)]
        a = int(rng.integers(-1, n))
        path_m = m.accept_draft(s, ctx, parent, a)
        path_l = kvp.seq_accept_draft(p, s, ctx, parent, a, stream=0)
        assert list(path_l) == path_m
        same(m, p, live)
        while len(live) > 12:
            x = live.pop(int(rng.integers(0, len(live))))
            m.free_seq(x)
            kvp.seq_free(p, x)
    same(m, p, live)
    kvp.kv_pool_destroy(p)


def test_bad_arguments_change_nothing():
    m, p = make(64, 4)
    s = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s, 15)
    t0, n0 = list(kvp.seq_block_table(p, s)), kvp.seq_len(p, s)
    for ctx, parent, a in [(6, [-1, 0, 5, 0, 0, 0, 0, 0, 0], 2),   # a parent after its child
                           (5, [-1] * 9, 0),                        # draft does not end the sequence
                           (6, [-1] * 9, 9),                        # accepted node out of range
                           (6, [-2] * 9, 0)]:                       # parent below -1
        with pytest.raises(kvp.KvpError) as e:
            kvp.seq_accept_draft(p, s, ctx, parent, a, stream=0)
        assert e.value.code == kvp.KVP_ERR_INVALID
        assert list(kvp.seq_block_table(p, s)) == t0 and kvp.seq_len(p, s) == n0
    # more than 64 draft tokens
    s2 = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s2, 70)
    with pytest.raises(kvp.KvpError):
        kvp.seq_accept_draft(p, s2, 0, [-1] * 70, 3, stream=0)
    kvp.kv_pool_destroy(p)


def test_copy_on_write_needs_a_free_block():
    # every block in use: the copy a shared block needs cannot be made
    m, p = make(4, 4)
    s = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s, 16)
    c = kvp.seq_fork(p, s)
    with pytest.raises(kvp.KvpError) as e:
        kvp.seq_accept_draft(p, s, 8, [-1] * 8, 7, stream=0)    # token 15 -> 8: block 2 written
    assert e.value.code == kvp.KVP_ERR_OOM
    assert kvp.seq_len(p, s) == 16 and kvp.block_refcount(p, kvp.seq_block_table(p, s)[2]) == 2
    kvp.kv_pool_destroy(p)
