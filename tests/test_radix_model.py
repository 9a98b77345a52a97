"""Pins of the oracle's radix-tree prefix cache ("SGLang RadixAttention",
sections on the node and edge structure, on match / split / insert and on
reference counting with LRU eviction; "Trellis", section "RadixAttention in
Trellis") to the pages' worked examples, to brute force over the inserted
sequences, to a hand-worked eviction order and to block conservation."""
import random

import pytest

from oracle import PoolModel, RadixModel, PoolError


def pool(nb=64, bs=1, seqs=16, mb=64):
    return PoolModel(nb, bs, seqs, mb, alloc_seed=0)


def seq_with(m, tokens):
    """A sequence holding len(tokens) tokens in fresh blocks (block ids in
    allocation order)."""
    s = m.alloc()
    m.append(s, len(tokens))
    return s, m.table(s)


def test_split_example_from_the_page():
    # "SGLang RadixAttention", edge splitting: an edge [A, B, C, D] and a new
    # request [A, B, E, F] give a node [A, B] with children [C, D], [E, F];
    # the blocks are divided by slicing, none is copied.
    A, B, C, D, E, F = 1, 2, 3, 4, 5, 6
    m = pool(bs=1)
    r = RadixModel(m)
    s1, b1 = seq_with(m, [A, B, C, D])
    r.insert([A, B, C, D], b1)
    s2, b2 = seq_with(m, [A, B, E, F])
    r.insert([A, B, E, F], b2)
    assert r.dump() == [(0, (A, B), tuple(b1[:2]), 0, 2),
                        (1, (C, D), tuple(b1[2:]), 0, 1),
                        (1, (E, F), tuple(b2[2:]), 0, 2)]
    # the cache holds one reference on each block it stores; the second
    # sequence's own copies of A, B are not cached
    for b in b1:
        assert m.refcount(b) == 2
    assert [m.refcount(b) for b in b2] == [1, 1, 2, 2]


def test_hello_my_name_is_example_stores_three_entries():
    # "Trellis", section "Prefix caching with RadixAttention": for
    # "hello my name is Alice" and "hello my name is Bob" the tree keeps
    # "hello my name is ", "Alice" and "Bob" (one token per word here).
    words = {"hello": 1, "my": 2, "name": 3, "is": 4, "Alice": 5, "Bob": 6}
    a = [words[w] for w in "hello my name is Alice".split()]
    b = [words[w] for w in "hello my name is Bob".split()]
    m = pool(bs=1)
    r = RadixModel(m)
    for t in (a, b):
        _, blk = seq_with(m, t)
        r.insert(t, blk)
    runs = sorted(d[1] for d in r.dump())
    assert runs == sorted([tuple(a[:4]), (5,), (6,)])


def brute_force_match(inserted, query, bs):
    """Longest prefix of `query` in whole blocks that some inserted sequence
    shares, and for each of those blocks the id the earliest such sequence
    stored it in."""
    nq = len(query) // bs
    best, ids = 0, []
    for j in range(nq):
        owner = None
        for toks, blks in inserted:
            if len(toks) // bs > j and len(blks) > j and toks[:(j + 1) * bs] == query[:(j + 1) * bs]:
                owner = blks[j]
                break
        if owner is None:
            break
        best, ids = j + 1, ids + [owner]
    return best, ids


@pytest.mark.parametrize("bs,seed", [(1, 0), (2, 1), (4, 2), (3, 3)])
def test_match_equals_brute_force(bs, seed):
    rng = random.Random(seed)
    m = PoolModel(4096, bs, 256, 64, alloc_seed=5)
    r = RadixModel(m)
    inserted = []
    base = [rng.randrange(3) for _ in range(12 * bs)]
    for _ in range(40):
        cut = rng.randrange(0, len(base) + 1)
        toks = base[:cut] + [rng.randrange(3) for _ in range(rng.randrange(0, 8 * bs))]
        s, blk = seq_with(m, toks)
        r.insert(toks, blk)
        inserted.append((toks, blk[:len(toks) // bs]))
        for _ in range(3):
            qcut = rng.randrange(0, len(base) + 1)
            q = base[:qcut] + [rng.randrange(3) for _ in range(rng.randrange(0, 8 * bs))]
            got, lock = r.match(q)
            want_n, want_ids = brute_force_match(inserted, q, bs)
            assert got == want_ids and len(got) == want_n
            r.unlock(lock)


def test_lru_leaf_first_eviction_with_cascade():
    # Inserts [1, 2], [1, 3, 4], [1, 3, 5] (bs 1, clock 1, 2, 3) give
    # root -> [1] -> {[2] (last used 1), [3] -> {[4] (2), [5] (3)}}.
    m = pool(nb=10, bs=1)
    r = RadixModel(m)
    blks = []
    for t in ([1, 2], [1, 3, 4], [1, 3, 5]):
        s, blk = seq_with(m, t)
        r.insert(t, blk)
        blks.append(blk)
        m.free_seq(s)                       # only the cache holds blocks now
    assert sorted((d[0], d[1], d[4]) for d in r.dump()) == \
        [(0, (1,), 3), (1, (2,), 1), (1, (3,), 3), (2, (4,), 2), (2, (5,), 3)]
    assert m.free_count() == 5
    # one block at a time, oldest unlocked leaf first: [2], [4], [5]; then
    # [3] is childless and unlocked, then [1] (the cascade up to the root)
    order = []
    for need in range(6, 11):
        assert r.evict(need) == (True, 1)
        order.append(m.free[0])
    assert order == [blks[0][1], blks[1][2], blks[2][2], blks[1][1], blks[0][0]]
    assert r.dump() == [] and m.free_count() == 10


def test_locked_path_is_not_evicted():
    m = pool(nb=6, bs=1)
    r = RadixModel(m)
    s, blk = seq_with(m, [7, 8, 9])
    r.insert([7, 8, 9], blk)
    m.free_seq(s)
    got, lock = r.match([7, 8, 5])           # agrees in part: locks [7, 8, 9]
    assert got == blk[:2]
    assert r.evict(6) == (False, 0)
    r.unlock(lock)
    assert r.evict(6) == (True, 3)
    assert list(m.free)[:3] == blk           # given back last to first
    with pytest.raises(PoolError):
        r.unlock(lock)


def test_split_inherits_locks():
    m = pool(nb=16, bs=1)
    r = RadixModel(m)
    _, blk = seq_with(m, [1, 2, 3, 4])
    r.insert([1, 2, 3, 4], blk)
    _, lock = r.match([1, 2, 3, 4])
    _, blk2 = seq_with(m, [1, 2, 9])
    r.insert([1, 2, 9], blk2)               # splits [1,2,3,4] under the lock
    locks = {d[1]: d[3] for d in r.dump()}
    assert locks == {(1, 2): 1, (3, 4): 1, (9,): 0}
    r.unlock(lock)
    assert all(d[3] == 0 for d in r.dump())


def test_blocks_are_conserved_over_random_traffic():
    # Every reference to a block is a sequence table entry or the cache.
    rng = random.Random(7)
    bs = 2
    m = PoolModel(512, bs, 64, 64, alloc_seed=3)
    r = RadixModel(m)
    live, locks = {}, []
    system = [rng.randrange(50) for _ in range(10 * bs)]
    for step in range(300):
        op = rng.random()
        if op < 0.45 and len(live) < 60:
            q = system[:rng.randrange(0, len(system) + 1)] + [rng.randrange(50) for _ in range(rng.randrange(1, 6 * bs))]
            got, lock = r.match(q)
            locks.append(lock)
            s = m.alloc_prefix(got)
            try:
                m.append(s, len(q) - len(got) * bs)
            except PoolError:
                m.free_seq(s)
                continue
            live[s] = q
        elif op < 0.75 and live:
            s = rng.choice(sorted(live))
            r.insert(live[s], m.table(s))
            m.free_seq(s)
            del live[s]
        elif op < 0.9 and locks:
            r.unlock(locks.pop(rng.randrange(len(locks))))
        else:
            r.evict(rng.randrange(0, 512))
        cached = [b for d in r.dump() for b in d[2]]
        assert len(cached) == len(set(cached))
        for b in range(m.NB):
            want = sum(t.count(b) for t in (m.table(s) for s in live)) + cached.count(b)
            assert m.refcount(b) == want
        assert m.free_count() == sum(1 for b in range(m.NB) if m.refcount(b) == 0)
