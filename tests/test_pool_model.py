"""Pins of the oracle's bookkeeping model (block pool, fork, copy-on-write,
free) to the pages' worked numbers, closed-form block counts and invariants."""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import PoolModel, PoolError, initial_free_list, splitmix64_stream
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_splitmix64_reference_vectors():
    for row in _golden_rows("splitmix64.txt"):
        g = splitmix64_stream(int(row[0]))
        assert [next(g) for _ in range(3)] == [int(x, 16) for x in row[1:]]


def test_free_list_is_a_permutation_and_seed0_is_identity():
    assert initial_free_list(50, 0) == list(range(50))
    p = initial_free_list(1000, 1)
    assert sorted(p) == list(range(1000)) and p != list(range(1000))
    assert initial_free_list(1000, 2) != p


def test_dendrite_api_example_fork_twice_shares_every_block():
    # "allocate a parent, fork two children": fork copies table pointers only.
    m = PoolModel(64, 16, 8, 16, alloc_seed=1)
    parent = m.alloc()
    m.append(parent, 100)
    free_before = m.free_count()
    c1, c2 = m.fork(parent), m.fork(parent)
    assert m.free_count() == free_before          # no KV block allocated
    assert m.table(c1) == m.table(parent) == m.table(c2)
    assert all(m.refcount(b) == 3 for b in m.table(parent))
    assert m.length(c1) == 100


def test_copy_on_write_of_a_shared_partial_block():
    # prefix 250 = 15 full blocks + 10 tokens; two children both append.
    m = PoolModel(64, 16, 8, 32, alloc_seed=3)
    p = m.alloc(); m.append(p, 250)
    a, b = m.fork(p), m.fork(p)
    last = m.table(p)[-1]
    assert m.refcount(last) == 3
    m.append(a, 1)
    assert m.cow_copies == 1 and m.table(a)[-1] != last and m.refcount(last) == 2
    assert m.table(a)[:-1] == m.table(p)[:-1]
    m.append(b, 30)          # 6 into the copy, 24 spill into 2 new blocks
    assert m.cow_copies == 2 and m.refcount(last) == 1
    assert len(m.table(b)) == 18
    m.append(p, 1)           # the parent now holds its block alone: in place
    assert m.cow_copies == 2 and m.table(p)[-1] == last
    # a full last block is never copied
    q = m.alloc(); m.append(q, 32); r = m.fork(q); m.append(r, 1)
    assert m.cow_copies == 2 and m.table(r)[:2] == m.table(q)


def test_cow_copies_used_slots_in_the_store():
    L, NB, Hkv, bs, d = 2, 16, 2, 4, 3
    kp = np.zeros((L, NB, Hkv, bs, d), np.uint16); vp = np.zeros_like(kp)
    m = PoolModel(NB, bs, 4, 8, alloc_seed=5, store=(kp, vp))
    p = m.alloc()
    k = np.arange(L * 6 * Hkv * d, dtype=np.uint16).reshape(L, 6, Hkv, d)
    m.append(p, 6, k, k + 1000)
    c = m.fork(p)
    k2 = np.full((L, 1, Hkv, d), 7, np.uint16)
    m.append(c, 1, k2, k2)
    old, new = m.table(p)[1], m.table(c)[1]
    assert old != new
    assert np.array_equal(kp[:, new, :, :2], kp[:, old, :, :2])
    assert np.array_equal(kp[:, new, :, 2], k2[:, 0])
    assert np.array_equal(vp[:, old, :, :2], (k + 1000)[:, 4:6].transpose(0, 2, 1, 3))


def test_errors_leave_state_unchanged():
    m = PoolModel(4, 16, 2, 3, alloc_seed=0)
    s = m.alloc()
    m.append(s, 40)
    with pytest.raises(PoolError) as e:
        m.append(s, 40)                  # needs 3 more blocks, only 1 free
    assert e.value.kind in ("oom", "invalid")
    assert m.length(s) == 40 and m.free_count() == 1
    m.alloc()
    with pytest.raises(PoolError):
        m.alloc()                        # max_seqs = 2
    with pytest.raises(PoolError):
        m.fork(7)
    m.free_seq(s)
    with pytest.raises(PoolError):
        m.free_seq(s)                    # double free
    with pytest.raises(PoolError):
        m.append(s, 1)


def test_refcounts_return_to_zero_after_free():
    w = W.random_trace(7, 3000)
    rw = oracle.replay(w, alloc_seed=9, with_store=False)
    m = rw.model
    # refcount == number of live tables holding the block
    held = np.zeros(m.NB, int)
    for s in m.live():
        for b in set(m.table(s)):
            held[b] += 1
    assert list(held) == m.ref
    assert m.free_count() + int((held > 0).sum()) == m.NB
    for s in m.live():
        m.free_seq(s)
    assert all(r == 0 for r in m.ref) and m.free_count() == m.NB
    assert sorted(m.free) == list(range(m.NB))


def test_lowest_free_sequence_id_is_reused():
    m = PoolModel(8, 4, 4, 4)
    a, b, c = m.alloc(), m.alloc(), m.alloc()
    m.free_seq(b)
    assert m.alloc() == b


# ------------------------------------------------------ workload block counts

def _blocks_in_use(rw):
    return rw.model.NB - rw.model.free_count()


def test_tiny_fork_block_count():
    rw = oracle.replay(W.tiny_fork(), with_store=False)
    assert _blocks_in_use(rw) == 16 + 4 * 2


def test_dendrite_block_count_and_sharing():
    w = W.dendrite()
    rw = oracle.replay(w, with_store=False)
    priv = w.info["private"]
    assert _blocks_in_use(rw) == 256 + sum(math.ceil(u / 16) for u in priv)
    root = rw.model.table(rw.ids[0])
    assert all(rw.model.refcount(b) == 7 for b in root)   # parent + 6 branches


def test_trellis_golden_block_counts_strictly_decrease():
    rows = [r for r in _golden_rows("trellis_prefix_blocks.txt") if r[0] != "hit_rate_cap"]
    cap = [r for r in _golden_rows("trellis_prefix_blocks.txt") if r[0] == "hit_rate_cap"][0]
    assert abs(float(cap[1]) - (512 / 32 - 1) / (512 / 32)) < 1e-15
    counts = []
    for phi, p, realised, blocks in rows:
        w = W.trellis(float(phi), layers=1)
        assert w.info["prefix_blocks"] == int(p)
        assert abs(w.info["realised_phi"] - float(realised)) < 1e-12
        rw = oracle.replay(w, with_store=False)
        # the timed step appends the 64th decode token: replay it too
        for nm in w.batch:
            rw.model.append(rw.ids[nm], 1)
        used = _blocks_in_use(rw)
        assert used == int(blocks)
        assert all(rw.model.length(rw.ids[nm]) == 576 for nm in w.batch)
        counts.append(used)
    assert all(a > b for a, b in zip(counts, counts[1:]))


def test_mcts_block_count_and_root_refcount():
    w = W.mcts(layers=1)
    rw = oracle.replay(w, with_store=False)
    assert _blocks_in_use(rw) == 128 + 340 * 4
    root = rw.model.table(rw.ids[0])
    assert all(rw.model.refcount(b) == 1 + 4 + 16 + 64 + 256 for b in root)
    leaf = rw.model.table(rw.ids[w.batch[0]])
    assert len(leaf) == 128 + 4 * 4 and rw.model.refcount(leaf[-1]) == 1
    assert rw.model.cow_copies == 0


def test_verify_block_count():
    for B in (1, 8):
        w = W.verify_tree(B, layers=1)
        rw = oracle.replay(w, with_store=False)
        assert _blocks_in_use(rw) == B * 132
        par = w.info["parents"]
        assert par.shape == (B, 64) and (par[:, 0] == -1).all()
        assert all(par[b, i] < i for b in range(B) for i in range(1, 64))


def test_draft_tree_depth_at_most_8():
    for s in range(5):
        par = W.draft_tree(s)
        depth = np.zeros(64, int)
        for i in range(64):
            depth[i] = 1 if par[i] < 0 else depth[par[i]] + 1
        assert depth.max() <= 8 and depth.max() >= 4


def test_alloc_seed_changes_ids_not_results():
    """Outputs are unchanged under a permutation of physical block ids, and a
    forked child with no private tokens reproduces its parent's output."""
    w = W.tiny_fork()
    w.ops += [("fork", 1, 9)]
    names = [1, 2, 3, 4, 9]
    res = []
    for seed in (0, 1, 12345):
        rw = oracle.replay(w, alloc_seed=seed)
        t, ln = rw.tables(names, w.max_blocks_per_seq)
        q = W.step_q(w, 0)
        qq = np.concatenate([q, q[:, :1]], axis=1)      # child 9 gets 1's query
        out, lse = oracle.decode_attention(qq, rw.k_pool, rw.v_pool, t, ln)
        res.append((t, out, lse))
    assert not np.array_equal(res[0][0], res[1][0])
    for t, out, lse in res[1:]:
        np.testing.assert_array_equal(out, res[0][1])
        np.testing.assert_array_equal(lse, res[0][2])
    np.testing.assert_array_equal(res[0][1][:, 4], res[0][1][:, 0])


# -- speculative accept after tree verify ("CAST", section on speculative
#    decoding: the target model accepts one path of the draft tree)

def _draft_pool(bs=4, ctx=6, n=9, seed=1, L=2, Hkv=2, d=3, NB=40):
    kp = np.zeros((L, NB, Hkv, bs, d), np.uint16)
    vp = np.zeros_like(kp)
    m = PoolModel(NB, bs, 8, 64, alloc_seed=seed, store=(kp, vp))
    s = m.alloc()
    tot = ctx + n
    k = (np.arange(L * tot * Hkv * d, dtype=np.uint16) + 1).reshape(L, tot, Hkv, d)
    m.append(s, tot, k, k + 5000)
    return m, s, kp, vp


def _rows(m, kp, s, lo, hi):
    bs = m.bs
    t = m.table(s)
    return np.stack([kp[:, t[p // bs], :, p % bs, :] for p in range(lo, hi)], 1)


def test_accept_on_a_chain_keeps_the_first_tokens_in_place():
    m, s, kp, vp = _draft_pool()
    before = _rows(m, kp, s, 0, 15)
    free0 = m.free_count()
    path = m.accept_draft(s, 6, [-1, 0, 1, 2, 3, 4, 5, 6, 7], 3)
    assert path == [0, 1, 2, 3]
    assert m.length(s) == 10 and len(m.table(s)) == 3
    assert m.free_count() == free0 + 1          # 15 -> 10 tokens: 4 -> 3 blocks
    assert np.array_equal(_rows(m, kp, s, 0, 10), before[:, :10])


def test_accept_on_a_star_moves_one_token():
    m, s, kp, vp = _draft_pool()
    before_k, before_v = _rows(m, kp, s, 0, 15), _rows(m, vp, s, 0, 15)
    path = m.accept_draft(s, 6, [-1] * 9, 5)
    assert path == [5] and m.length(s) == 7
    assert np.array_equal(_rows(m, kp, s, 0, 6), before_k[:, :6])
    assert np.array_equal(_rows(m, kp, s, 6, 7)[:, 0], before_k[:, 6 + 5])
    assert np.array_equal(_rows(m, vp, s, 6, 7)[:, 0], before_v[:, 6 + 5])


def test_accept_none_drops_the_draft():
    m, s, kp, vp = _draft_pool()
    assert m.accept_draft(s, 6, [-1, 0, 0, 1, 1, 2, 2, 3, 3], -1) == []
    assert m.length(s) == 6 and len(m.table(s)) == 2


def test_accept_random_trees_against_brute_force():
    rng = np.random.default_rng(4)
    for trial in range(40):
        bs = int(rng.choice([1, 2, 4, 16]))
        ctx, n = int(rng.integers(0, 20)), int(rng.integers(1, 20))
        m, s, kp, vp = _draft_pool(bs=bs, ctx=ctx, n=n, NB=200, seed=trial)
        parent = [-1] + [int(rng.integers(-1, i)) for i in range(1, n)]
        a = int(rng.integers(-1, n))
        before = _rows(m, kp, s, 0, ctx + n)
        # ancestors-or-self of a, found by marking rather than walking
        anc = set()
        for j in range(n):
            x = a
            while x > j:
                x = parent[x]
            if x == j and a >= 0:
                anc.add(j)
        path = m.accept_draft(s, ctx, parent, a)
        assert path == sorted(anc)
        assert m.length(s) == ctx + len(path)
        assert len(m.table(s)) == -(-(ctx + len(path)) // bs)
        got = _rows(m, kp, s, 0, ctx + len(path))
        want = np.concatenate([before[:, :ctx], before[:, [ctx + j for j in path]]], 1)
        assert np.array_equal(got, want)
        assert m.free_count() == sum(1 for b in range(m.NB) if m.refcount(b) == 0)


def test_accept_copies_a_shared_block_before_moving_into_it():
    m, s, kp, vp = _draft_pool(bs=4, ctx=6, n=9)
    sib = m.fork(s)                              # every block shared
    sib_before = _rows(m, kp, sib, 0, 15)
    cow0 = m.cow_copies
    path = m.accept_draft(s, 6, [-1] * 9, 8)     # token 14 moves to 6: block 1 written
    assert path == [8] and m.cow_copies == cow0 + 1
    assert m.table(s)[0] == m.table(sib)[0] and m.table(s)[1] != m.table(sib)[1]
    assert np.array_equal(_rows(m, kp, sib, 0, 15), sib_before)
    assert np.array_equal(_rows(m, kp, s, 6, 7)[:, 0], sib_before[:, 14])
    for b in range(m.NB):
        want = sum(m.table(x).count(b) for x in m.live())
        assert m.refcount(b) == want


def test_accept_rejects_bad_input_without_change():
    m, s, kp, vp = _draft_pool()
    t0, n0 = m.table(s), m.length(s)
    for ctx, parent, a in [(6, [-1, 0, 5, 0, 0, 0, 0, 0, 0], 2),   # parent after child
                           (5, [-1] * 9, 0),                        # draft region mismatch
                           (6, [-1] * 9, 9)]:                       # node out of range
        with pytest.raises(PoolError):
            m.accept_draft(s, ctx, parent, a)
        assert m.table(s) == t0 and m.length(s) == n0
