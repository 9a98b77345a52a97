"""The library's pool bookkeeping (C++) against the oracle model (Python):
bit-exact block tables, lengths, refcounts, free-list state, slot mapping and
copy-on-write decisions over seeded random op traces and the workloads."""
import numpy as np
import pytest

import oracle
import paged_prefix_shared_decode_gb300 as kvp
import workloads as W


def lib_pool(w, seed):
    s = w.shapes
    return kvp.kv_pool_create(kvp.PoolDesc(s.L, w.num_blocks, s.bs, s.Hkv, s.d, w.max_seqs,
                                           w.max_blocks_per_seq, seed))


def compare(model, p, ids_m, ids_l):
    assert kvp.kvp_free_block_count(p) == model.free_count()
    for nm in ids_m:
        sm, sl = ids_m[nm], ids_l[nm]
        assert sm == sl
        assert list(kvp.seq_block_table(p, sl)) == model.table(sm)
        assert kvp.seq_len(p, sl) == model.length(sm)
    for b in range(model.NB):
        assert kvp.block_refcount(p, b) == model.refcount(b)
    assert kvp.kvp_cow_count(p) == model.cow_copies


@pytest.mark.parametrize("seed,bs,alloc_seed", [(1, 16, 1), (2, 32, 7), (3, 4, 0), (4, 16, 99)])
def test_random_trace_bit_exact(seed, bs, alloc_seed):
    w = W.random_trace(seed, 10_000 if seed == 1 else 3000, bs=bs)
    m = oracle.PoolModel(w.num_blocks, bs, w.max_seqs, w.max_blocks_per_seq, alloc_seed)
    p = lib_pool(w, alloc_seed)
    ids_m, ids_l = {}, {}
    for i, op in enumerate(w.ops):
        if op[0] == "alloc":
            ids_m[op[1]] = m.alloc(); ids_l[op[1]] = kvp.seq_alloc(p)
        elif op[0] == "fork":
            ids_m[op[2]] = m.fork(ids_m[op[1]]); ids_l[op[2]] = kvp.seq_fork(p, ids_l[op[1]])
        elif op[0] == "append":
            sm = m.append(ids_m[op[1]], op[2])
            cow_before = m.cow_copies
            slots, cow = kvp.seq_reserve(p, ids_l[op[1]], op[2])
            assert [b * bs + s for b, s in sm] == list(slots)
        elif op[0] == "free":
            m.free_seq(ids_m.pop(op[1])); kvp.seq_free(p, ids_l.pop(op[1]))
        if i % 500 == 0:
            compare(m, p, ids_m, ids_l)
    compare(m, p, ids_m, ids_l)
    for nm in list(ids_m):
        m.free_seq(ids_m.pop(nm)); kvp.seq_free(p, ids_l.pop(nm))
    compare(m, p, ids_m, ids_l)
    assert kvp.kvp_free_block_count(p) == w.num_blocks
    kvp.kv_pool_destroy(p)


def test_cow_triple_matches_model():
    m = oracle.PoolModel(64, 16, 8, 32, 3)
    p = kvp.kv_pool_create(kvp.PoolDesc(1, 64, 16, 1, 8, 8, 32, 3))
    a = m.alloc(); b = kvp.seq_alloc(p)
    m.append(a, 250); kvp.seq_reserve(p, b, 250)
    ca, cb = m.fork(a), kvp.seq_fork(p, b)
    last = m.table(a)[-1]
    m.append(ca, 3)
    slots, cow = kvp.seq_reserve(p, cb, 3)
    assert cow[0] == last and cow[1] == m.table(ca)[-1] and cow[2] == 250 % 16
    assert list(slots) == [m.table(ca)[-1] * 16 + 10 + i for i in range(3)]
    _, cow2 = kvp.seq_reserve(p, b, 1)        # parent now alone: in place
    assert cow2[0] == -1
    kvp.kv_pool_destroy(p)


@pytest.mark.parametrize("make", [W.tiny_fork, lambda: W.dendrite(layers=1),
                                  lambda: W.trellis(0.5, layers=1), lambda: W.mcts(layers=1),
                                  lambda: W.verify_tree(8, layers=1)])
def test_workloads_bit_exact(make):
    w = make()
    for seed in (0, 1):
        rw = oracle.replay(w, alloc_seed=seed, with_store=False)
        p = lib_pool(w, seed)
        ids = {}
        for op in w.ops:
            if op[0] == "alloc":
                ids[op[1]] = kvp.seq_alloc(p)
            elif op[0] == "fork":
                ids[op[2]] = kvp.seq_fork(p, ids[op[1]])
            elif op[0] == "append":
                kvp.seq_reserve(p, ids[op[1]], op[2])
        compare(rw.model, p, rw.ids, ids)
        kvp.kv_pool_destroy(p)


def test_errors_and_all_or_nothing():
    p = kvp.kv_pool_create(kvp.PoolDesc(1, 4, 16, 1, 8, 2, 3, 0))
    s = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s, 40)
    with pytest.raises(kvp.KvpError) as e:
        kvp.seq_reserve(p, s, 40)             # table capacity 3 blocks
    assert e.value.code == kvp.KVP_ERR_INVALID
    t = kvp.seq_alloc(p)
    with pytest.raises(kvp.KvpError) as e:
        kvp.seq_reserve(p, t, 17)              # 2 blocks, 1 free
    assert e.value.code == kvp.KVP_ERR_OOM
    assert kvp.seq_len(p, t) == 0 and kvp.kvp_free_block_count(p) == 1
    with pytest.raises(kvp.KvpError):
        kvp.seq_alloc(p)                       # max_seqs 2
    kvp.seq_free(p, s)
    with pytest.raises(kvp.KvpError):
        kvp.seq_free(p, s)                     # double free
    with pytest.raises(kvp.KvpError):
        kvp.seq_fork(p, 5)
    with pytest.raises(kvp.KvpError):
        kvp.block_refcount(p, 4)
    kvp.kv_pool_destroy(p)


def test_fork_latency_is_microseconds():
    import time
    w = W.dendrite(layers=1)
    p = lib_pool(w, 1)
    s = kvp.seq_alloc(p)
    kvp.seq_reserve(p, s, 4096)
    lib = kvp.load()
    import ctypes
    c = ctypes.c_int32()
    n = 2000
    t0 = time.perf_counter()
    for _ in range(n):
        lib.seq_fork(p, s, ctypes.byref(c))
        lib.seq_free(p, c.value)
    dt = (time.perf_counter() - t0) / n
    assert dt < 200e-6      # generous: ctypes overhead included
    kvp.kv_pool_destroy(p)
