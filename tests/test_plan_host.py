"""The decode planner on the host (no GPU): what it reports through
kvp_decode_plan_stats and the workspace-size calls, checked against values
computed here from the block tables alone.

- unique KV bytes = distinct blocks referenced x their valid tokens x bytes
  per token (a block shared by several sequences has the same valid length
  for every one of them, so it counts once), and with sharing off the sum
  of the sequences' lengths;
- row tiles = ceil(sequences / (64 / G)) on the mma.sync path;
- the plan's shape (items, KV tiles, partial rows) depends on which blocks
  are shared, not on their ids: the same batch built on a differently
  shuffled free list plans the same shape;
- the pool-table and host-table entry points size the same workspace;
- the plan keeps its own invariants (checked inside kvp_decode_plan_stats)
  on both kernels' shapes: head dim 64 (mma.sync only) and head dim 128 with
  many-row items on the tcgen05 kernel, on bf16 and on 4-bit pages."""
import random

import numpy as np
import pytest

import paged_prefix_shared_decode_gb300 as kvp

L, HQ, HKV, D = 2, 32, 4, 64


def fork_batch(seed, alloc_seed, bs, n=24, nb=4096, mb=96):
    """A random fork tree of sequences on a bookkeeping pool: every sequence
    forks an earlier one (or starts fresh) and appends a few tokens."""
    rng = random.Random(seed)
    p = kvp.kv_pool_create(kvp.PoolDesc(L, nb, bs, HKV, D, n + 1, mb, alloc_seed))
    seqs = []
    for i in range(n):
        if seqs and rng.random() < 0.8:
            s = kvp.seq_fork(p, rng.choice(seqs))
        else:
            s = kvp.seq_alloc(p)
        kvp.seq_reserve(p, s, rng.randrange(1, 5 * bs))
        seqs.append(s)
    return p, seqs


def unique_bytes(tables, lens, bs, tok_bytes):
    valid = {}
    for row, n in zip(tables, lens):
        for j in range((n + bs - 1) // bs):
            v = min(bs, n - j * bs)
            assert valid.setdefault(int(row[j]), v) == v   # sharers agree on a block's valid length
    return sum(valid.values()) * tok_bytes


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("seed", range(6))
def test_plan_stats_against_the_tables(bs, seed):
    p, seqs = fork_batch(seed, alloc_seed=seed + 1, bs=bs)
    t, ln = kvp.kvp_gather_tables(p, seqs, 96)
    tok_bytes = 2 * HKV * D * 2 * L
    on = kvp.AttnDesc(L, HQ, HKV, D, bs, 4096, 0.0, 1)
    off = kvp.AttnDesc(L, HQ, HKV, D, bs, 4096, 0.0, 0)
    st = kvp.kvp_decode_plan_stats(on, t, ln)
    assert st["unique_kv_bytes"] == unique_bytes(t, ln, bs, tok_bytes)
    per_tile = 64 // (HQ // HKV)
    assert st["row_tiles"] == -(-len(seqs) // per_tile)
    st0 = kvp.kvp_decode_plan_stats(off, t, ln)
    assert st0["unique_kv_bytes"] == int(ln.sum()) * tok_bytes
    assert st0["row_tiles"] == len(seqs)
    # sharing never reads more tiles than reading every sequence on its own
    assert st["kv_tiles"] <= st0["kv_tiles"]
    assert kvp.kvp_pool_decode_workspace_size(p, seqs, on) == kvp.kvp_decode_workspace_size(on, t, ln)
    # the same batch on another block shuffle: the same plan shape
    q, seqs2 = fork_batch(seed, alloc_seed=seed + 101, bs=bs)
    t2, ln2 = kvp.kvp_gather_tables(q, seqs2, 96)
    assert not np.array_equal(t2, t) and np.array_equal(ln2, ln)
    st2 = kvp.kvp_decode_plan_stats(on, t2, ln2)
    assert st2 == st
    kvp.kv_pool_destroy(p)
    kvp.kv_pool_destroy(q)


def test_plan_is_repeatable_and_rejects_bad_tables():
    p, seqs = fork_batch(3, alloc_seed=2, bs=16)
    t, ln = kvp.kvp_gather_tables(p, seqs, 96)
    d = kvp.AttnDesc(L, HQ, HKV, D, 16, 4096, 0.0, 1)
    assert kvp.kvp_decode_plan_stats(d, t, ln) == kvp.kvp_decode_plan_stats(d, t, ln)
    bad = t.copy()
    bad[0, 0] = 4096            # a block id outside the pool
    with pytest.raises(kvp.KvpError):
        kvp.kvp_decode_plan_stats(d, bad, ln)
    empty = ln.copy()
    empty[1] = 0                # an empty sequence
    with pytest.raises(kvp.KvpError):
        kvp.kvp_decode_plan_stats(d, t, empty)
    kvp.kv_pool_destroy(p)


@pytest.mark.parametrize("kv4", [False, True])
@pytest.mark.parametrize("seed", range(4))
def test_plan_invariants_with_tcgen05_items(seed, kv4):
    # head dim 128, GQA 4: items of more than 32 rows go to the tcgen05
    # kernel, the rest to mma.sync; a wide fork gives both (on bf16 and on
    # 4-bit pages alike)
    rng = random.Random(seed)
    bs, n = 16, 48
    p = kvp.kv_pool_create(kvp.PoolDesc(2, 4096, bs, 8, 128, n + 1, 96, seed + 7))
    root = kvp.seq_alloc(p)
    kvp.seq_reserve(p, root, 700 + seed)
    seqs = []
    for i in range(n):
        s = kvp.seq_fork(p, rng.choice([root] + seqs))
        kvp.seq_reserve(p, s, rng.randrange(1, 3 * bs))
        seqs.append(s)
    t, ln = kvp.kvp_gather_tables(p, seqs, 96)
    fmt = kvp.KVP_KV_4BIT if kv4 else kvp.KVP_KV_BF16
    d = kvp.AttnDesc(2, 32, 8, 128, bs, 4096, 0.0, 1, fmt)
    st = kvp.kvp_decode_plan_stats(d, t, ln)
    per_tok = 2 * 8 * (128 // 2 + 1) * 2 if kv4 else 2 * 8 * 128 * 2 * 2
    assert st["unique_kv_bytes"] == unique_bytes(t, ln, bs, per_tok)
    assert st["row_tiles"] == -(-n // (256 // 4))
    kvp.kv_pool_destroy(p)
