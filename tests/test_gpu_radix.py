"""The radix-tree prefix cache end to end on the GPU, in the Trellis session
pattern: a system prompt is warmed into the cache; each session matches its
prompt, starts from the cached blocks (seq_alloc_prefix), appends the rest of
its prompt and decoded tokens through the device append kernel, and some
sessions branch (a fork whose first append copies the shared partial last
block: copy-on-write on top of cached blocks); every decode step runs paged
decode attention over all live sessions; finished sessions are cached,
unlocked and freed, and the cache evicts under pool pressure so that later
sessions reuse blocks that went back to the pool.

Checked against the oracle side -- PoolModel with its own host K/V store and
RadixModel -- bit-exactly on block tables, lengths, refcounts, the free
count, copy-on-write copies, the cache's tree and eviction results, and on
the attention outputs against the fp64 oracle within max-abs 1e-2 and
rel-RMS 5e-3 (lse 1e-3)."""
import random

import numpy as np
import pytest

import oracle
import workloads as W
from _util import check_close, check_lse, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_prefix_shared_decode_gb300 as kvp  # noqa: E402
from paged_prefix_shared_decode_gb300.runner import bf16_tensor  # noqa: E402

L, HQ, HKV, D = 2, 32, 4, 64


class Both:
    """The library (device pool + prefix cache) and the oracle (model pool
    with a host K/V store + radix model), driven in lockstep."""

    def __init__(self, nb, bs, seqs=40, mb=64, seed=5):
        self.bs, self.nb = bs, nb
        shape = (L, nb, HKV, bs, D)
        self.kp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.vp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.pool = kvp.kv_pool_create(kvp.PoolDesc(L, nb, bs, HKV, D, seqs, mb, seed), self.kp, self.vp)
        self.cache = kvp.kvp_radix_create(self.pool)
        store = (np.zeros(shape, np.uint16), np.zeros(shape, np.uint16))
        self.m = oracle.PoolModel(nb, bs, seqs, mb, alloc_seed=seed, store=store)
        self.r = oracle.RadixModel(self.m)
        self.stream = 0      # counter-based K/V streams, one per append
        self.mb = mb

    def close(self):
        kvp.kvp_radix_destroy(self.cache)
        kvp.kv_pool_destroy(self.pool)

    def append(self, seqs, ntoks):
        """One batched device append; the model applies the same appends in order."""
        total = sum(ntoks)
        if total == 0:
            return
        self.stream += 1
        k = W.normal_bf16(77, self.stream, (L, total, HKV, D))
        v = W.normal_bf16(78, self.stream, (L, total, HKV, D))
        kvp.seq_append_batch(self.pool, seqs, ntoks, bf16_tensor(k), bf16_tensor(v))
        off = 0
        for s, n in zip(seqs, ntoks):
            self.m.append(s, n, k[:, off:off + n], v[:, off:off + n])
            off += n

    def same(self):
        assert kvp.kvp_radix_dump(self.cache) == self.r.dump()
        assert kvp.kvp_free_block_count(self.pool) == self.m.free_count()
        assert kvp.kvp_cow_count(self.pool) == self.m.cow_copies
        for b in range(self.nb):
            assert kvp.block_refcount(self.pool, b) == self.m.refcount(b)
        for s in self.m.live():
            assert list(kvp.seq_block_table(self.pool, s)) == self.m.table(s)
            assert kvp.seq_len(self.pool, s) == self.m.length(s)

    def decode(self, seqs, step):
        """Paged decode attention over `seqs` against the fp64 oracle."""
        S = len(seqs)
        t, ln = kvp.kvp_gather_tables(self.pool, seqs, self.mb)
        tm = np.full((S, self.mb), -1, np.int32)
        for i, s in enumerate(seqs):
            tb = self.m.table(s)
            tm[i, :len(tb)] = tb
        assert np.array_equal(t, tm)
        q = W.normal_bf16(79, step, (L, S, HQ, D))
        desc = kvp.AttnDesc(L, HQ, HKV, D, self.bs, self.nb, 0.0, 1)
        ws = torch.empty(kvp.kvp_decode_workspace_size(desc, t, ln), dtype=torch.uint8, device="cuda")
        out = torch.empty((L, S, HQ, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((L, S, HQ), dtype=torch.float32, device="cuda")
        kvp.paged_decode_attention(bf16_tensor(q), self.kp, self.vp, t, ln, desc, out, lse, ws)
        torch.cuda.synchronize()
        assert kvp.kvp_device_error(ws) == 0
        want, want_lse = oracle.decode_attention(q, self.m.store[0], self.m.store[1], tm, ln)
        check_close(to_f64(out), want)
        check_lse(to_f64(lse), want_lse)


@pytest.mark.parametrize("bs,seed", [(16, 0), (32, 1)])
def test_sessions_share_cached_prefix_blocks(bs, seed):
    rng = random.Random(seed)
    # a pool small enough that the cache has to evict before the last sessions
    both = Both(nb=26 if bs == 16 else 24, bs=bs)
    evictions = 0

    def make_room(need):
        # pool pressure: the cache gives back least recently used leaves
        nonlocal evictions
        if both.m.free_count() >= need:
            return
        met_m, freed_m = both.r.evict(need)
        assert kvp.kvp_radix_evict(both.cache, need) == (met_m, freed_m)
        assert met_m
        evictions += freed_m
    sysp = [rng.randrange(32000) for _ in range(5 * bs + 7)]     # 5 whole blocks cached, 7 tokens not
    s0 = both.m.alloc()
    assert kvp.seq_alloc(both.pool) == s0
    both.append([s0], [len(sysp)])
    both.r.insert(sysp, both.m.table(s0))
    kvp.kvp_radix_insert(both.cache, sysp, kvp.seq_block_table(both.pool, s0))
    both.m.free_seq(s0)
    kvp.seq_free(both.pool, s0)
    both.same()

    step = 0
    served = 0
    for wave in range(3):
        live = []        # (seq, tokens so far, lock)
        for i in range(4):
            prompt = sysp + [rng.randrange(32000) for _ in range(rng.randrange(1, 2 * bs))]
            if i == 0 and len(prompt) % bs == 0:   # the branching session ends in a partial block
                prompt.append(rng.randrange(32000))
            got_m, lock_m = both.r.match(prompt)
            got_l, lock_l = kvp.kvp_radix_match(both.cache, prompt)
            assert list(got_l) == got_m and (lock_m is None) == (lock_l == -1)
            served += len(got_m) * bs
            sm = both.m.alloc_prefix(got_m)
            assert kvp.seq_alloc_prefix(both.pool, got_l) == sm
            rest = len(prompt) - len(got_m) * bs
            make_room(rest // bs + 2)
            both.append([sm], [rest])
            live.append([sm, prompt, (lock_m, lock_l)])
        # one session branches: the fork shares the partial last block, and
        # the first append of each copies it (copy-on-write)
        parent = live[0]
        child = both.m.fork(parent[0])
        assert kvp.seq_fork(both.pool, parent[0]) == child
        live.append([child, list(parent[1]), (None, -1)])
        both.same()
        # decode steps: each live session appends its token, then attention
        make_room(2 * len(live))
        for _ in range(3):
            seqs = [x[0] for x in live]
            both.append(seqs, [1] * len(seqs))
            for x in live:
                x[1] = x[1] + [rng.randrange(32000)]
            both.decode(seqs, step)
            step += 1
        both.same()
        assert both.m.cow_copies >= 1
        # sessions end: cached, unlocked, freed
        for sm, toks, (lock_m, lock_l) in live:
            both.r.insert(toks, both.m.table(sm))
            kvp.kvp_radix_insert(both.cache, toks, kvp.seq_block_table(both.pool, sm))
            if lock_m is not None:
                both.r.unlock(lock_m)
                kvp.kvp_radix_unlock(both.cache, lock_l)
            both.m.free_seq(sm)
            kvp.seq_free(both.pool, sm)
        both.same()
    assert served >= 12 * 5 * bs     # every session found the system prompt's whole blocks
    assert evictions > 0             # and the pool ran short at least once
    # drop the whole cache: every block goes back
    met_m, freed_m = both.r.evict(both.nb)
    assert kvp.kvp_radix_evict(both.cache, both.nb) == (met_m, freed_m)
    assert met_m and kvp.kvp_free_block_count(both.pool) == both.nb
    both.same()
    both.close()
