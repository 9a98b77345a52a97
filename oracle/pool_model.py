"""Oracle bookkeeping model of the block-paged KV pool (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this.
It is written from the pages' description and the allocation policy stated
below; it shares no code with the library.

What it models:
  * a pool of NB fixed-size token blocks with a free list and per-block
    refcounts ("Dendrite", section details: paged cache of 16-token blocks, a
    tree-shaped KV cache with reference counting, no duplicate allocation of a
    shared prefix; "Trellis", section "RadixAttention in Trellis": a session
    holds an ordered list of block ids and *acquires* shared prefix blocks by
    bumping their refcount instead of allocating);
  * fork: the child gets a copy of the parent's block table and every block's
    refcount goes up by one; no KV bytes move ("Dendrite", section details:
    copy-on-write fork copies block-table pointers, not data);
  * append with copy-on-write: writing into a partial last block that other
    live sequences also hold first gives the writer its own copy of that
    block (the used slots are copied); a full last block just gets a new
    block; a block held only by the writer is written in place;
  * free: every block's refcount goes down by one and a block whose count
    reaches zero returns to the free list ("SGLang RadixAttention", section on
    reference counting: a block referenced by a live request is never
    reclaimed).

Allocation policy (the pages do not state one; this is the reading both sides
implement): the free list starts as a Fisher-Yates shuffle of [0, NB) driven
by splitmix64 (Vigna) seeded with alloc_seed (the identity when the seed is
0): for i = NB-1 down to 1, j = next() mod (i+1), swap(a[i], a[j]).
Allocation pops the front; a freed block is pushed on the front; a freed
sequence releases its table from the last entry to the first.  Sequence ids
are the lowest unused id.

With `store` (host arrays k[L][NB][Hkv][bs][d], v likewise, uint16 bf16
bits) the model also writes the appended K/V into its own host pool and
performs the copy-on-write copies there, so the oracle's attention reads KV
that never went through the CUDA path.
"""
from __future__ import annotations

from collections import deque

MASK64 = (1 << 64) - 1


class PoolError(Exception):
    def __init__(self, kind: str, msg: str = ""):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind   # "oom" | "invalid" | "state"


def splitmix64_stream(seed: int):
    state = seed & MASK64
    while True:
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def initial_free_list(num_blocks: int, alloc_seed: int) -> list:
    a = list(range(num_blocks))
    if alloc_seed != 0:
        rng = splitmix64_stream(alloc_seed)
        for i in range(num_blocks - 1, 0, -1):
            j = next(rng) % (i + 1)
            a[i], a[j] = a[j], a[i]
    return a


class PoolModel:
    def __init__(self, num_blocks: int, block_size: int, max_seqs: int,
                 max_blocks_per_seq: int, alloc_seed: int = 0, store=None):
        self.NB = num_blocks
        self.bs = block_size
        self.max_seqs = max_seqs
        self.MB = max_blocks_per_seq
        self.free = deque(initial_free_list(num_blocks, alloc_seed))
        self.ref = [0] * num_blocks
        self.tables = {}     # seq id -> list of block ids
        self.lens = {}       # seq id -> token count
        self.cow_copies = 0
        self.store = store   # (k_pool, v_pool) numpy uint16 or None

    # -- queries
    def table(self, s):
        self._live(s)
        return list(self.tables[s])

    def length(self, s):
        self._live(s)
        return self.lens[s]

    def refcount(self, b):
        if not 0 <= b < self.NB:
            raise PoolError("invalid", f"block {b}")
        return self.ref[b]

    def free_count(self):
        return len(self.free)

    def live(self):
        return sorted(self.tables)

    def _live(self, s):
        if s not in self.tables:
            raise PoolError("invalid", f"sequence {s} is not live")

    def _pop(self):
        b = self.free.popleft()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _new_id(self):
        for i in range(self.max_seqs):
            if i not in self.tables:
                return i
        raise PoolError("oom", "no free sequence id")

    # -- operations
    def alloc(self):
        s = self._new_id()
        self.tables[s] = []
        self.lens[s] = 0
        return s

    def fork(self, parent):
        self._live(parent)
        s = self._new_id()
        self.tables[s] = list(self.tables[parent])
        self.lens[s] = self.lens[parent]
        for b in self.tables[s]:
            self.ref[b] += 1
        return s

    def blocks_needed(self, s, ntok):
        """(copy-on-write copies, fresh blocks) an append of ntok would take."""
        n = self.lens[s]
        t = self.tables[s]
        used = n % self.bs
        cow = 1 if (ntok > 0 and used != 0 and self.ref[t[-1]] > 1) else 0
        fresh = -(-(n + ntok) // self.bs) - len(t)
        return cow, fresh

    def append(self, s, ntok, k=None, v=None):
        """Append ntok tokens.  k, v: [L][ntok][Hkv][d] uint16 (with a store).
        Returns the list of (block, slot) the tokens went to."""
        self._live(s)
        if ntok < 0:
            raise PoolError("invalid", "negative token count")
        cow, fresh = self.blocks_needed(s, ntok)
        if len(self.tables[s]) + fresh > self.MB:
            raise PoolError("invalid", "block table capacity exceeded")
        if cow + fresh > len(self.free):
            raise PoolError("oom", f"need {cow + fresh} blocks, {len(self.free)} free")
        t = self.tables[s]
        n = self.lens[s]
        if cow:
            old = t[-1]
            new = self._pop()
            self.ref[old] -= 1
            t[-1] = new
            self.cow_copies += 1
            if self.store is not None:
                used = n % self.bs
                for arr in self.store:
                    arr[:, new, :, :used, :] = arr[:, old, :, :used, :]
        slots = []
        for i in range(ntok):
            pos = n + i
            if pos % self.bs == 0:
                t.append(self._pop())
            slots.append((t[pos // self.bs], pos % self.bs))
        self.lens[s] = n + ntok
        if self.store is not None and ntok:
            kp, vp = self.store
            for i, (b, sl) in enumerate(slots):
                kp[:, b, :, sl, :] = k[:, i, :, :]
                vp[:, b, :, sl, :] = v[:, i, :, :]
        return slots

    def free_seq(self, s):
        self._live(s)
        for b in reversed(self.tables[s]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.appendleft(b)
        del self.tables[s]
        del self.lens[s]

    # -- holders other than sequences (the prefix cache) and sequences that
    #    start from blocks someone already holds ("Trellis", section
    #    "RadixAttention in Trellis": a session acquires existing prefix
    #    blocks by raising their refcount instead of allocating)
    def hold_block(self, b):
        """One more reference to a live block."""
        if not 0 <= b < self.NB or self.ref[b] <= 0:
            raise PoolError("invalid", f"block {b} is not in use")
        self.ref[b] += 1

    def drop_block(self, b) -> bool:
        """One reference fewer; True when the block went back to the pool."""
        if not 0 <= b < self.NB or self.ref[b] <= 0:
            raise PoolError("invalid", f"block {b} is not in use")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.appendleft(b)
            return True
        return False

    def alloc_prefix(self, blocks):
        """A new sequence whose table is `blocks` (one more reference each),
        holding len(blocks) full blocks of tokens."""
        if len(blocks) > self.MB:
            raise PoolError("invalid", "block table capacity exceeded")
        for b in blocks:
            if not 0 <= b < self.NB or self.ref[b] <= 0:
                raise PoolError("invalid", f"block {b} is not in use")
        s = self._new_id()
        self.tables[s] = list(blocks)
        self.lens[s] = len(blocks) * self.bs
        for b in blocks:
            self.ref[b] += 1
        return s

    def accept_draft(self, s, ctx_len, parent, accepted):
        """Speculative accept after tree verify: keep the draft path from a
        root of the draft tree down to node `accepted` (-1: keep none) and
        drop the rest ("CAST", section on speculative decoding: the target
        accepts a path of the draft tree).  Draft node i sits at position
        ctx_len + i.  The path's tokens move to positions ctx_len, ctx_len+1,
        ... in order; the length becomes ctx_len + len(path); blocks past the
        new end are released (last to first).  A block that receives a moved
        token and is shared with another sequence is copied first (copy on
        write, in increasing block order, before anything is released).
        Returns the path."""
        self._live(s)
        n = len(parent)
        if ctx_len < 0 or ctx_len + n != self.lens[s] or not -1 <= accepted < n:
            raise PoolError("invalid", "draft region does not match the sequence")
        for i, p in enumerate(parent):
            if not -1 <= p < i:
                raise PoolError("invalid", f"parent of draft node {i}")
        path = []
        j = accepted
        while j >= 0:
            path.append(j)
            j = parent[j]
        path.reverse()
        bs = self.bs
        t = self.tables[s]
        written = sorted({(ctx_len + i) // bs for i, node in enumerate(path) if node != i})
        shared = [j for j in written if self.ref[t[j]] > 1]
        if len(shared) > len(self.free):
            raise PoolError("oom", "copy-on-write blocks")
        for j in shared:
            old, new = t[j], self._pop()
            self.ref[old] -= 1
            t[j] = new
            self.cow_copies += 1
            if self.store is not None:
                for arr in self.store:
                    arr[:, new] = arr[:, old]
        if self.store is not None:
            for arr in self.store:
                kept = [arr[:, t[(ctx_len + node) // bs], :, (ctx_len + node) % bs, :].copy() for node in path]
                for i, row in enumerate(kept):
                    dp = ctx_len + i
                    arr[:, t[dp // bs], :, dp % bs, :] = row
        new_len = ctx_len + len(path)
        keep = -(-new_len // bs)
        for b in reversed(t[keep:]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.appendleft(b)
        del t[keep:]
        self.lens[s] = new_len
        return path
