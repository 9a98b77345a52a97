"""Oracle model of a radix-tree prefix cache over the pool's blocks (test
infrastructure: only the tests and the benchmark's CPU leg use it; it shares
no code with the library).

What the pages describe ("SGLang RadixAttention", sections on the node and
edge structure, on the three operations match / split / insert, and on
reference counting with LRU eviction; "Trellis", section "RadixAttention in
Trellis" and the benchmark definitions):
  * a tree whose root is the empty sequence; the edge into a node holds a run
    of token ids and the ids of the pool blocks that store those tokens;
  * match: from the root, follow the edges that agree with the prompt for as
    long as they agree; the blocks of the agreeing part are reused, and every
    node the match used is locked (its counter of active requests goes up)
    and marked as just used;
  * split: an edge that agrees with a new sequence for only part of its run
    is cut into an upper edge (the common part) and a lower one (the rest);
    the blocks are divided by slicing the id list, nothing is copied;
  * insert: walk as in match, splitting where needed; what is left of the
    sequence becomes a new leaf holding its blocks;
  * eviction: while fewer blocks are free than needed, take the unlocked leaf
    used longest ago, give its blocks back and remove it; a parent that is
    left without children and unlocked is then a leaf like any other.

Readings adopted where the pages leave a step open:
  * granularity is whole blocks: runs are whole numbers of blocks of bs
    tokens, a match is rounded down to whole agreeing blocks and splits fall
    on block boundaries (the Trellis benchmark rounds the shared region to
    whole blocks; a partial block cannot be shared by reference);
  * the cache holds one pool reference on each block in the tree (taken when
    a leaf is made, dropped at eviction), so a block leaves the pool only
    when neither the cache nor any sequence holds it; the per-node lock
    counter only decides what may be evicted;
  * "last used" is a logical clock that every match and insert advances,
    stamped on every node of the path that operation used (wall-clock time
    would make runs unrepeatable);
  * a split's upper node inherits the lower node's lock count (the requests
    that locked the lower node used the upper part too) and is stamped by
    the insert that split it; the lower node keeps its stamp;
  * a match also locks a node whose edge agreed only in part (the request
    reuses some of its blocks); blocks are given back last to first.
"""
from __future__ import annotations

from .pool_model import PoolError


class _Node:
    __slots__ = ("parent", "run", "blocks", "kids", "locks", "stamp")

    def __init__(self, parent, run, blocks):
        self.parent = parent
        self.run = list(run)        # token ids, len(run) == len(blocks) * bs
        self.blocks = list(blocks)  # pool block ids of this edge
        self.kids = {}              # first block's tokens (tuple) -> child
        self.locks = 0
        self.stamp = 0


class RadixModel:
    def __init__(self, pool):
        self.pool = pool
        self.bs = pool.bs
        self.clock = 0
        self.root = _Node(None, [], [])

    # -- helpers
    def _key(self, tokens, at):
        return tuple(tokens[at:at + self.bs])

    def _agree(self, node, tokens, at, end):
        """Whole blocks of node's run equal to tokens[at:end], from the start."""
        bs = self.bs
        k = 0
        while k < len(node.blocks) and at + (k + 1) * bs <= end and \
                node.run[k * bs:(k + 1) * bs] == list(tokens[at + k * bs:at + (k + 1) * bs]):
            k += 1
        return k

    def nodes(self):
        out, todo = [], [self.root]
        while todo:
            n = todo.pop()
            out.append(n)
            todo.extend(n.kids.values())
        return out

    # -- operations
    def match(self, tokens):
        """Longest cached prefix in whole blocks: (block ids, lock), lock is
        the deepest node used (None when nothing matched)."""
        self.clock += 1
        end = len(tokens) // self.bs * self.bs
        node, at, got, used = self.root, 0, [], []
        while at < end:
            kid = node.kids.get(self._key(tokens, at))
            if kid is None:
                break
            k = self._agree(kid, tokens, at, end)
            got.extend(kid.blocks[:k])
            used.append(kid)
            at += k * self.bs
            if k < len(kid.blocks):
                break
            node = kid
        for n in used:
            n.locks += 1
            n.stamp = self.clock
        return got, (used[-1] if used else None)

    def unlock(self, lock):
        n = lock
        while n is not None and n is not self.root:
            if n.locks <= 0:
                raise PoolError("state", "unlock of a node that is not locked")
            n.locks -= 1
            n = n.parent

    def insert(self, tokens, blocks):
        """Caches the whole blocks of a sequence whose tokens are `tokens` and
        whose blocks are `blocks`."""
        self.clock += 1
        nblk = min(len(tokens) // self.bs, len(blocks))
        end = nblk * self.bs
        node, at = self.root, 0
        while at < end:
            key = self._key(tokens, at)
            kid = node.kids.get(key)
            if kid is None:
                leaf = _Node(node, tokens[at:end], blocks[at // self.bs:nblk])
                leaf.stamp = self.clock
                for b in leaf.blocks:
                    self.pool.hold_block(b)
                node.kids[key] = leaf
                return
            k = self._agree(kid, tokens, at, end)
            if k < len(kid.blocks):
                upper = _Node(node, kid.run[:k * self.bs], kid.blocks[:k])
                upper.locks = kid.locks
                kid.run = kid.run[k * self.bs:]
                kid.blocks = kid.blocks[k:]
                kid.parent = upper
                upper.kids[tuple(kid.run[:self.bs])] = kid
                node.kids[key] = upper
                kid = upper
            kid.stamp = self.clock
            node = kid
            at += k * self.bs

    def evict(self, need_free):
        """(met, blocks returned to the pool)."""
        freed = 0
        while self.pool.free_count() < need_free:
            leaves = [n for n in self.nodes() if n is not self.root and not n.kids and n.locks == 0]
            if not leaves:
                return False, freed
            v = min(leaves, key=lambda n: n.stamp)
            for b in reversed(v.blocks):
                if self.pool.drop_block(b):
                    freed += 1
            del v.parent.kids[tuple(v.run[:self.bs])]
        return True, freed

    def dump(self):
        """Canonical form: depth-first from the root, children in increasing
        order of their first block's tokens; per node (depth, tokens, blocks,
        locks, stamp)."""
        out = []

        def walk(n, depth):
            for key in sorted(n.kids):
                c = n.kids[key]
                out.append((depth, tuple(c.run), tuple(c.blocks), c.locks, c.stamp))
                walk(c, depth + 1)
        walk(self.root, 0)
        return out
