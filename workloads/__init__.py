"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no attention or pool arithmetic.  It only states *what*
happens in a workload (which sequences are allocated, forked and appended to,
how many tokens each append carries, which sequences are queried) and draws
the random values that go in (K, V, Q as bf16 bit patterns, draft-tree parent
pointers).  Each side turns an op trace into block tables and results on its
own.

Random values: N(0, 1) from numpy's Philox4x32 counter-based generator (Salmon
et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11), one stream per
(seed, op, tensor, layer), rounded to bf16 round-to-nearest-even and stored as
uint16 bit patterns.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Shapes", "Workload", "normal_bf16", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "tiny_fork", "dendrite", "trellis", "mcts", "verify_tree", "random_trace",
    "append_kv", "step_kv", "step_q", "verify_q", "TINYLLAMA", "LLAMA3_8B", "prefix_cache_sessions",
]


@dataclass(frozen=True)
class Shapes:
    """Attention shapes: layers, query heads, kv heads, head dim, block size."""
    L: int
    Hq: int
    Hkv: int
    d: int
    bs: int

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def token_bytes(self) -> int:
        """K+V bytes of one token in one layer (bf16)."""
        return 2 * self.Hkv * self.d * 2


TINYLLAMA = dict(Hq=32, Hkv=4, d=64)     # TinyLlama-1.1B attention: 22 layers
LLAMA3_8B = dict(Hq=32, Hkv=8, d=128)    # Llama-3-8B attention: 32 layers


@dataclass
class Workload:
    """An op trace over named sequences plus the decode batch.

    ops: ("alloc", sid) | ("fork", parent_sid, child_sid) | ("append", sid, ntok)
         | ("free", sid)
    batch: sids queried by one decode step, in row order of q/out.
    step_tokens: tokens each batch sequence appends at the start of a step
         (1 for a decode step; the query then attends to them too).
    """
    name: str
    shapes: Shapes
    ops: list
    batch: list
    seed: int = 0
    step_tokens: int = 1
    num_blocks: int = 0
    max_seqs: int = 0
    max_blocks_per_seq: int = 0
    info: dict = field(default_factory=dict)

    def total_appended(self) -> int:
        return sum(op[2] for op in self.ops if op[0] == "append")


# ----------------------------------------------------------------- values

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_POOL = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _philox(seed: int, stream: int, sub: int) -> np.random.Generator:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF,
                    ((stream & 0xFFFFFFFF) << 32) | (sub & 0xFFFFFFFF)], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def normal_bf16(seed: int, stream: int, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values as bf16 bits; the leading axis is drawn from
    independent sub-streams in parallel (deterministic for a given shape)."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size == 0:
        return out
    lead = shape[0]
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    flat = out.reshape(lead, inner)

    def fill(i):
        g = _philox(seed, stream, i)
        x = g.standard_normal(inner, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        flat[i] = f32_to_bf16_bits(x)

    if lead * inner >= (1 << 20) and lead > 1:
        list(_pool().map(fill, range(lead)))
    else:
        for i in range(lead):
            fill(i)
    return out


# streams: op i uses 4*i (K) and 4*i+1 (V); steps and queries use high ranges
_STEP_BASE = 1 << 28
_Q_BASE = 1 << 29


def append_kv(w: Workload, op_index: int):
    """K and V of append op `op_index`: two [L][ntok][Hkv][d] bf16-bit arrays."""
    kind, _sid, ntok = w.ops[op_index]
    assert kind == "append"
    s = w.shapes
    k = normal_bf16(w.seed, 4 * op_index, (s.L, ntok, s.Hkv, s.d))
    v = normal_bf16(w.seed, 4 * op_index + 1, (s.L, ntok, s.Hkv, s.d))
    return k, v


def step_kv(w: Workload, step: int):
    """K and V appended by a decode step: [L][S*step_tokens][Hkv][d] each,
    sequence-major within a layer (the batch order, step_tokens per sequence)."""
    s = w.shapes
    n = len(w.batch) * w.step_tokens
    k = normal_bf16(w.seed, _STEP_BASE + 4 * step, (s.L, n, s.Hkv, s.d))
    v = normal_bf16(w.seed, _STEP_BASE + 4 * step + 1, (s.L, n, s.Hkv, s.d))
    return k, v


def step_q(w: Workload, step: int, scale: float = 1.0):
    """Decode queries of a step: [L][S][Hq][d]."""
    s = w.shapes
    return normal_bf16(w.seed, _Q_BASE + step, (s.L, len(w.batch), s.Hq, s.d), scale)


def verify_q(w: Workload, scale: float = 1.0):
    """Draft-token queries: [L][B*n][Hq][d] (sequence-major, then node)."""
    s = w.shapes
    nq = len(w.batch) * w.info["n_draft"]
    return normal_bf16(w.seed, _Q_BASE + 7777, (s.L, nq, s.Hq, s.d), scale)


# ----------------------------------------------------------------- workloads

def _finish(w: Workload, extra_blocks: int = 0, seq_slack: int = 0) -> Workload:
    """Size the pool: enough blocks for every appended token even with no
    sharing, plus CoW copies and `extra_blocks` decode steps' worth."""
    bs = w.shapes.bs
    live = {}
    need = 0
    nseq = 0
    maxlen = 0
    for op in w.ops:
        if op[0] == "alloc":
            live[op[1]] = 0
            nseq += 1
        elif op[0] == "fork":
            live[op[2]] = live[op[1]]
            nseq += 1
        elif op[0] == "append":
            live[op[1]] += op[2]
            need += math.ceil(op[2] / bs) + 1
            maxlen = max(maxlen, live[op[1]])
    need += extra_blocks + len(w.batch) * 2
    w.num_blocks = w.num_blocks or int(need)
    w.max_seqs = w.max_seqs or (nseq + seq_slack + 1)
    w.max_blocks_per_seq = w.max_blocks_per_seq or (math.ceil((maxlen + 64 * w.step_tokens) / bs) + 2)
    return w


def tiny_fork(seed: int = 0) -> Workload:
    """1 layer, 32q/4kv heads, d 64, block 16: a 256-token parent forked into
    4 children that each append 32 private tokens; one query per child."""
    sh = Shapes(L=1, bs=16, **TINYLLAMA)
    ops = [("alloc", 0), ("append", 0, 256)]
    for c in range(1, 5):
        ops += [("fork", 0, c), ("append", c, 32)]
    w = Workload("tiny_fork", sh, ops, batch=[1, 2, 3, 4], seed=seed, step_tokens=0)
    return _finish(w)


def dendrite(seed: int = 0, layers: int = 22, prefix: int = 4096, branches: int = 6,
             max_private: int = 512) -> Workload:
    """TinyLlama shapes, block 16: a 4096-token prefix forked into 6 branches,
    each with U{0..512} private tokens; each step appends one token per branch
    and queries it."""
    sh = Shapes(L=layers, bs=16, **TINYLLAMA)
    g = _philox(seed, 999_001, 0)
    priv = [int(x) for x in g.integers(0, max_private + 1, size=branches)]
    ops = [("alloc", 0), ("append", 0, prefix)]
    for b in range(1, branches + 1):
        ops.append(("fork", 0, b))
        if priv[b - 1] > 0:
            ops.append(("append", b, priv[b - 1]))
    w = Workload("dendrite", sh, ops, batch=list(range(1, branches + 1)), seed=seed,
                 info=dict(prefix=prefix, private=priv))
    return _finish(w, extra_blocks=branches * 8)


def trellis_prefix_blocks(phi: float, L_prompt: int = 512, block: int = 32) -> int:
    """prefixBlocks = round(phi * L / 32) with round-half-up, capped at
    L/32 - 1 (the probe always differs in the warm prompt's last block)."""
    p = int(math.floor(phi * L_prompt / block + 0.5))
    return min(p, L_prompt // block - 1)


def trellis(phi: float, seed: int = 0, layers: int = 22, sessions: int = 64,
            L_prompt: int = 512, decode: int = 64) -> Workload:
    """TinyLlama head shapes, block 32: a warm prefix of 32p tokens forked into
    N sessions; each appends its 512-32p suffix and decode-1 generated tokens;
    the step appends the last decode token (length 576) and queries it."""
    sh = Shapes(L=layers, bs=32, **TINYLLAMA)
    p = trellis_prefix_blocks(phi, L_prompt, 32)
    ops = [("alloc", 0)]
    if p > 0:
        ops.append(("append", 0, 32 * p))
    for s in range(1, sessions + 1):
        ops.append(("fork", 0, s))
        ops.append(("append", s, L_prompt - 32 * p + decode - 1))
    w = Workload(f"trellis_phi{phi}", sh, ops, batch=list(range(1, sessions + 1)), seed=seed,
                 info=dict(phi=phi, prefix_blocks=p, realised_phi=32 * p / L_prompt))
    return _finish(w, extra_blocks=sessions * 4)


def prefix_cache_sessions(phi: float, seed: int = 0, sessions: int = 64, L_prompt: int = 512,
                          decode: int = 64, vocab: int = 32000):
    """Token ids for the Trellis benchmark's session pattern: one shared
    system prompt of 32 * prefixBlocks tokens, then per session a distinct
    user suffix up to L_prompt tokens and `decode` generated tokens.
    Returns (system, prompts, generated) as lists of int lists."""
    p = trellis_prefix_blocks(phi, L_prompt, 32)
    g = _philox(seed, 999_004, 0)
    system = g.integers(0, vocab, 32 * p).tolist()
    prompts, generated = [], []
    for _ in range(sessions):
        # a suffix that differs from every other one in its first token
        suffix = g.integers(0, vocab, L_prompt - 32 * p).tolist()
        suffix[0] = len(prompts) % vocab
        prompts.append(system + suffix)
        generated.append(g.integers(0, vocab, decode).tolist())
    return system, prompts, generated


def mcts(seed: int = 0, layers: int = 32, root: int = 2048, branching: int = 4,
         depth: int = 4, edge: int = 64) -> Workload:
    """Llama-3-8B shapes, block 16: a 2048-token root; every node is forked
    `branching` times level by level (breadth first) and each child appends a
    64-token edge; all nodes stay alive; each leaf decodes one token."""
    sh = Shapes(L=layers, bs=16, **LLAMA3_8B)
    ops = [("alloc", 0), ("append", 0, root)]
    level = [0]
    nxt = 1
    for _ in range(depth):
        new = []
        for parent in level:
            for _c in range(branching):
                ops += [("fork", parent, nxt), ("append", nxt, edge)]
                new.append(nxt)
                nxt += 1
        level = new
    w = Workload("mcts", sh, ops, batch=level, seed=seed,
                 info=dict(root=root, branching=branching, depth=depth, edge=edge))
    return _finish(w, extra_blocks=len(level) * 4)


def draft_tree(seed: int, n: int = 64, max_depth: int = 8, stream: int = 0) -> np.ndarray:
    """Parent pointers of an n-node draft tree: node 0 is the root (parent -1,
    depth 1); node i picks its parent uniformly among j < i with depth <= 7."""
    g = _philox(seed, 999_002, stream)
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int32)
    depth[0] = 1
    for i in range(1, n):
        cand = np.nonzero(depth[:i] <= max_depth - 1)[0]
        j = int(cand[int(g.integers(0, len(cand)))])
        parent[i] = j
        depth[i] = depth[j] + 1
    return parent


def verify_tree(batch: int, seed: int = 0, layers: int = 32, ctx: int = 2048,
                n_draft: int = 64) -> Workload:
    """Llama-3-8B shapes, block 16: B independent 2048-token contexts, each
    followed by n = 64 draft tokens in its pages, and a random draft tree per
    sequence; 64 queries per sequence."""
    sh = Shapes(L=layers, bs=16, **LLAMA3_8B)
    ops = []
    for b in range(batch):
        ops += [("alloc", b), ("append", b, ctx), ("append", b, n_draft)]
    parents = np.stack([draft_tree(seed, n_draft, stream=b) for b in range(batch)])
    w = Workload(f"verify_B{batch}", sh, ops, batch=list(range(batch)), seed=seed, step_tokens=0,
                 info=dict(ctx=ctx, n_draft=n_draft, parents=parents))
    return _finish(w)


def random_trace(seed: int, n_ops: int, bs: int = 16, max_live: int = 24,
                 max_append: int = 40, layers: int = 1, Hq: int = 4, Hkv: int = 2,
                 d: int = 8, max_len: int = 400) -> Workload:
    """A random op trace (alloc / fork / append 1-40 tokens / free) over at most
    `max_live` live sequences, for bookkeeping parity."""
    g = _philox(seed, 999_003, 0)
    sh = Shapes(L=layers, Hq=Hq, Hkv=Hkv, d=d, bs=bs)
    ops = []
    live = {}
    nxt = 0
    for _ in range(n_ops):
        r = float(g.random())
        names = sorted(live)
        if not names or (r < 0.12 and len(names) < max_live):
            ops.append(("alloc", nxt)); live[nxt] = 0; nxt += 1
        elif r < 0.35 and len(names) < max_live:
            p = names[int(g.integers(0, len(names)))]
            ops.append(("fork", p, nxt)); live[nxt] = live[p]; nxt += 1
        elif r < 0.85:
            s = names[int(g.integers(0, len(names)))]
            n = int(g.integers(1, max_append + 1))
            if live[s] + n <= max_len:
                ops.append(("append", s, n)); live[s] += n
        else:
            s = names[int(g.integers(0, len(names)))]
            ops.append(("free", s)); del live[s]
    w = Workload(f"trace{seed}", sh, ops, batch=sorted(live), seed=seed, step_tokens=0)
    w.max_seqs = nxt + 1
    w.max_blocks_per_seq = max_len // bs + 2
    w.num_blocks = max_live * (max_len // bs + 2) + 8
    return w
