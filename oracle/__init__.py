"""Oracle for paged / prefix-shared decode attention and tree-verify attention.

TEST INFRASTRUCTURE.  Only `tests/`, `__graft_entry__.smoke()` and the
`cpu_baseline` / `--impl reference` legs of `bench.py` may import this
package.  The library (`paged_prefix_shared_decode_gb300`) never does, and
this package never imports the library.

Contents:
  attention.c    -- fp64 definition of decode and tree-verify attention (C,
                    OpenMP over (layer, query, head)), built into liboracle.so
  pool_model.py  -- the block pool / fork / copy-on-write bookkeeping model
  radix_model.py -- the radix-tree prefix cache over the pool's blocks
  kv4.py         -- a 4-bit KV page format (codes and per-row scales)
  this file      -- ctypes wrappers and a helper that replays a workload's
                    op trace through the model into the oracle's own host pool

Every function here is pinned by `tests/test_oracle_pins.py` to brute force,
closed forms and invariants, and by `tests/golden/` to the pages' own worked
numbers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .pool_model import PoolModel, PoolError, initial_free_list, splitmix64_stream  # noqa: F401
from .radix_model import RadixModel  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int32), ("nq", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("bs", ctypes.c_int32),
                ("NB", ctypes.c_int32), ("MB", ctypes.c_int32), ("scale", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile attention.c with gcc (-O2, OpenMP, IEEE fp64: no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            lib.oracle_decode.argtypes = [ctypes.POINTER(_Shape), P, P, P, P, P, P,
                                          ctypes.c_int64, P, P, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_verify.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, ctypes.c_int,
                                          P, P, P, P, P, P, P, ctypes.c_int64, P, P, ctypes.c_int]
            lib.oracle_verify.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return _load().oracle_max_threads()


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def decode_attention(q, k_pool, v_pool, tables, lens, scale=None, samples=None, threads=0):
    """fp64 paged decode attention.

    q: uint16 [L][nq][Hq][d]; k_pool, v_pool: uint16 [L][NB][Hkv][bs][d];
    tables: int32 [nq][MB]; lens: int32 [nq].  samples: optional int32
    [n][3] of (layer, query, head).  Returns (out fp64, lse fp64) shaped
    [L][nq][Hq][d], [L][nq][Hq] (or [n][d], [n] when sampled).
    """
    q = _c(q, np.uint16); k_pool = _c(k_pool, np.uint16); v_pool = _c(v_pool, np.uint16)
    tables = _c(tables, np.int32); lens = _c(lens, np.int32)
    L, nq, Hq, d = q.shape
    _, NB, Hkv, bs, d2 = k_pool.shape
    assert d2 == d and tables.shape[0] == nq and lens.shape == (nq,)
    sh = _Shape(L, nq, Hq, Hkv, d, bs, NB, tables.shape[1],
                (1.0 / np.sqrt(d)) if scale is None else float(scale))
    if samples is not None:
        samples = _c(samples, np.int32).reshape(-1, 3)
        n = samples.shape[0]
        out = np.empty((n, d)); lse = np.empty(n)
    else:
        n = 0
        out = np.empty((L, nq, Hq, d)); lse = np.empty((L, nq, Hq))
    rc = _load().oracle_decode(ctypes.byref(sh), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(tables),
                               _ptr(lens), _ptr(samples), n, _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_decode: empty sequence or block id outside the pool")
    return out, lse


def verify_attention(q, k_pool, v_pool, tables, ctx_lens, parents, scale=None, samples=None,
                     threads=0):
    """fp64 tree-verify attention.

    q: uint16 [L][B*n][Hq][d]; tables int32 [B][MB]; ctx_lens int32 [B];
    parents int32 [B][n] with parents[b][i] < i (-1 for a root).  Draft token
    j of sequence b sits at position ctx_lens[b] + j of its table.
    """
    q = _c(q, np.uint16); k_pool = _c(k_pool, np.uint16); v_pool = _c(v_pool, np.uint16)
    tables = _c(tables, np.int32); ctx_lens = _c(ctx_lens, np.int32); parents = _c(parents, np.int32)
    L, nq, Hq, d = q.shape
    B, n = parents.shape
    assert nq == B * n
    _, NB, Hkv, bs, _ = k_pool.shape
    sh = _Shape(L, nq, Hq, Hkv, d, bs, NB, tables.shape[1],
                (1.0 / np.sqrt(d)) if scale is None else float(scale))
    if samples is not None:
        samples = _c(samples, np.int32).reshape(-1, 3)
        m = samples.shape[0]
        out = np.empty((m, d)); lse = np.empty(m)
    else:
        m = 0
        out = np.empty((L, nq, Hq, d)); lse = np.empty((L, nq, Hq))
    rc = _load().oracle_verify(ctypes.byref(sh), B, n, _ptr(q), _ptr(k_pool), _ptr(v_pool),
                               _ptr(tables), _ptr(ctx_lens), _ptr(parents), _ptr(samples), m,
                               _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_verify: bad parent pointer or block id outside the pool")
    return out, lse


class ReplayedWorkload:
    """A workload's op trace replayed through the oracle's own pool model."""

    def __init__(self, model, k_pool, v_pool, ids):
        self.model = model
        self.k_pool = k_pool
        self.v_pool = v_pool
        self.ids = ids           # workload sequence name -> model sequence id

    def tables(self, names, width):
        t = np.full((len(names), width), -1, dtype=np.int32)
        lens = np.zeros(len(names), dtype=np.int32)
        for r, nm in enumerate(names):
            tb = self.model.table(self.ids[nm])
            t[r, :len(tb)] = tb
            lens[r] = self.model.length(self.ids[nm])
        return t, lens


def replay(w, alloc_seed: int = 1, with_store: bool = True, kv_fn=None) -> ReplayedWorkload:
    """Run workload `w`'s ops through a fresh PoolModel.  K/V values come from
    `kv_fn(w, op_index)` (the shared seeded generator by default)."""
    from workloads import append_kv
    kv_fn = kv_fn or append_kv
    s = w.shapes
    store = None
    if with_store:
        kp = np.zeros((s.L, w.num_blocks, s.Hkv, s.bs, s.d), dtype=np.uint16)
        vp = np.zeros_like(kp)
        store = (kp, vp)
    m = PoolModel(w.num_blocks, s.bs, w.max_seqs, w.max_blocks_per_seq, alloc_seed, store)
    ids = {}
    for i, op in enumerate(w.ops):
        if op[0] == "alloc":
            ids[op[1]] = m.alloc()
        elif op[0] == "fork":
            ids[op[2]] = m.fork(ids[op[1]])
        elif op[0] == "append":
            k = v = None
            if with_store:
                k, v = kv_fn(w, i)
            m.append(ids[op[1]], op[2], k, v)
        elif op[0] == "free":
            m.free_seq(ids.pop(op[1]))
    return ReplayedWorkload(m, store[0] if store else None, store[1] if store else None, ids)


def replay_step(rw: ReplayedWorkload, w, step_k, step_v):
    """Append one decode step's tokens (w.step_tokens per batch sequence, in
    batch order) through the model."""
    n = w.step_tokens
    for r, nm in enumerate(w.batch):
        sl = slice(r * n, (r + 1) * n)
        rw.model.append(rw.ids[nm], n, step_k[:, sl], step_v[:, sl])
