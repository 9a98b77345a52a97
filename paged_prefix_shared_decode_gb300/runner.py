"""Drives a workload op trace (alloc / fork / append / free, then decode or
verify queries) through the C ABI, with torch supplying device memory and
streams.  Used by the benchmark and the tests; every step of the path runs in
libkvp's kernels.
"""
from __future__ import annotations

import numpy as np

from . import (AttnDesc, PoolDesc, KVP_KV_BF16, KVP_KV_4BIT, kv_pool_create, kv_pool_create_kv4, kv_pool_destroy,
               seq_alloc, seq_fork, seq_free,
               seq_append, seq_append_batch, seq_reserve, kvp_gather_tables, paged_decode_attention,
               kvp_decode_workspace_size, tree_verify_attention, kvp_verify_workspace_size)


def _torch():
    import torch
    return torch


def bf16_tensor(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns (numpy) -> torch bfloat16 tensor on `device`."""
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


class PoolRunner:
    """A pool with device K/V storage and a name -> sequence id map.  With
    kv4 the pool holds 4-bit pages (k_pool / v_pool are the codes, k_exp /
    v_exp the row exponents); appends still take bf16 K/V."""

    def __init__(self, w, alloc_seed: int = 1, device: bool = True, poison: bool = False,
                 num_blocks: int | None = None, kv4: bool = False):
        torch = _torch()
        s = w.shapes
        self.w = w
        self.shapes = s
        self.NB = num_blocks or w.num_blocks
        self.k_pool = self.v_pool = self.k_exp = self.v_exp = None
        self.kv4 = kv4
        desc = PoolDesc(s.L, self.NB, s.bs, s.Hkv, s.d, w.max_seqs, w.max_blocks_per_seq, alloc_seed)
        if kv4:
            self.k_pool = torch.zeros((s.L, self.NB, s.Hkv, s.bs, s.d // 2), dtype=torch.uint8, device="cuda")
            self.v_pool = torch.zeros_like(self.k_pool)
            self.k_exp = torch.zeros((s.L, self.NB, s.Hkv, s.bs), dtype=torch.int8, device="cuda")
            self.v_exp = torch.zeros_like(self.k_exp)
            self.pool = kv_pool_create_kv4(desc, self.k_pool, self.k_exp, self.v_pool, self.v_exp)
            self.ids = {}
            return
        if device:
            shape = (s.L, self.NB, s.Hkv, s.bs, s.d)
            if poison:   # bf16 NaN in every slot: any read of an unwritten slot shows up
                self.k_pool = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
                self.v_pool = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            else:
                self.k_pool = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
                self.v_pool = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        self.pool = kv_pool_create(desc, self.k_pool, self.v_pool)
        self.ids = {}

    def close(self):
        if self.pool:
            kv_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def run_ops(self, kv_fn=None, device_kv=True, kv_dev_fn=None):
        """Replay the workload's ops.  kv_fn(w, i) gives host (k, v) bits for
        append op i (the shared seeded generator by default); kv_dev_fn(w, i)
        instead gives device tensors directly; with device_kv=False only the
        bookkeeping runs."""
        from workloads import append_kv
        kv_fn = kv_fn or append_kv
        for i, op in enumerate(self.w.ops):
            if op[0] == "alloc":
                self.ids[op[1]] = seq_alloc(self.pool)
            elif op[0] == "fork":
                self.ids[op[2]] = seq_fork(self.pool, self.ids[op[1]])
            elif op[0] == "append":
                if not device_kv:
                    seq_reserve(self.pool, self.ids[op[1]], op[2])
                elif kv_dev_fn is not None:
                    k, v = kv_dev_fn(self.w, i)
                    seq_append(self.pool, self.ids[op[1]], k, v, op[2])
                else:
                    k, v = kv_fn(self.w, i)
                    seq_append(self.pool, self.ids[op[1]], bf16_tensor(k), bf16_tensor(v), op[2])
            elif op[0] == "free":
                seq_free(self.pool, self.ids.pop(op[1]))

    def append_step(self, k_dev, v_dev, names=None, ntok=None):
        """One decode step's appends (ntok per sequence, batch order) in one launch."""
        names = names if names is not None else self.w.batch
        ntok = self.w.step_tokens if ntok is None else ntok
        seqs = [self.ids[n] for n in names]
        seq_append_batch(self.pool, seqs, [ntok] * len(seqs), k_dev, v_dev)

    def tables(self, names=None, width=None):
        names = names if names is not None else self.w.batch
        width = width or self.w.max_blocks_per_seq
        return kvp_gather_tables(self.pool, [self.ids[n] for n in names], width)

    def attn_desc(self, use_sharing=True, scale=0.0) -> AttnDesc:
        s = self.shapes
        return AttnDesc(s.L, s.Hq, s.Hkv, s.d, s.bs, self.NB, scale, 1 if use_sharing else 0,
                        KVP_KV_4BIT if self.kv4 else KVP_KV_BF16)


class DecodeCall:
    """Buffers for paged_decode_attention over a fixed batch: host tables,
    out, lse and a workspace sized for the current tables."""

    def __init__(self, runner: PoolRunner, use_sharing=True, scale=0.0):
        torch = _torch()
        self.r = runner
        s = runner.shapes
        self.desc = runner.attn_desc(use_sharing, scale)
        S = len(runner.w.batch)
        self.out = torch.empty((s.L, S, s.Hq, s.d), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((s.L, S, s.Hq), dtype=torch.float32, device="cuda")
        self.ws = torch.empty(0, dtype=torch.uint8, device="cuda")
        self.h_tables = self.h_lens = None

    def refresh(self):
        """Re-read tables from the pool and grow the workspace if needed."""
        torch = _torch()
        t, ln = self.r.tables()
        self.h_tables, self.h_lens = t, ln
        need = kvp_decode_workspace_size(self.desc, t, ln)
        if self.ws.numel() < need:
            self.ws = torch.empty(need + (1 << 20), dtype=torch.uint8, device="cuda")

    def __call__(self, q_dev, stream=None):
        paged_decode_attention(q_dev, self.r.k_pool, self.r.v_pool, self.h_tables, self.h_lens,
                               self.desc, self.out, self.lse, self.ws, stream=stream)
        return self.out, self.lse


class VerifyCall:
    def __init__(self, runner: PoolRunner, scale=0.0):
        torch = _torch()
        w = runner.w
        s = runner.shapes
        self.r = runner
        self.n = w.info["n_draft"]
        self.B = len(w.batch)
        self.desc = runner.attn_desc(True, scale)
        t, ln = runner.tables()
        self.ctx = (ln - self.n).astype(np.int32)
        self.h_tables = t
        self.parent = torch.from_numpy(np.ascontiguousarray(w.info["parents"], np.int32)).cuda()
        self.out = torch.empty((s.L, self.B * self.n, s.Hq, s.d), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((s.L, self.B * self.n, s.Hq), dtype=torch.float32, device="cuda")
        need = kvp_verify_workspace_size(self.desc, t, self.ctx, self.n)
        self.ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def __call__(self, q_dev, stream=None):
        tree_verify_attention(q_dev, self.parent, self.n, self.r.k_pool, self.r.v_pool, self.h_tables,
                              self.ctx, self.desc, self.out, self.lse, self.ws, stream=stream)
        return self.out, self.lse
