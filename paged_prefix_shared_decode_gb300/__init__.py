"""Python binding of libkvp (paged, prefix-shared KV pool + attention on GB300).

Argument marshalling only: every function forwards to the C ABI entry point
of the same name declared in include/kvp.h.  Device arguments are torch CUDA
tensors (or raw integer device addresses); host arrays are numpy int32
arrays; `stream` defaults to torch's current CUDA stream.  There is no CPU
fallback: importing works without a GPU, but every call needs libkvp.so
(built by `paged_prefix_shared_decode_gb300.build`) and raises KvpError if it
is missing.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "KvpError", "PoolDesc", "AttnDesc", "load", "lib_path",
    "kv_pool_create", "kv_pool_create_kv4", "kv_pool_destroy", "seq_alloc", "seq_fork", "seq_free", "seq_append",
    "seq_append_batch", "seq_reserve", "seq_block_table", "seq_len", "block_refcount",
    "kvp_free_block_count", "kvp_cow_count", "kvp_gather_tables", "kvp_export_tables",
    "kvp_decode_workspace_size", "paged_decode_attention", "kvp_verify_workspace_size",
    "tree_verify_attention", "kvp_device_error", "kvp_decode_plan_stats", "kvp_strerror",
    "kvp_set_kernel_events", "kvp_kernel_launches", "paged_decode_attention_noalloc",
    "paged_decode_attention_kv4", "KVP_KV_BF16", "KVP_KV_4BIT",
    "kvp_pool_decode_workspace_size", "paged_decode_attention_pool", "StepIO", "step_io", "kvp_decode_step",
    "DecodeStep", "KVP_STEP_HOST_MAPPED", "kvp_step_plan_create", "kvp_step_plan_destroy",
    "kvp_decode_step_plan", "kvp_decode_step_run", "StepPlan",
    "KVP_STATIC_WORKSPACE_BYTES",
    "KVP_OK", "KVP_ERR_INVALID", "KVP_ERR_OOM", "KVP_ERR_STATE", "KVP_ERR_CUDA", "KVP_ERR_DEVICE",
    "KVP_ERR_WORKSPACE",
]

KVP_OK, KVP_ERR_INVALID, KVP_ERR_OOM, KVP_ERR_STATE, KVP_ERR_CUDA, KVP_ERR_DEVICE = 0, -1, -2, -3, -4, -5
KVP_ERR_WORKSPACE = -6
KVP_KV_BF16, KVP_KV_4BIT = 0, 1   # page formats (kvp_attn_desc.kv_format)
KVP_STATIC_WORKSPACE_BYTES = 32 << 20   # size of the library's own workspace (include/kvp.h)

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVP_LIB_PATH points the binding at another build of the same C ABI.
lib_path = os.environ.get("KVP_LIB_PATH") or os.path.join(_HERE, "libkvp.so")
_lib = None


class KvpError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = _strerror(code)
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")


def _strerror(code):
    try:
        return load().kvp_strerror(code).decode()
    except Exception:  # library missing: still describe the code
        return {0: "ok", -1: "invalid argument", -2: "out of blocks or sequence slots",
                -3: "operation not possible in this state", -4: "CUDA runtime error",
                -5: "device-side check failed", -6: "workspace too small"}.get(code, "unknown error")


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("alloc_seed", ctypes.c_uint64)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("scale", ctypes.c_float), ("use_sharing", ctypes.c_int32),
                ("kv_format", ctypes.c_int32)]


class StepIO(ctypes.Structure):
    """kvp_step_io: host (h_*) and device (d_*) buffers of one decode step."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("h_k_new", "h_v_new", "h_q", "h_out", "h_lse",
                                               "d_k_new", "d_v_new", "d_q", "d_out", "d_lse")] + \
               [("flags", ctypes.c_uint32)]


KVP_STEP_HOST_MAPPED = 1   # kvp_step_io.flags: host buffers page-locked and device-addressable


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I32P = ctypes.POINTER(ctypes.c_int32)
_SIGS = {
    "kv_pool_create": ([ctypes.POINTER(PoolDesc), _P, _P, ctypes.POINTER(_P)], ctypes.c_int),
    "kv_pool_create_kv4": ([ctypes.POINTER(PoolDesc), _P, _P, _P, _P, ctypes.POINTER(_P)], ctypes.c_int),
    "kv_pool_destroy": ([_P], ctypes.c_int),
    "seq_alloc": ([_P, _I32P], ctypes.c_int),
    "seq_fork": ([_P, _I32, _I32P], ctypes.c_int),
    "seq_free": ([_P, _I32], ctypes.c_int),
    "seq_append": ([_P, _I32, _P, _P, _I32, _P], ctypes.c_int),
    "seq_append_batch": ([_P, _I32, _P, _P, _P, _P, _P], ctypes.c_int),
    "seq_reserve": ([_P, _I32, _I32, _P, _P], ctypes.c_int),
    "seq_block_table": ([_P, _I32, _P, _I32, _I32P], ctypes.c_int),
    "seq_len": ([_P, _I32, _I32P], ctypes.c_int),
    "block_refcount": ([_P, _I32, _I32P], ctypes.c_int),
    "kvp_free_block_count": ([_P, _I32P], ctypes.c_int),
    "kvp_cow_count": ([_P, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "kvp_gather_tables": ([_P, _P, _I32, _I32, _P, _P], ctypes.c_int),
    "kvp_export_tables": ([_P, _P, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "kvp_decode_workspace_size": ([ctypes.POINTER(AttnDesc), _P, _P, _I32, _I32], ctypes.c_size_t),
    "paged_decode_attention": ([_P, _P, _P, _P, _P, _I32, _I32, ctypes.POINTER(AttnDesc),
                                _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "paged_decode_attention_kv4": ([_P, _P, _P, _P, _P, _P, _P, _I32, _I32, ctypes.POINTER(AttnDesc),
                                    _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "kvp_verify_workspace_size": ([ctypes.POINTER(AttnDesc), _P, _P, _I32, _I32, _I32], ctypes.c_size_t),
    "tree_verify_attention": ([_P, _P, _I32, _P, _P, _P, _P, _I32, _I32, ctypes.POINTER(AttnDesc),
                               _P, _P, _P, ctypes.c_size_t, _P], ctypes.c_int),
    "kvp_device_error": ([_P, _P, _I32P], ctypes.c_int),
    "kvp_decode_plan_stats": ([ctypes.POINTER(AttnDesc), _P, _P, _I32, _I32, _I32, _I32P, _I32P,
                               _I32P, _I32P, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "kvp_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "kvp_set_kernel_events": ([_P, _P], ctypes.c_int),
    "paged_decode_attention_noalloc": ([_P, _P, _P, _P, _P, _I32, _I32, ctypes.POINTER(AttnDesc), _P, _P,
                                        _P], ctypes.c_int),
    "kvp_kernel_launches": ([ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "kvp_pool_decode_workspace_size": ([_P, _P, _I32, ctypes.POINTER(AttnDesc)], ctypes.c_size_t),
    "paged_decode_attention_pool": ([_P, _P, _I32, _P, _P, _P, ctypes.POINTER(AttnDesc), _P, ctypes.c_size_t,
                                     _P], ctypes.c_int),
    "kvp_decode_step": ([_P, _P, _I32, _I32, ctypes.POINTER(StepIO), ctypes.POINTER(AttnDesc), _P,
                         ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t), _P], ctypes.c_int),
    "kvp_step_plan_create": ([], _P),
    "kvp_step_plan_destroy": ([_P], None),
    "kvp_decode_step_plan": ([_P, _P, _I32, _I32, ctypes.POINTER(AttnDesc), _P, ctypes.POINTER(ctypes.c_size_t)],
                             ctypes.c_int),
    "kvp_decode_step_run": ([_P, ctypes.POINTER(StepIO), _P, ctypes.c_size_t, _P], ctypes.c_int),
    "seq_alloc_prefix": ([_P, _P, _I32, _I32P], ctypes.c_int),
    "seq_accept_draft": ([_P, _I32, _I32, _P, _I32, _I32, _P, _I32P, _P], ctypes.c_int),
    "kvp_radix_create": ([_P, ctypes.POINTER(_P)], ctypes.c_int),
    "kvp_radix_destroy": ([_P], ctypes.c_int),
    "kvp_radix_match": ([_P, _P, _I32, _P, _I32, _I32P, _I32P], ctypes.c_int),
    "kvp_radix_unlock": ([_P, _I32], ctypes.c_int),
    "kvp_radix_insert": ([_P, _P, _I32, _P, _I32], ctypes.c_int),
    "kvp_radix_evict": ([_P, _I32, _I32P], ctypes.c_int),
    "kvp_radix_dump": ([_P, _P, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
}


def load():
    """Load libkvp.so (raises KvpError-compatible RuntimeError if not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise RuntimeError(f"libkvp.so is not built ({lib_path}); run "
                               "`python -m paged_prefix_shared_decode_gb300.build`")
        lib = ctypes.CDLL(lib_path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(rc, what):
    if rc != KVP_OK:
        raise KvpError(rc, what)


def _dev(x):
    """Device address of a torch CUDA tensor (or an int address / None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _host_i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data


# ------------------------------------------------------------------ pool

def kv_pool_create(desc: PoolDesc, k_storage=None, v_storage=None):
    h = _P()
    _check(load().kv_pool_create(ctypes.byref(desc), _dev(k_storage), _dev(v_storage), ctypes.byref(h)),
           "kv_pool_create")
    return h.value


def kv_pool_create_kv4(desc: PoolDesc, k_codes, k_exps, v_codes, v_exps):
    """A pool of 4-bit pages over caller storage: codes [L][NB][Hkv][bs][d/2]
    uint8 and exponents [L][NB][Hkv][bs] int8, for K and for V."""
    h = _P()
    _check(load().kv_pool_create_kv4(ctypes.byref(desc), _dev(k_codes), _dev(k_exps), _dev(v_codes),
                                     _dev(v_exps), ctypes.byref(h)), "kv_pool_create_kv4")
    return h.value


def kv_pool_destroy(pool):
    _check(load().kv_pool_destroy(pool), "kv_pool_destroy")


def seq_alloc(pool) -> int:
    s = _I32()
    _check(load().seq_alloc(pool, ctypes.byref(s)), "seq_alloc")
    return s.value


def seq_fork(pool, parent: int) -> int:
    s = _I32()
    _check(load().seq_fork(pool, parent, ctypes.byref(s)), "seq_fork")
    return s.value


def seq_free(pool, seq: int):
    _check(load().seq_free(pool, seq), "seq_free")


def seq_append(pool, seq: int, k, v, ntok: int, stream=None):
    _check(load().seq_append(pool, seq, _dev(k), _dev(v), ntok, _stream(stream)), "seq_append")


def seq_append_batch(pool, seqs, ntoks, k, v, stream=None):
    s, sp = _host_i32(seqs)
    n, np_ = _host_i32(ntoks)
    _check(load().seq_append_batch(pool, len(s), sp, np_, _dev(k), _dev(v), _stream(stream)),
           "seq_append_batch")


def seq_reserve(pool, seq: int, ntok: int):
    """Bookkeeping-only append: returns (slots int32 [ntok], cow int32 [3])."""
    slots = np.zeros(max(ntok, 1), np.int32)
    cow = np.zeros(3, np.int32)
    _check(load().seq_reserve(pool, seq, ntok, slots.ctypes.data, cow.ctypes.data),
           "seq_reserve")
    return slots[:ntok], cow


def seq_accept_draft(pool, seq: int, ctx_len: int, parent, accepted: int, stream=None) -> np.ndarray:
    """Keep the draft path from a root to `accepted` (-1: none) right after
    the context; returns the kept node ids, root first."""
    par, pp = _host_i32(parent)
    out = np.zeros(max(len(par), 1), np.int32)
    n = _I32()
    _check(load().seq_accept_draft(pool, seq, ctx_len, pp, len(par), accepted, out.ctypes.data,
                                   ctypes.byref(n), _stream(stream)), "seq_accept_draft")
    return out[:n.value]


def seq_alloc_prefix(pool, blocks) -> int:
    """A new sequence whose table is `blocks` (already held elsewhere, e.g. a
    prefix cache match) and whose length is len(blocks) * block_size."""
    b, bp = _host_i32(blocks)
    s = _I32()
    _check(load().seq_alloc_prefix(pool, bp, len(b), ctypes.byref(s)), "seq_alloc_prefix")
    return s.value


def seq_block_table(pool, seq: int) -> np.ndarray:
    n = _I32()
    _check(load().seq_block_table(pool, seq, None, 0, ctypes.byref(n)), "seq_block_table")
    out = np.zeros(max(n.value, 1), np.int32)
    _check(load().seq_block_table(pool, seq, out.ctypes.data, len(out), ctypes.byref(n)),
           "seq_block_table")
    return out[:n.value]


def seq_len(pool, seq: int) -> int:
    n = _I32()
    _check(load().seq_len(pool, seq, ctypes.byref(n)), "seq_len")
    return n.value


def block_refcount(pool, block: int) -> int:
    n = _I32()
    _check(load().block_refcount(pool, block, ctypes.byref(n)), "block_refcount")
    return n.value


def kvp_free_block_count(pool) -> int:
    n = _I32()
    _check(load().kvp_free_block_count(pool, ctypes.byref(n)), "kvp_free_block_count")
    return n.value


def kvp_cow_count(pool) -> int:
    n = ctypes.c_int64()
    _check(load().kvp_cow_count(pool, ctypes.byref(n)), "kvp_cow_count")
    return n.value


def kvp_gather_tables(pool, seqs, width: int):
    s, sp = _host_i32(seqs)
    t = np.empty((len(s), width), np.int32)   # rows are padded with -1 by the library
    lens = np.empty(len(s), np.int32)
    _check(load().kvp_gather_tables(pool, sp, len(s), width, t.ctypes.data,
                                    lens.ctypes.data), "kvp_gather_tables")
    return t, lens


def kvp_export_tables(pool, seqs, width: int, d_tables, d_lens=None, stream=None):
    s, sp = _host_i32(seqs)
    _check(load().kvp_export_tables(pool, sp, len(s), width, _dev(d_tables), _dev(d_lens),
                                    _stream(stream)), "kvp_export_tables")


# ------------------------------------------------------------- attention

def kvp_decode_workspace_size(desc: AttnDesc, h_tables, h_lens) -> int:
    t, tp = _host_i32(h_tables)
    ln, lp = _host_i32(h_lens)
    n = load().kvp_decode_workspace_size(ctypes.byref(desc), tp, lp, t.shape[0], t.shape[1])
    if n == 0:
        raise KvpError(KVP_ERR_INVALID, "kvp_decode_workspace_size")
    return n


def _ws_bytes(workspace, ws_bytes):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    return ws_bytes


def paged_decode_attention(q, k_pool, v_pool, block_tables, seq_lens, desc: AttnDesc, out, lse,
                           workspace, ws_bytes=None, stream=None):
    """block_tables [S][MB] / seq_lens [S]: host int32 arrays."""
    t, tp = _host_i32(block_tables)
    ln, lp = _host_i32(seq_lens)
    _check(load().paged_decode_attention(_dev(q), _dev(k_pool), _dev(v_pool), tp, lp, t.shape[0],
                                         t.shape[1], ctypes.byref(desc), _dev(out), _dev(lse),
                                         _dev(workspace), _ws_bytes(workspace, ws_bytes),
                                         _stream(stream)), "paged_decode_attention")


def paged_decode_attention_kv4(q, k_codes, k_exps, v_codes, v_exps, block_tables, seq_lens,
                               desc: AttnDesc, out, lse, workspace, ws_bytes=None, stream=None):
    """Decode attention over a pool of 4-bit pages (desc.kv_format = KVP_KV_4BIT)."""
    t, tp = _host_i32(block_tables)
    ln, lp = _host_i32(seq_lens)
    _check(load().paged_decode_attention_kv4(_dev(q), _dev(k_codes), _dev(k_exps), _dev(v_codes), _dev(v_exps),
                                             tp, lp, t.shape[0], t.shape[1], ctypes.byref(desc), _dev(out),
                                             _dev(lse), _dev(workspace), _ws_bytes(workspace, ws_bytes),
                                             _stream(stream)), "paged_decode_attention_kv4")


def paged_decode_attention_noalloc(q, k_pool, v_pool, block_tables, seq_lens, desc: AttnDesc, out,
                                   lse, stream=None):
    """paged_decode_attention without a caller workspace: for callers that
    cannot allocate device memory.  The library's own KVP_STATIC_WORKSPACE_BYTES
    array is used; calls on one device must not overlap."""
    t, tp = _host_i32(block_tables)
    ln, lp = _host_i32(seq_lens)
    _check(load().paged_decode_attention_noalloc(_dev(q), _dev(k_pool), _dev(v_pool), tp, lp, t.shape[0],
                                                 t.shape[1], ctypes.byref(desc), _dev(out), _dev(lse),
                                                 _stream(stream)), "paged_decode_attention_noalloc")


def kvp_pool_decode_workspace_size(pool, seq_ids, desc: AttnDesc) -> int:
    s, sp = _host_i32(seq_ids)
    n = load().kvp_pool_decode_workspace_size(pool, sp, len(s), ctypes.byref(desc))
    if n == 0:
        raise KvpError(KVP_ERR_INVALID, "kvp_pool_decode_workspace_size")
    return n


def paged_decode_attention_pool(pool, seq_ids, q, out, lse, desc: AttnDesc, workspace, ws_bytes=None,
                                stream=None):
    """Decode attention over pool sequences (tables read from the pool)."""
    s, sp = _host_i32(seq_ids)
    _check(load().paged_decode_attention_pool(pool, sp, len(s), _dev(q), _dev(out), _dev(lse),
                                              ctypes.byref(desc), _dev(workspace),
                                              _ws_bytes(workspace, ws_bytes), _stream(stream)),
           "paged_decode_attention_pool")


def _host(x):
    """Address of a host buffer: a CPU torch tensor (page-locked for
    asynchronous copies), a numpy array, an int address or None."""
    if x is None or isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("expected a contiguous array")
        return x.ctypes.data
    if x.is_cuda:
        raise ValueError("expected a host tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


def step_io(d_q, d_out, d_lse=None, d_k_new=None, d_v_new=None, h_k_new=None, h_v_new=None, h_q=None,
            h_out=None, h_lse=None, host_mapped=None) -> StepIO:
    """A kvp_step_io.  It holds raw addresses: keep the tensors alive while it
    is in use.  host_mapped (default: every host buffer given is a pinned
    torch tensor) sets KVP_STEP_HOST_MAPPED."""
    hosts = [x for x in (h_k_new, h_v_new, h_q, h_out, h_lse) if x is not None]
    if host_mapped is None:
        host_mapped = bool(hosts) and all(not isinstance(x, (int, np.ndarray)) and x.is_pinned() for x in hosts)
    return StepIO(_host(h_k_new), _host(h_v_new), _host(h_q), _host(h_out), _host(h_lse),
                  _dev(d_k_new), _dev(d_v_new), _dev(d_q), _dev(d_out), _dev(d_lse),
                  KVP_STEP_HOST_MAPPED if host_mapped else 0)


def kvp_decode_step(pool, seq_ids, ntok: int, io: StepIO, desc: AttnDesc, workspace, ws_bytes=None,
                    stream=None) -> int:
    """One decode step (copies in, append, attention, copies out) on
    `stream`; returns the workspace bytes the attention needed.  A
    KVP_ERR_WORKSPACE error carries them as .ws_needed."""
    s, sp = _host_i32(seq_ids)
    need = ctypes.c_size_t(0)
    rc = load().kvp_decode_step(pool, sp, len(s), ntok, ctypes.byref(io), ctypes.byref(desc), _dev(workspace),
                                _ws_bytes(workspace, ws_bytes), ctypes.byref(need), _stream(stream))
    if rc != KVP_OK:
        e = KvpError(rc, "kvp_decode_step")
        e.ws_needed = need.value
        raise e
    return need.value


class DecodeStep:
    """kvp_decode_step with its arguments marshalled once, for a loop that
    repeats the step on the same sequences and buffers: each call is then a
    single foreign call.  Keep `io`'s tensors alive while it is in use."""

    def __init__(self, pool, seq_ids, ntok: int, io: StepIO, desc: AttnDesc, workspace, ws_bytes=None,
                 stream=None):
        self._seqs = np.ascontiguousarray(seq_ids, dtype=np.int32)
        self._io, self._desc = io, desc
        self.ws_needed = ctypes.c_size_t(0)
        self._fn = load().kvp_decode_step
        self._args = (ctypes.c_void_p(pool), ctypes.c_void_p(self._seqs.ctypes.data), _I32(len(self._seqs)),
                      _I32(ntok), ctypes.byref(io), ctypes.byref(desc), ctypes.c_void_p(_dev(workspace)),
                      ctypes.c_size_t(_ws_bytes(workspace, ws_bytes)), ctypes.byref(self.ws_needed),
                      ctypes.c_void_p(_stream(stream)))

    def __call__(self) -> int:
        rc = self._fn(*self._args)
        if rc != KVP_OK:
            e = KvpError(rc, "kvp_decode_step")
            e.ws_needed = self.ws_needed.value
            raise e
        return self.ws_needed.value


def kvp_step_plan_create():
    h = load().kvp_step_plan_create()
    if not h:
        raise KvpError(KVP_ERR_OOM, "kvp_step_plan_create")
    return h


def kvp_step_plan_destroy(plan) -> None:
    load().kvp_step_plan_destroy(plan)


def kvp_decode_step_plan(pool, seq_ids, ntok: int, desc: AttnDesc, plan) -> int:
    """Host half of a decode step (the append's bookkeeping and the attention
    plan over the grown sequences) into `plan`; returns the workspace bytes
    its run needs."""
    s, sp = _host_i32(seq_ids)
    need = ctypes.c_size_t(0)
    _check(load().kvp_decode_step_plan(pool, sp, len(s), ntok, ctypes.byref(desc), plan, ctypes.byref(need)),
           "kvp_decode_step_plan")
    return need.value


def kvp_decode_step_run(plan, io: StepIO, workspace, ws_bytes=None, stream=None) -> None:
    """Device half of a planned decode step on `stream`."""
    _check(load().kvp_decode_step_run(plan, ctypes.byref(io), _dev(workspace), _ws_bytes(workspace, ws_bytes),
                                      _stream(stream)), "kvp_decode_step_run")


class StepPlan:
    """kvp_decode_step_plan / kvp_decode_step_run on one plan object with
    their arguments marshalled once: plan() is the host half of the next
    step, run() its device half.  A loop can plan step i + 1 right after
    running step i, while the device works.  Keep `io`'s tensors alive while
    it is in use; close() frees the plan object."""

    def __init__(self, pool, seq_ids, ntok: int, io: StepIO, desc: AttnDesc, workspace, ws_bytes=None,
                 stream=None):
        lib = load()
        self._seqs = np.ascontiguousarray(seq_ids, dtype=np.int32)
        self._io, self._desc = io, desc
        self._h = kvp_step_plan_create()
        self.ws_needed = ctypes.c_size_t(0)
        self._plan, self._run, self._destroy = lib.kvp_decode_step_plan, lib.kvp_decode_step_run, \
            lib.kvp_step_plan_destroy
        h = ctypes.c_void_p(self._h)
        self._pargs = (ctypes.c_void_p(pool), ctypes.c_void_p(self._seqs.ctypes.data), _I32(len(self._seqs)),
                       _I32(ntok), ctypes.byref(desc), h, ctypes.byref(self.ws_needed))
        self._rargs = (h, ctypes.byref(io), ctypes.c_void_p(_dev(workspace)),
                       ctypes.c_size_t(_ws_bytes(workspace, ws_bytes)), ctypes.c_void_p(_stream(stream)))

    def plan(self) -> int:
        _check(self._plan(*self._pargs), "kvp_decode_step_plan")
        return self.ws_needed.value

    def run(self) -> None:
        _check(self._run(*self._rargs), "kvp_decode_step_run")

    def close(self) -> None:
        if self._h:
            self._destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kvp_verify_workspace_size(desc: AttnDesc, block_tables, ctx_lens, n_draft: int) -> int:
    t, tp = _host_i32(block_tables)
    c, cp = _host_i32(ctx_lens)
    n = load().kvp_verify_workspace_size(ctypes.byref(desc), tp, cp, len(c), n_draft, t.shape[1])
    if n == 0:
        raise KvpError(KVP_ERR_INVALID, "kvp_verify_workspace_size")
    return n


def tree_verify_attention(q, tree_parent, n_draft: int, k_pool, v_pool, block_tables, ctx_lens,
                          desc: AttnDesc, out, lse, workspace, ws_bytes=None, stream=None):
    """tree_parent: device int32 [B][n]; block_tables [B][MB] / ctx_lens [B]: host."""
    t, tp = _host_i32(block_tables)
    c, cp = _host_i32(ctx_lens)
    _check(load().tree_verify_attention(_dev(q), _dev(tree_parent), n_draft, _dev(k_pool), _dev(v_pool),
                                        tp, cp, len(c), t.shape[1], ctypes.byref(desc), _dev(out),
                                        _dev(lse), _dev(workspace), _ws_bytes(workspace, ws_bytes),
                                        _stream(stream)), "tree_verify_attention")


def kvp_device_error(workspace, stream=None) -> int:
    e = _I32()
    _check(load().kvp_device_error(_dev(workspace), _stream(stream), ctypes.byref(e)), "kvp_device_error")
    return e.value


def kvp_decode_plan_stats(desc: AttnDesc, h_tables, h_lens, sm_count: int = 152) -> dict:
    t, tp = _host_i32(h_tables)
    ln, lp = _host_i32(h_lens)
    vals = [_I32() for _ in range(4)]
    ub = ctypes.c_int64()
    _check(load().kvp_decode_plan_stats(ctypes.byref(desc), tp, lp, t.shape[0], t.shape[1], sm_count,
                                        *[ctypes.byref(v) for v in vals], ctypes.byref(ub)),
           "kvp_decode_plan_stats")
    return dict(items=vals[0].value, row_tiles=vals[1].value, kv_tiles=vals[2].value,
                partial_rows=vals[3].value, unique_kv_bytes=ub.value)


def kvp_set_kernel_events(before=None, after=None):
    """before/after: torch.cuda.Event (recorded once already) or raw handles."""
    def h(e):
        if e is None:
            return None
        return e if isinstance(e, int) else e.cuda_event
    _check(load().kvp_set_kernel_events(h(before), h(after)), "kvp_set_kernel_events")


def kvp_kernel_launches() -> int:
    n = ctypes.c_int64()
    _check(load().kvp_kernel_launches(ctypes.byref(n)), "kvp_kernel_launches")
    return n.value


def kvp_strerror(code: int) -> str:
    return load().kvp_strerror(code).decode()


# ---------------------------------------------------------- prefix cache

def kvp_radix_create(pool):
    h = _P()
    _check(load().kvp_radix_create(pool, ctypes.byref(h)), "kvp_radix_create")
    return h.value


def kvp_radix_destroy(cache):
    _check(load().kvp_radix_destroy(cache), "kvp_radix_destroy")


def kvp_radix_match(cache, tokens):
    """(block ids of the longest cached prefix, lock); lock -1 when none."""
    t, tp = _host_i32(tokens)
    out = np.zeros(max(len(t), 1), np.int32)   # at least n_tokens / block_size
    n, lock = _I32(), _I32()
    _check(load().kvp_radix_match(cache, tp, len(t), out.ctypes.data, len(out), ctypes.byref(n),
                                  ctypes.byref(lock)), "kvp_radix_match")
    return out[:n.value], lock.value


def kvp_radix_unlock(cache, lock: int):
    _check(load().kvp_radix_unlock(cache, lock), "kvp_radix_unlock")


def kvp_radix_insert(cache, tokens, blocks):
    t, tp = _host_i32(tokens)
    b, bp = _host_i32(blocks)
    _check(load().kvp_radix_insert(cache, tp, len(t), bp, len(b)), "kvp_radix_insert")


def kvp_radix_evict(cache, need_free: int):
    """(met, blocks returned to the pool)."""
    freed = _I32()
    rc = load().kvp_radix_evict(cache, need_free, ctypes.byref(freed))
    if rc not in (KVP_OK, KVP_ERR_OOM):
        _check(rc, "kvp_radix_evict")
    return rc == KVP_OK, freed.value


def kvp_radix_dump(cache):
    """Canonical tree: [(depth, tokens, blocks, locks, stamp)] depth first,
    children in increasing order of their first block's tokens."""
    n = ctypes.c_int64()
    load().kvp_radix_dump(cache, None, 0, ctypes.byref(n))   # sizes the buffer
    w = np.zeros(max(n.value, 1), np.int32)
    _check(load().kvp_radix_dump(cache, w.ctypes.data, len(w), ctypes.byref(n)), "kvp_radix_dump")
    out, i = [], 0
    w = w[:n.value].tolist()
    while i < len(w):
        depth, locks, stamp, nt = w[i:i + 4]
        toks = tuple(w[i + 4:i + 4 + nt])
        nb = w[i + 4 + nt]
        blks = tuple(w[i + 5 + nt:i + 5 + nt + nb])
        out.append((depth, toks, blks, locks, stamp))
        i += 5 + nt + nb
    return out
