"""The C ABI library loads without a GPU and exports every symbol that
include/kvp.h declares; error codes map to messages."""
import ctypes

import numpy as np
import os
import re

import pytest

import paged_prefix_shared_decode_gb300 as kvp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, re.M):
            if m.group(1) not in ("if", "while", "for", "sizeof", "return"):
                names.append(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for must in ("kv_pool_create", "seq_alloc", "seq_fork", "seq_append", "seq_free",
                 "paged_decode_attention", "tree_verify_attention"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(kvp.load()._name)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_exposes_same_names():
    missing = [n for n in declared_functions() if not hasattr(kvp, n)]
    assert not missing, missing


def test_strerror_and_invalid_arguments():
    assert kvp.kvp_strerror(kvp.KVP_ERR_OOM) == "out of blocks or sequence slots"
    lib = kvp.load()
    assert lib.kv_pool_create(None, None, None, None) == kvp.KVP_ERR_INVALID
    assert lib.seq_alloc(None, None) == kvp.KVP_ERR_INVALID
    d = kvp.PoolDesc(1, 4, 16, 1, 12, 2, 2, 0)          # head_dim not a multiple of 8
    with pytest.raises(kvp.KvpError):
        kvp.kv_pool_create(d)


def test_bookkeeping_pool_refuses_device_appends():
    p = kvp.kv_pool_create(kvp.PoolDesc(1, 8, 16, 1, 8, 2, 4, 0))
    s = kvp.seq_alloc(p)
    with pytest.raises(kvp.KvpError) as e:
        kvp.seq_append(p, s, 0, 0, 1, stream=0)
    assert e.value.code == kvp.KVP_ERR_STATE
    kvp.kv_pool_destroy(p)


def test_kv4_pool_and_descriptor_checks():
    # a 4-bit pool needs d 64 or 128, blocks of a multiple of 16 tokens and
    # four 16-byte aligned arrays; nothing is touched on the device here
    a = 1 << 20   # any 16-byte aligned address: pool creation only records it
    for d, bs in ((64, 16), (128, 32)):
        p = kvp.kv_pool_create_kv4(kvp.PoolDesc(1, 8, bs, 2, d, 2, 4, 0), a, a, a, a)
        kvp.kv_pool_destroy(p)
    for d, bs in ((96, 16), (64, 8), (32, 16)):
        with pytest.raises(kvp.KvpError):
            kvp.kv_pool_create_kv4(kvp.PoolDesc(1, 8, bs, 2, d, 2, 4, 0), a, a, a, a)
    with pytest.raises(kvp.KvpError):
        kvp.kv_pool_create_kv4(kvp.PoolDesc(1, 8, 16, 2, 64, 2, 4, 0), a, a + 8, a, a)
    with pytest.raises(kvp.KvpError):
        kvp.kv_pool_create_kv4(kvp.PoolDesc(1, 8, 16, 2, 64, 2, 4, 0), a, 0, a, a)
    # the 4-bit descriptor is refused by the bf16 entry points and vice versa
    t = np.zeros((1, 1), np.int32)
    ln = np.ones(1, np.int32)
    d4 = kvp.AttnDesc(1, 4, 2, 64, 16, 8, 0.0, 1, kvp.KVP_KV_4BIT)
    d16 = kvp.AttnDesc(1, 4, 2, 64, 16, 8, 0.0, 1, kvp.KVP_KV_BF16)
    assert kvp.kvp_decode_workspace_size(d4, t, ln) > 0
    with pytest.raises(kvp.KvpError):
        kvp.paged_decode_attention(a, a, a, t, ln, d4, a, a, a, 1 << 20, stream=0)
    with pytest.raises(kvp.KvpError):
        kvp.paged_decode_attention_kv4(a, a, a, a, a, t, ln, d16, a, a, a, 1 << 20, stream=0)
    bad = kvp.AttnDesc(1, 4, 2, 64, 16, 8, 0.0, 1, 7)   # no such page format
    with pytest.raises(kvp.KvpError):
        kvp.kvp_decode_workspace_size(bad, t, ln)


def test_pool_decode_entry_points_on_the_host():
    # tables read from the pool plan exactly like host tables of the same
    # sequences; argument and state errors come back before any device work
    p = kvp.kv_pool_create(kvp.PoolDesc(2, 64, 16, 2, 64, 8, 16, 3))
    root = kvp.seq_alloc(p)
    kvp.seq_reserve(p, root, 100)
    kids = [kvp.seq_fork(p, root) for _ in range(3)]
    for i, k in enumerate(kids):
        kvp.seq_reserve(p, k, 5 + 17 * i)
    seqs = [root] + kids
    desc = kvp.AttnDesc(2, 8, 2, 64, 16, 64, 0.0, 1)
    t, ln = kvp.kvp_gather_tables(p, seqs, 16)
    assert kvp.kvp_pool_decode_workspace_size(p, seqs, desc) == kvp.kvp_decode_workspace_size(desc, t, ln)
    for bad in (kvp.AttnDesc(2, 8, 2, 64, 16, 63, 0.0, 1),            # block count differs
                kvp.AttnDesc(1, 8, 2, 64, 16, 64, 0.0, 1),            # layers differ
                kvp.AttnDesc(2, 8, 2, 64, 16, 64, 0.0, 1, kvp.KVP_KV_4BIT)):
        with pytest.raises(kvp.KvpError):
            kvp.kvp_pool_decode_workspace_size(p, seqs, bad)
    with pytest.raises(kvp.KvpError):
        kvp.kvp_pool_decode_workspace_size(p, seqs + [7], desc)     # not a live sequence
    a = 1 << 20
    io = kvp.StepIO(None, None, None, None, None, a, a, a, a, a)
    with pytest.raises(kvp.KvpError) as e:                           # no device storage
        kvp.kvp_decode_step(p, seqs, 1, io, desc, a, 1 << 20, stream=0)
    assert e.value.code == kvp.KVP_ERR_STATE
    io_bad = kvp.StepIO(None, None, None, None, None, a, a, a + 8, a, a)   # misaligned q
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step(p, seqs, 1, io_bad, desc, a, 1 << 20, stream=0)
    assert e.value.code == kvp.KVP_ERR_INVALID
    assert [kvp.seq_len(p, s) for s in seqs] == list(ln)              # nothing changed
    assert kvp.kvp_strerror(kvp.KVP_ERR_WORKSPACE) == "workspace too small"
    kvp.kv_pool_destroy(p)
