"""GPU parity: tree-verify attention through the C ABI against the fp64 oracle
on draft trees of 64 nodes over paged 2048-token contexts (Llama-3-8B head
shapes), plus chain / star / forest trees and a bad parent pointer."""
import numpy as np
import pytest

import oracle
import workloads as W
from _util import (MAX_ABS, bf16_absmax, check_close, check_lse, oracle_side, peaked_max_abs,
                   sample_triples, to_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_prefix_shared_decode_gb300 as kvp  # noqa: E402
from paged_prefix_shared_decode_gb300.runner import PoolRunner, VerifyCall, bf16_tensor  # noqa: E402


def run_verify(w, alloc_seed=1, samples=None, parents=None, q_scale=1.0):
    if parents is not None:
        w.info["parents"] = np.ascontiguousarray(parents, np.int32)
    r = PoolRunner(w, alloc_seed=alloc_seed)
    r.run_ops()
    call = VerifyCall(r)
    q = W.verify_q(w, scale=q_scale)
    call(bf16_tensor(q))
    torch.cuda.synchronize()
    rw = oracle_side(w, alloc_seed)
    t, ln = rw.tables(w.batch, w.max_blocks_per_seq)
    assert np.array_equal(t, call.h_tables)
    ctx = ln - w.info["n_draft"]
    if samples is None:
        want_o, want_l = oracle.verify_attention(q, rw.k_pool, rw.v_pool, t, ctx, w.info["parents"])
        got_o, got_l = to_f64(call.out), to_f64(call.lse)
    else:
        want_o, want_l = oracle.verify_attention(q, rw.k_pool, rw.v_pool, t, ctx, w.info["parents"],
                                                 samples=samples)
        o, ls = call.out.float().cpu().numpy(), call.lse.cpu().numpy()
        got_o = np.stack([o[l, s, h] for l, s, h in samples]).astype(np.float64)
        got_l = np.array([ls[l, s, h] for l, s, h in samples], np.float64)
    tol = MAX_ABS if q_scale == 1.0 else peaked_max_abs(want_o, bf16_absmax(rw.v_pool))
    check_close(got_o, want_o, max_abs_tol=tol)
    check_lse(got_l, want_l)
    assert kvp.kvp_device_error(call.ws) == 0
    return r, call


def test_verify_B1_full():
    run_verify(W.verify_tree(1, layers=2))


def test_verify_B8_sampled():
    w = W.verify_tree(8, layers=2)
    run_verify(w, samples=sample_triples(np.random.default_rng(1), 2, 8 * 64, 32, 800))


def test_verify_B32_sampled():
    w = W.verify_tree(32, layers=1)
    run_verify(w, samples=sample_triples(np.random.default_rng(2), 1, 32 * 64, 32, 800))


def test_verify_peaked_queries():
    run_verify(W.verify_tree(1, layers=1), q_scale=4.0)


@pytest.mark.parametrize("kind", ["chain", "star", "forest"])
def test_verify_tree_shapes(kind):
    n = 64
    if kind == "chain":
        par = np.arange(-1, n - 1)
    elif kind == "star":
        par = np.array([-1] + [0] * (n - 1))
    else:
        par = np.array([-1 if i % 8 == 0 else i - 1 for i in range(n)])
    w = W.verify_tree(2, layers=1, ctx=300)
    run_verify(w, parents=np.stack([par, par]))


def test_verify_short_draft_and_tinyllama_shapes():
    sh = W.Shapes(L=1, Hq=32, Hkv=4, d=64, bs=16)
    ops = [("alloc", 0), ("append", 0, 77), ("append", 0, 13)]
    w = W.Workload("v", sh, ops, batch=[0], step_tokens=0,
                   info=dict(ctx=77, n_draft=13, parents=np.array([W.draft_tree(5, 13)])))
    run_verify(W._finish(w))


def test_verify_bad_parent_sets_error_word():
    w = W.verify_tree(1, layers=1, ctx=100)
    par = W.draft_tree(0).copy()
    par[10] = 12                      # not an earlier node
    w.info["parents"] = par[None]
    r = PoolRunner(w)
    r.run_ops()
    call = VerifyCall(r)
    call(bf16_tensor(W.verify_q(w)))
    assert kvp.kvp_device_error(call.ws) == 2


def growing_kv(w, i):
    """Keys of the context's second half scaled 30x: a later step's scores
    exceed the running max of the earlier steps by far more than the kernel's
    headroom (p would overflow fp32), so its rescale-and-recompute path runs."""
    k, v = W.append_kv(w, i)
    ntok = w.ops[i][2]
    if ntok > w.info["n_draft"]:
        kf = W.bf16_bits_to_f32(k)
        kf[:, ntok // 2:] *= 30.0
        k = W.f32_to_bf16_bits(kf)
    return k, v


def test_verify_growing_scores():
    w = W.verify_tree(1, layers=1)
    r = PoolRunner(w, alloc_seed=1)
    r.run_ops(kv_fn=growing_kv)
    call = VerifyCall(r)
    q = W.verify_q(w)
    call(bf16_tensor(q))
    torch.cuda.synchronize()
    rw = oracle.replay(w, alloc_seed=1, kv_fn=growing_kv)
    t, ln = rw.tables(w.batch, w.max_blocks_per_seq)
    ctx = ln - w.info["n_draft"]
    want_o, want_l = oracle.verify_attention(q, rw.k_pool, rw.v_pool, t, ctx, w.info["parents"])
    check_close(to_f64(call.out), want_o, max_abs_tol=peaked_max_abs(want_o, bf16_absmax(rw.v_pool)))
    check_lse(to_f64(call.lse), want_l)
    assert kvp.kvp_device_error(call.ws) == 0


def test_verify_output_16_byte_aligned():
    # An output only 16-byte aligned (the documented minimum) takes the
    # tcgen05 epilogue's 16-byte stores instead of its 32-byte ones: same bits.
    w = W.verify_tree(2, layers=1)
    r, call = run_verify(w)
    ref_o, ref_l = call.out.clone(), call.lse.clone()
    buf = torch.empty(call.out.numel() + 8, dtype=torch.bfloat16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    off = buf[8:].view(call.out.shape)   # 16 bytes past a 32-byte boundary
    q = bf16_tensor(W.verify_q(w))
    kvp.tree_verify_attention(q, call.parent, call.n, r.k_pool, r.v_pool, call.h_tables, call.ctx, call.desc,
                              off, call.lse, call.ws)
    torch.cuda.synchronize()
    assert torch.equal(off.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(call.lse, ref_l)


def test_verify_partly_filled_pair_unit():
    # 40 draft nodes x G 4 = 160 query rows: a pair unit whose second 128-row
    # tile holds 32 rows (its Q boxes past the members read zeros; that
    # tile's output rows are written row by row), over a context that ends
    # inside a block
    run_verify(W.verify_tree(2, layers=1, ctx=1000, n_draft=40))
