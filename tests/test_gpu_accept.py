"""GPU parity of speculative accept after tree verify: on verify-shaped
sequences (2048-token contexts, 64-node draft trees, Llama-3-8B head shapes,
block 16), `seq_accept_draft` on the device pool against the oracle model on
its host pool, bit-exact on K and V of every live token of every live
sequence, including forked siblings whose shared blocks are copied before a
token moves into them; then decode attention over the compacted batch
against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from _util import check_close, check_lse, oracle_side, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_prefix_shared_decode_gb300 as kvp  # noqa: E402
from paged_prefix_shared_decode_gb300.runner import PoolRunner, DecodeCall, bf16_tensor  # noqa: E402


def host_pool(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("seed", [0, 1])
def test_accept_bit_exact_then_decode(seed):
    w = W.verify_tree(8, layers=2)
    w.num_blocks += 64       # room for the copies
    w.max_seqs += 4          # and the siblings
    r = PoolRunner(w, alloc_seed=1)
    r.run_ops()
    rw = oracle_side(w, 1)
    parents = w.info["parents"]
    n = w.info["n_draft"]
    bs = w.shapes.bs
    rng = np.random.default_rng(seed)
    # siblings of the first three sequences share all their blocks
    for nm in w.batch[:3]:
        assert rw.model.fork(rw.ids[nm]) == kvp.seq_fork(r.pool, r.ids[nm])
    accepted = [int(rng.integers(-1, n)) for _ in w.batch]
    accepted[0] = n - 1          # a deep node in a shared sequence: moves into copied blocks
    for b, nm in enumerate(w.batch):
        sm, sl = rw.ids[nm], r.ids[nm]
        ctx = rw.model.length(sm) - n
        pm = rw.model.accept_draft(sm, ctx, [int(x) for x in parents[b]], accepted[b])
        pl = kvp.seq_accept_draft(r.pool, sl, ctx, parents[b], accepted[b])
        assert list(pl) == pm
    torch.cuda.synchronize()
    assert kvp.kvp_cow_count(r.pool) == rw.model.cow_copies
    kp, vp = host_pool(r.k_pool), host_pool(r.v_pool)
    for s in rw.model.live():
        table = rw.model.table(s)
        assert list(kvp.seq_block_table(r.pool, s)) == table
        length = rw.model.length(s)
        assert kvp.seq_len(r.pool, s) == length
        for j, blk in enumerate(table):
            used = min(bs, length - j * bs)
            assert np.array_equal(kp[:, blk, :, :used], rw.k_pool[:, blk, :, :used])
            assert np.array_equal(vp[:, blk, :, :used], rw.v_pool[:, blk, :, :used])
    for blk in range(w.num_blocks):
        assert kvp.block_refcount(r.pool, blk) == rw.model.refcount(blk)
    # decode attention over the compacted sequences
    call = DecodeCall(r)
    call.refresh()
    q = W.step_q(w, 0)
    call(bf16_tensor(q))
    torch.cuda.synchronize()
    t, ln = rw.tables(w.batch, w.max_blocks_per_seq)
    assert np.array_equal(t, call.h_tables) and np.array_equal(ln, call.h_lens)
    want_o, want_l = oracle.decode_attention(q, rw.k_pool, rw.v_pool, t, ln)
    check_close(to_f64(call.out), want_o)
    check_lse(to_f64(call.lse), want_l)
    assert kvp.kvp_device_error(call.ws) == 0
