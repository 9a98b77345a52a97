"""GPU parity: paged decode attention through the C ABI against the fp64 oracle,
on the workloads' shapes (tiny fork, Dendrite at full size in the benchmark's
launch configuration, the Trellis phi sweep, the MCTS tree) and edge cases.
Block tables and refcounts are compared bit-exactly with the oracle model."""
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
from paged_prefix_shared_decode_gb300.runner import (PoolRunner, DecodeCall, bf16_tensor)  # noqa: E402


def run_decode(w, alloc_seed=1, steps=1, use_sharing=True, q_scale=1.0, poison=False, samples=None):
    """Replay w on both sides, run `steps` decode steps (append, then attend),
    compare the last step's outputs.  Returns (runner, call, rw)."""
    r = PoolRunner(w, alloc_seed=alloc_seed, poison=poison)
    r.run_ops()
    call = DecodeCall(r, use_sharing=use_sharing)
    steps_kv = []
    for st in range(steps):
        if w.step_tokens:
            k, v = W.step_kv(w, st)
            steps_kv.append((k, v))
            r.append_step(bf16_tensor(k), bf16_tensor(v))
        q = W.step_q(w, st, scale=q_scale)
        call.refresh()
        call(bf16_tensor(q))
    torch.cuda.synchronize()
    rw = oracle_side(w, alloc_seed, steps_kv)
    # bookkeeping is bit-exact
    t_model, l_model = rw.tables(w.batch, w.max_blocks_per_seq)
    assert np.array_equal(call.h_tables, t_model)
    assert np.array_equal(call.h_lens, l_model)
    ref = [kvp.block_refcount(r.pool, b) for b in range(w.num_blocks)]
    assert ref == rw.model.ref
    if samples is None:
        want_o, want_l = oracle.decode_attention(q, rw.k_pool, rw.v_pool, t_model, l_model)
        got_o, got_l = to_f64(call.out), to_f64(call.lse)
    else:
        want_o, want_l = oracle.decode_attention(q, rw.k_pool, rw.v_pool, t_model, l_model,
                                                 samples=samples)
        o, ls = call.out.float().cpu().numpy(), call.lse.cpu().numpy()
        got_o = np.stack([o[l, s, h] for l, s, h in samples]).astype(np.float64)
        got_l = np.array([ls[l, s, h] for l, s, h in samples], np.float64)
    tol = MAX_ABS if q_scale == 1.0 else peaked_max_abs(want_o, bf16_absmax(rw.v_pool))
    check_close(got_o, want_o, max_abs_tol=tol)
    check_lse(got_l, want_l)
    assert kvp.kvp_device_error(call.ws) == 0
    return r, call, rw


@pytest.mark.parametrize("use_sharing", [True, False])
@pytest.mark.parametrize("alloc_seed", [0, 1])
def test_tiny_fork(use_sharing, alloc_seed):
    run_decode(W.tiny_fork(), alloc_seed=alloc_seed, use_sharing=use_sharing)


def test_tiny_fork_peaked_query():
    run_decode(W.tiny_fork(), q_scale=4.0)


def test_dendrite_full_size_bench_configuration():
    """22 layers, 4096-token prefix, 6 branches, two decode steps, exactly the
    calls bench.py times; every output compared."""
    run_decode(W.dendrite(), steps=2)


def test_dendrite_sharing_equals_no_sharing():
    w = W.dendrite(layers=2)
    _, c1, _ = run_decode(w, use_sharing=True)
    _, c2, _ = run_decode(w, use_sharing=False)
    d = (c1.out.float() - c2.out.float()).abs().max().item()
    assert d <= 1e-2


@pytest.mark.parametrize("phi", [0.0, 0.25, 0.5, 0.75, 0.9])
def test_trellis_phi_sweep(phi):
    run_decode(W.trellis(phi, layers=3))


def test_mcts_tree_sampled():
    w = W.mcts(layers=2)
    rng = np.random.default_rng(0)
    samples = sample_triples(rng, 2, len(w.batch), 32, 600)
    run_decode(w, samples=samples)


def test_mcts_one_layer_full():
    run_decode(W.mcts(layers=1, depth=3))


def _custom(lens_private, prefix, bs=16, Hq=32, Hkv=8, d=128, layers=2, seed=3, step_tokens=1):
    sh = W.Shapes(L=layers, Hq=Hq, Hkv=Hkv, d=d, bs=bs)
    ops = [("alloc", 0)]
    if prefix:
        ops.append(("append", 0, prefix))
    batch = []
    for i, u in enumerate(lens_private):
        ops.append(("fork", 0, i + 1))
        if u:
            ops.append(("append", i + 1, u))
        batch.append(i + 1)
    w = W.Workload("custom", sh, ops, batch=batch, seed=seed, step_tokens=step_tokens)
    return W._finish(w)


@pytest.mark.parametrize("bs", [16, 32])
def test_ragged_lengths_and_tiles(bs):
    # lengths that end mid-block and mid-tile, one single-token sequence,
    # a fork with nothing private; several tiles and a ragged tail
    w = _custom([0, 1, 5, 63, 64, 65, 200, 333], prefix=130, bs=bs, step_tokens=0)
    w.ops.append(("alloc", 99)); w.ops.append(("append", 99, 1)); w.batch.append(99)
    w.num_blocks = w.max_seqs = w.max_blocks_per_seq = 0
    w = W._finish(w)
    run_decode(w)


def test_cow_of_shared_partial_block_on_device():
    # prefix 250 ends mid-block; every child's first append copies it
    w = _custom([3, 17, 0, 40], prefix=250, Hq=8, Hkv=2, d=64)
    r, call, rw = run_decode(w, steps=2, poison=True)
    assert kvp.kvp_cow_count(r.pool) == rw.model.cow_copies >= 3
    # device pool contents of every live block equal the oracle's host pool
    kp = r.k_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    vp = r.v_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    for s in rw.model.live():
        n = rw.model.length(s)
        for j, b in enumerate(rw.model.table(s)):
            used = min(16, n - j * 16)
            assert np.array_equal(kp[:, b, :, :used], rw.k_pool[:, b, :, :used])
            assert np.array_equal(vp[:, b, :, :used], rw.v_pool[:, b, :, :used])


def test_gqa_group_16_and_single_sequence():
    w = _custom([70], prefix=0, Hq=32, Hkv=2, d=64, layers=1)
    run_decode(w)


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 8, 64), (8, 4, 128), (12, 2, 64), (32, 2, 128), (24, 8, 128)])
def test_gqa_groups_with_split_prefix(Hq, Hkv, d):
    """Query-head groups of 1, 2 and 16 (merged a whole group per warp) and of
    6 and 3 (merged one head per warp), with a prefix long enough to be split
    into many key ranges, so a query merges many partial rows."""
    w = _custom([5, 0, 77], prefix=3000, Hq=Hq, Hkv=Hkv, d=d, layers=1)
    run_decode(w)


def test_fork_child_without_private_tokens_equals_parent():
    w = _custom([0, 0], prefix=300, step_tokens=0)
    w.batch = [0, 1, 2]
    r, call, _ = run_decode(w)
    q = W.step_q(w, 0)
    qq = np.repeat(q[:, :1], 3, axis=1)                # same query for all three
    call(bf16_tensor(qq))
    torch.cuda.synchronize()
    o = call.out.float()
    assert torch.equal(o[:, 0], o[:, 1]) and torch.equal(o[:, 0], o[:, 2])


def test_empty_sequence_and_bad_tables_are_rejected():
    w = _custom([4], prefix=20, step_tokens=0)
    r = PoolRunner(w)
    r.run_ops()
    call = DecodeCall(r)
    call.refresh()
    q = bf16_tensor(W.step_q(w, 0))
    lens = call.h_lens.copy(); lens[0] = 0
    with pytest.raises(kvp.KvpError) as e:
        kvp.paged_decode_attention(q, r.k_pool, r.v_pool, call.h_tables, lens,
                                   call.desc, call.out, call.lse, call.ws)
    assert e.value.code == kvp.KVP_ERR_INVALID
    bad = call.h_tables.copy(); bad[0, 0] = r.NB
    with pytest.raises(kvp.KvpError):
        kvp.paged_decode_attention(q, r.k_pool, r.v_pool, bad, call.h_lens,
                                   call.desc, call.out, call.lse, call.ws)
    with pytest.raises(kvp.KvpError):      # workspace too small
        kvp.paged_decode_attention(q, r.k_pool, r.v_pool, call.h_tables, call.h_lens,
                                   call.desc, call.out, call.lse, call.ws, ws_bytes=256)
    import ctypes
    d = kvp.AttnDesc(call.desc.num_layers, 32, 8, 128, 24, r.NB, 0.0, 1)   # bs not a power of 2
    with pytest.raises(kvp.KvpError):
        kvp.paged_decode_attention(q, r.k_pool, r.v_pool, call.h_tables, call.h_lens,
                                   d, call.out, call.lse, call.ws)


def test_repeated_calls_and_error_word_clean():
    """The workspace's atomic work counter and error word are reset by every
    call's plan upload: back-to-back calls give identical results."""
    w = _custom([10, 3], prefix=40, step_tokens=0)
    r = PoolRunner(w)
    r.run_ops()
    call = DecodeCall(r)
    call.refresh()
    q = bf16_tensor(W.step_q(w, 0))
    call(q)
    first = call.out.clone()
    for _ in range(3):
        call(q)
    torch.cuda.synchronize()
    assert torch.equal(first, call.out)
    assert kvp.kvp_device_error(call.ws) == 0
