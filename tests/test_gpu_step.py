"""The pool-table entry points on the GPU:

- kvp_decode_step from host buffers (page-locked torch tensors through the
  prepared DecodeStep call, crossing in copy kernels or copy-engine
  transfers, and pageable numpy arrays): the pool's tables, lengths and copy-on-write count follow the
  oracle's pool model, and out / lse match the fp64 oracle over the model's
  host K/V store, step after step, on a forked batch whose first appends copy
  a shared partial block;
- paged_decode_attention_pool and kvp_decode_step give the same bits as
  paged_decode_attention on host tables gathered from the same pool (the same
  plan and kernels), for bf16 and 4-bit pages;
- a too-small workspace returns KVP_ERR_WORKSPACE with the size needed after
  the append, and paged_decode_attention_pool finishes the step; an append
  that does not fit returns KVP_ERR_OOM with the pool unchanged;
- a step too large for the one-kernel input path (more than 64 appended
  tokens, or a plan image above 24 KB) takes the copy kernel, plan upload and
  write kernel instead, with the same results;
- the step in two halves (kvp_decode_step_plan, kvp_decode_step_run): a
  planned-then-run step gives the same bits as the host-table entry point,
  a loop that plans step i + 1 while the device runs step i follows the
  oracle step after step, and the plan object's states (run before plan,
  plan twice, a short workspace) give the documented errors."""
import numpy as np
import pytest

import oracle
import workloads as W
from _util import check_close, check_lse, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_prefix_shared_decode_gb300 as kvp  # noqa: E402
from paged_prefix_shared_decode_gb300.runner import bf16_tensor  # noqa: E402

L, HQ, HKV, D, BS = 2, 32, 4, 64, 16


def host_bf16(bits, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pinned else t


class Pool:
    """A device pool (bf16 or 4-bit pages) and the oracle's pool model with a
    host K/V store, driven in lockstep."""

    def __init__(self, nb=96, kv4=False, seqs=16, mb=32, seed=4):
        self.nb, self.mb, self.kv4 = nb, mb, kv4
        shape = (L, nb, HKV, BS, D)
        desc = kvp.PoolDesc(L, nb, BS, HKV, D, seqs, mb, seed)
        if kv4:
            self.kp = torch.zeros((L, nb, HKV, BS, D // 2), dtype=torch.uint8, device="cuda")
            self.vp = torch.zeros_like(self.kp)
            self.ke = torch.zeros((L, nb, HKV, BS), dtype=torch.int8, device="cuda")
            self.ve = torch.zeros_like(self.ke)
            self.pool = kvp.kv_pool_create_kv4(desc, self.kp, self.ke, self.vp, self.ve)
        else:
            self.kp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            self.vp = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            self.pool = kvp.kv_pool_create(desc, self.kp, self.vp)
        self.m = oracle.PoolModel(nb, BS, seqs, mb, alloc_seed=seed,
                                  store=(np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)))
        self.desc = kvp.AttnDesc(L, HQ, HKV, D, BS, nb, 0.0, 1, kvp.KVP_KV_4BIT if kv4 else kvp.KVP_KV_BF16)
        self.draw = 0

    def close(self):
        kvp.kv_pool_destroy(self.pool)

    def kv(self, total):
        self.draw += 1
        return (W.normal_bf16(61, self.draw, (L, total, HKV, D)),
                W.normal_bf16(62, self.draw, (L, total, HKV, D)))

    def append(self, seqs, ntoks):
        k, v = self.kv(sum(ntoks))
        kvp.seq_append_batch(self.pool, seqs, ntoks, bf16_tensor(k), bf16_tensor(v))
        self.model_append(seqs, ntoks, k, v)

    def model_append(self, seqs, ntoks, k, v):
        off = 0
        for s, n in zip(seqs, ntoks):
            self.m.append(s, n, k[:, off:off + n], v[:, off:off + n])
            off += n

    def forked_batch(self):
        root = self.m.alloc()
        assert kvp.seq_alloc(self.pool) == root
        self.append([root], [150])                 # ends in a partial block
        kids = []
        for _ in range(4):
            c = self.m.fork(root)
            assert kvp.seq_fork(self.pool, root) == c
            kids.append(c)
        return kids

    def same(self, seqs):
        assert kvp.kvp_cow_count(self.pool) == self.m.cow_copies
        assert kvp.kvp_free_block_count(self.pool) == self.m.free_count()
        for s in seqs:
            assert list(kvp.seq_block_table(self.pool, s)) == self.m.table(s)
            assert kvp.seq_len(self.pool, s) == self.m.length(s)

    def oracle(self, q, seqs):
        t = np.full((len(seqs), self.mb), -1, np.int32)
        for i, s in enumerate(seqs):
            tb = self.m.table(s)
            t[i, :len(tb)] = tb
        ln = np.array([self.m.length(s) for s in seqs], np.int32)
        return oracle.decode_attention(q, self.m.store[0], self.m.store[1], t, ln)

    def reference_call(self, q_dev, seqs):
        """paged_decode_attention on host tables gathered from the pool."""
        S = len(seqs)
        t, ln = kvp.kvp_gather_tables(self.pool, seqs, self.mb)
        ws = torch.empty(kvp.kvp_decode_workspace_size(self.desc, t, ln), dtype=torch.uint8, device="cuda")
        out = torch.empty((L, S, HQ, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((L, S, HQ), dtype=torch.float32, device="cuda")
        if self.kv4:
            kvp.paged_decode_attention_kv4(q_dev, self.kp, self.ke, self.vp, self.ve, t, ln, self.desc, out, lse, ws)
        else:
            kvp.paged_decode_attention(q_dev, self.kp, self.vp, t, ln, self.desc, out, lse, ws)
        torch.cuda.synchronize()
        return out, lse


@pytest.mark.parametrize("mode", ["mapped", "pinned", "pageable"])
def test_decode_step_from_host_buffers(mode):
    # mapped: page-locked buffers crossing in one copy kernel each way;
    # pinned: the same buffers through copy-engine transfers; pageable: numpy
    pinned = mode != "pageable"
    p = Pool()
    seqs = p.forked_batch()
    S = len(seqs)
    d_k = torch.empty((L, S, HKV, D), dtype=torch.bfloat16, device="cuda")
    d_v = torch.empty_like(d_k)
    d_q = torch.empty((L, S, HQ, D), dtype=torch.bfloat16, device="cuda")
    d_out = torch.empty_like(d_q)
    d_lse = torch.empty((L, S, HQ), dtype=torch.float32, device="cuda")
    h_out = torch.empty(d_out.shape, dtype=torch.bfloat16)
    h_lse = torch.empty(d_lse.shape, dtype=torch.float32)
    if pinned:
        h_out, h_lse = h_out.pin_memory(), h_lse.pin_memory()
    ws = torch.empty(4 << 20, dtype=torch.uint8, device="cuda")
    for step in range(4):
        k, v = p.kv(S)
        q = W.normal_bf16(63, step, (L, S, HQ, D))
        if pinned:
            hk, hv, hq = host_bf16(k), host_bf16(v), host_bf16(q)
        else:   # pageable numpy buffers
            hk, hv, hq = k, v, q
        io = kvp.step_io(d_q, d_out, d_lse, d_k, d_v, h_k_new=hk, h_v_new=hv, h_q=hq,
                         h_out=h_out if pinned else None, h_lse=h_lse if pinned else None,
                         host_mapped=mode == "mapped")
        assert io.flags == (kvp.KVP_STEP_HOST_MAPPED if mode == "mapped" else 0)
        if pinned:   # the prepared call (arguments marshalled once)
            need = kvp.DecodeStep(p.pool, seqs, 1, io, p.desc, ws)()
        else:
            need = kvp.kvp_decode_step(p.pool, seqs, 1, io, p.desc, ws)
        torch.cuda.synchronize()
        assert 0 < need <= ws.numel()
        assert kvp.kvp_device_error(ws) == 0
        p.model_append(seqs, [1] * S, k, v)
        p.same(seqs)
        got = (h_out, h_lse) if pinned else (d_out.cpu(), d_lse.cpu())
        want, want_lse = p.oracle(q, seqs)
        check_close(to_f64(got[0]), want)
        check_lse(to_f64(got[1]), want_lse)
        # the same bits as the host-table entry point on the same pool state
        ro, rl = p.reference_call(bf16_tensor(q), seqs)
        assert torch.equal(ro.cpu(), got[0].cpu()) and torch.equal(rl.cpu(), got[1].cpu())
    assert p.m.cow_copies >= 4      # every child's first append copied the shared partial block
    p.close()


@pytest.mark.parametrize("kv4", [False, True])
def test_pool_tables_entry_matches_host_tables(kv4):
    p = Pool(kv4=kv4)
    seqs = p.forked_batch()
    p.append(seqs, [3, 17, 40, 1])
    S = len(seqs)
    q = bf16_tensor(W.normal_bf16(64, 0, (L, S, HQ, D)))
    ws = torch.empty(kvp.kvp_pool_decode_workspace_size(p.pool, seqs, p.desc), dtype=torch.uint8, device="cuda")
    out = torch.empty((L, S, HQ, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((L, S, HQ), dtype=torch.float32, device="cuda")
    kvp.paged_decode_attention_pool(p.pool, seqs, q, out, lse, p.desc, ws)
    torch.cuda.synchronize()
    ro, rl = p.reference_call(q, seqs)
    assert torch.equal(out, ro) and torch.equal(lse, rl)
    # a device-only step (inputs already on the device, outputs left there)
    k, v = p.kv(S)
    io = kvp.step_io(q, out, lse, bf16_tensor(k), bf16_tensor(v))
    kvp.kvp_decode_step(p.pool, seqs, 1, io, p.desc, torch.empty(4 << 20, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    p.model_append(seqs, [1] * S, k, v)
    p.same(seqs)
    ro, rl = p.reference_call(q, seqs)
    assert torch.equal(out, ro) and torch.equal(lse, rl)
    p.close()


def test_small_workspace_and_full_pool():
    p = Pool(nb=40)     # small enough that one sequence can take every free block
    seqs = p.forked_batch()
    S = len(seqs)
    k, v = p.kv(S)
    q = bf16_tensor(W.normal_bf16(65, 0, (L, S, HQ, D)))
    out = torch.empty((L, S, HQ, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((L, S, HQ), dtype=torch.float32, device="cuda")
    io = kvp.step_io(q, out, lse, bf16_tensor(k), bf16_tensor(v))
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step(p.pool, seqs, 1, io, p.desc, small)
    assert e.value.code == kvp.KVP_ERR_WORKSPACE and e.value.ws_needed > 1024
    p.model_append(seqs, [1] * S, k, v)     # the append went through
    p.same(seqs)
    ws = torch.empty(e.value.ws_needed, dtype=torch.uint8, device="cuda")
    kvp.paged_decode_attention_pool(p.pool, seqs, q, out, lse, p.desc, ws)
    torch.cuda.synchronize()
    want, want_lse = p.oracle(W.normal_bf16(65, 0, (L, S, HQ, D)), seqs)
    check_close(to_f64(out), want)
    check_lse(to_f64(lse), want_lse)
    # fill the pool: a step whose appends need more blocks than are free
    # changes nothing
    free = kvp.kvp_free_block_count(p.pool)
    filler = p.m.alloc()
    assert kvp.seq_alloc(p.pool) == filler
    p.append([filler], [free * BS])
    assert kvp.kvp_free_block_count(p.pool) == 0
    lens = [kvp.seq_len(p.pool, s) for s in seqs]
    k, v = p.kv(S * BS)
    io = kvp.step_io(q, out, lse, bf16_tensor(k), bf16_tensor(v))
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step(p.pool, seqs, BS, io, p.desc, ws)
    assert e.value.code == kvp.KVP_ERR_OOM
    assert [kvp.seq_len(p.pool, s) for s in seqs] == lens
    p.same(seqs + [filler])
    p.close()


def step_buffers(S, ntok=1):
    d_k = torch.empty((L, S * ntok, HKV, D), dtype=torch.bfloat16, device="cuda")
    d_q = torch.empty((L, S, HQ, D), dtype=torch.bfloat16, device="cuda")
    return dict(d_k=d_k, d_v=torch.empty_like(d_k), d_q=d_q, d_out=torch.empty_like(d_q),
                d_lse=torch.empty((L, S, HQ), dtype=torch.float32, device="cuda"),
                h_k=torch.empty(d_k.shape, dtype=torch.bfloat16).pin_memory(),
                h_v=torch.empty(d_k.shape, dtype=torch.bfloat16).pin_memory(),
                h_q=torch.empty(d_q.shape, dtype=torch.bfloat16).pin_memory(),
                h_out=torch.empty(d_q.shape, dtype=torch.bfloat16).pin_memory(),
                h_lse=torch.empty((L, S, HQ), dtype=torch.float32).pin_memory())


def bits_into(dst, bits):
    dst.copy_(torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16))


@pytest.mark.parametrize("mapped", [True, False])
def test_planned_steps_overlap_the_device(mapped):
    p = Pool()
    seqs = p.forked_batch()
    S = len(seqs)
    b = step_buffers(S)
    io = kvp.step_io(b["d_q"], b["d_out"], b["d_lse"], b["d_k"], b["d_v"], h_k_new=b["h_k"], h_v_new=b["h_v"],
                     h_q=b["h_q"], h_out=b["h_out"], h_lse=b["h_lse"], host_mapped=mapped)
    ws = torch.empty(4 << 20, dtype=torch.uint8, device="cuda")
    sp = kvp.StepPlan(p.pool, seqs, 1, io, p.desc, ws)
    need = sp.plan()                          # step 0's host half
    assert 0 < need <= ws.numel()
    # the sequences hold the planned token at once
    assert [kvp.seq_len(p.pool, s) for s in seqs] == [p.m.length(s) + 1 for s in seqs]
    steps = 4
    for step in range(steps):
        k, v = p.kv(S)
        q = W.normal_bf16(66, step, (L, S, HQ, D))
        bits_into(b["h_k"], k)
        bits_into(b["h_v"], v)
        bits_into(b["h_q"], q)
        sp.run()
        if step + 1 < steps:
            sp.plan()                         # step + 1's host half, while the device runs this step
        torch.cuda.synchronize()
        assert kvp.kvp_device_error(ws) == 0
        p.model_append(seqs, [1] * S, k, v)
        want, want_lse = p.oracle(q, seqs)
        check_close(to_f64(b["h_out"]), want)
        check_lse(to_f64(b["h_lse"]), want_lse)
    p.same(seqs)
    sp.close()
    p.close()


def test_planned_step_matches_host_tables_and_errors():
    p = Pool()
    seqs = p.forked_batch()
    S = len(seqs)
    b = step_buffers(S)
    io = kvp.step_io(b["d_q"], b["d_out"], b["d_lse"], b["d_k"], b["d_v"])
    ws = torch.empty(4 << 20, dtype=torch.uint8, device="cuda")
    plan = kvp.kvp_step_plan_create()
    # a run with nothing planned
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step_run(plan, io, ws)
    assert e.value.code == kvp.KVP_ERR_INVALID
    k, v = p.kv(S)
    q = W.normal_bf16(67, 0, (L, S, HQ, D))
    b["d_k"].copy_(bf16_tensor(k))
    b["d_v"].copy_(bf16_tensor(v))
    b["d_q"].copy_(bf16_tensor(q))
    kvp.kvp_decode_step_plan(p.pool, seqs, 1, p.desc, plan)
    # a second plan while the first waits for its run: its tokens are already in
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step_plan(p.pool, seqs, 1, p.desc, plan)
    assert e.value.code == kvp.KVP_ERR_INVALID
    kvp.kvp_decode_step_run(plan, io, ws)
    torch.cuda.synchronize()
    p.model_append(seqs, [1] * S, k, v)
    p.same(seqs)
    ro, rl = p.reference_call(b["d_q"], seqs)
    assert torch.equal(ro, b["d_out"]) and torch.equal(rl, b["d_lse"])
    want, want_lse = p.oracle(q, seqs)
    check_close(to_f64(b["d_out"]), want)
    check_lse(to_f64(b["d_lse"]), want_lse)
    # a short workspace: the append is written, the plan is used up
    k, v = p.kv(S)
    b["d_k"].copy_(bf16_tensor(k))
    b["d_v"].copy_(bf16_tensor(v))
    need = kvp.kvp_decode_step_plan(p.pool, seqs, 1, p.desc, plan)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    assert need > small.numel()
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step_run(plan, io, small)
    assert e.value.code == kvp.KVP_ERR_WORKSPACE
    with pytest.raises(kvp.KvpError) as e:
        kvp.kvp_decode_step_run(plan, io, ws)
    assert e.value.code == kvp.KVP_ERR_INVALID
    p.model_append(seqs, [1] * S, k, v)
    p.same(seqs)
    kvp.paged_decode_attention_pool(p.pool, seqs, b["d_q"], b["d_out"], b["d_lse"], p.desc, ws)
    torch.cuda.synchronize()
    want, want_lse = p.oracle(q, seqs)
    check_close(to_f64(b["d_out"]), want)
    check_lse(to_f64(b["d_lse"]), want_lse)
    kvp.kvp_step_plan_destroy(plan)
    p.close()


@pytest.mark.parametrize("case", ["many_tokens", "big_plan"])
def test_planned_step_beyond_the_one_kernel_path(case):
    # many_tokens: 4 sequences x 20 appended tokens (80 > 64 slots);
    # big_plan: 160 forked sequences with their own tails, whose plan image
    # is larger than the 24 KB the one-kernel path carries
    if case == "many_tokens":
        p, ntok = Pool(), 20
        seqs = p.forked_batch()
    else:
        p, ntok = Pool(nb=4096, seqs=170, mb=32), 1
        root = p.m.alloc()
        assert kvp.seq_alloc(p.pool) == root
        p.append([root], [100])
        seqs = []
        for i in range(160):
            c = p.m.fork(root)
            assert kvp.seq_fork(p.pool, root) == c
            seqs.append(c)
        # tails of up to 400 tokens: about 500 KV tiles, a plan image near 28 KB
        p.append(seqs, [1 + (37 * i) % 400 for i in range(160)])
    S = len(seqs)
    b = step_buffers(S, ntok)
    io = kvp.step_io(b["d_q"], b["d_out"], b["d_lse"], b["d_k"], b["d_v"], h_k_new=b["h_k"], h_v_new=b["h_v"],
                     h_q=b["h_q"], h_out=b["h_out"], h_lse=b["h_lse"], host_mapped=True)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    sp = kvp.StepPlan(p.pool, seqs, ntok, io, p.desc, ws)
    sp.plan()
    k, v = p.kv(S * ntok)
    q = W.normal_bf16(68, 0, (L, S, HQ, D))
    bits_into(b["h_k"], k)
    bits_into(b["h_v"], v)
    bits_into(b["h_q"], q)
    sp.run()
    torch.cuda.synchronize()
    assert kvp.kvp_device_error(ws) == 0
    p.model_append(seqs, [ntok] * S, k, v)
    p.same(seqs)
    want, want_lse = p.oracle(q, seqs)
    check_close(to_f64(b["h_out"]), want)
    check_lse(to_f64(b["h_lse"]), want_lse)
    sp.close()
    p.close()
