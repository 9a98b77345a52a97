"""4-bit KV pages on the GPU against the oracle format (oracle/kv4.py):

- quantise on append (seq_append_batch on a kv_pool_create_kv4 pool):
  every live token's codes and exponent, K and V, every layer and kv head,
  bit-exact against kv4.quantize of the same bf16 rows, including rows that
  reached their block by copy-on-write and rows moved by speculative accept;
- decode attention over the pool (paged_decode_attention_kv4) against the
  fp64 oracle over the dequantised pool (code * 2^e, exact in bf16) within
  max-abs 1e-2 and rel-RMS 5e-3 (lse 1e-3), on Dendrite-shaped forks (d 64,
  block 16) and MCTS-shaped trees (d 128, block 16 and 32)."""
import numpy as np
import pytest

import oracle
import workloads as W
from oracle import kv4
from _util import check_close, check_lse, peaked_max_abs, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_prefix_shared_decode_gb300 as kvp  # noqa: E402
from paged_prefix_shared_decode_gb300.runner import bf16_tensor  # noqa: E402


class Kv4Pool:
    """A 4-bit device pool and the oracle's bf16 model pool, in lockstep."""

    def __init__(self, L, Hkv, d, bs, nb, seqs=32, mb=160, seed=3):
        self.L, self.Hkv, self.d, self.bs, self.nb, self.mb = L, Hkv, d, bs, nb, mb
        self.kc = torch.zeros((L, nb, Hkv, bs, d // 2), dtype=torch.uint8, device="cuda")
        self.vc = torch.zeros_like(self.kc)
        self.ke = torch.zeros((L, nb, Hkv, bs), dtype=torch.int8, device="cuda")
        self.ve = torch.zeros_like(self.ke)
        self.pool = kvp.kv_pool_create_kv4(kvp.PoolDesc(L, nb, bs, Hkv, d, seqs, mb, seed),
                                           self.kc, self.ke, self.vc, self.ve)
        shape = (L, nb, Hkv, bs, d)
        self.m = oracle.PoolModel(nb, bs, seqs, mb, alloc_seed=seed,
                                  store=(np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)))
        self.stream = 0

    def close(self):
        kvp.kv_pool_destroy(self.pool)

    def alloc(self):
        s = self.m.alloc()
        assert kvp.seq_alloc(self.pool) == s
        return s

    def fork(self, p):
        s = self.m.fork(p)
        assert kvp.seq_fork(self.pool, p) == s
        return s

    def append(self, seqs, ntoks, scale=1.0):
        total = sum(ntoks)
        self.stream += 1
        k = W.normal_bf16(91, self.stream, (self.L, total, self.Hkv, self.d), scale)
        v = W.normal_bf16(92, self.stream, (self.L, total, self.Hkv, self.d), scale)
        kvp.seq_append_batch(self.pool, seqs, ntoks, bf16_tensor(k), bf16_tensor(v))
        off = 0
        for s, n in zip(seqs, ntoks):
            self.m.append(s, n, k[:, off:off + n], v[:, off:off + n])
            off += n

    def check_pages(self):
        """Codes and exponents of every live token row, bit-exact."""
        torch.cuda.synchronize()
        assert kvp.kvp_cow_count(self.pool) == self.m.cow_copies
        dev = [t.cpu().numpy() for t in (self.kc, self.ke, self.vc, self.ve)]
        live = set()   # distinct (block, slot) of live tokens
        for s in self.m.live():
            table = self.m.table(s)
            assert list(kvp.seq_block_table(self.pool, s)) == table
            live.update((table[pos // self.bs], pos % self.bs) for pos in range(self.m.length(s)))
        bl = np.array(sorted(live), np.int64)
        b, sl = bl[:, 0], bl[:, 1]
        for (codes, exps), store in ((dev[0:2], self.m.store[0]), (dev[2:4], self.m.store[1])):
            rows = W.bf16_bits_to_f32(store[:, b, :, sl, :]).astype(np.float64)   # [L][n][Hkv][d]
            want_c, want_e = kv4.quantize(rows)
            byt = codes[:, b, :, sl, :]
            lo = (byt & 0xF).astype(np.int16)
            hi = (byt >> 4).astype(np.int16)
            got_c = np.empty(want_c.shape, np.int16)
            got_c[..., 0::2] = np.where(lo >= 8, lo - 16, lo)
            got_c[..., 1::2] = np.where(hi >= 8, hi - 16, hi)
            assert np.array_equal(got_c, want_c.astype(np.int16))
            assert np.array_equal(exps[:, b, :, sl].astype(np.int16), want_e.astype(np.int16))
        return len(live)

    def dequantised_store(self):
        """The pool's values (code * 2^e) as bf16 bits, from the oracle format."""
        out = []
        for store in self.m.store:
            x = W.bf16_bits_to_f32(store).astype(np.float64)
            y = kv4.dequantize(*kv4.quantize(x))
            out.append(W.f32_to_bf16_bits(y.astype(np.float32)))
        return out

    def decode(self, seqs, Hq, step, q_scale=1.0):
        S = len(seqs)
        t, ln = kvp.kvp_gather_tables(self.pool, seqs, self.mb)
        q = W.normal_bf16(93, step, (self.L, S, Hq, self.d), q_scale)
        desc = kvp.AttnDesc(self.L, Hq, self.Hkv, self.d, self.bs, self.nb, 0.0, 1, kvp.KVP_KV_4BIT)
        ws = torch.empty(kvp.kvp_decode_workspace_size(desc, t, ln), dtype=torch.uint8, device="cuda")
        out = torch.empty((self.L, S, Hq, self.d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((self.L, S, Hq), dtype=torch.float32, device="cuda")
        kvp.paged_decode_attention_kv4(bf16_tensor(q), self.kc, self.ke, self.vc, self.ve, t, ln, desc, out, lse, ws)
        torch.cuda.synchronize()
        assert kvp.kvp_device_error(ws) == 0
        kd, vd = self.dequantised_store()
        want, want_lse = oracle.decode_attention(q, kd, vd, t, ln)
        # largest |v| among the keys these sequences attend to
        vals = [W.bf16_bits_to_f32(vd[:, t[i, pos // self.bs], :, pos % self.bs, :])
                for i in range(S) for pos in range(int(ln[i]))]
        self.v_absmax = float(np.abs(np.stack(vals)).max())
        return to_f64(out), to_f64(lse), want, want_lse


def test_quantise_on_append_fork_cow_and_decode_d64():
    p = Kv4Pool(L=2, Hkv=4, d=64, bs=16, nb=160)
    root = p.alloc()
    p.append([root], [250])                       # a partial last block
    kids = [p.fork(root) for _ in range(4)]
    p.append(kids, [1, 17, 40, 64])               # each first append copies the shared partial block
    p.append([root] + kids, [3, 1, 1, 1, 1])
    p.check_pages()
    assert p.m.cow_copies >= 4
    for step in range(2):
        p.append(kids, [1] * len(kids))
        got, got_l, want, want_l = p.decode(kids, Hq=32, step=step)
        check_close(got, want)
        check_lse(got_l, want_l)
    p.check_pages()
    p.close()


@pytest.mark.parametrize("bs", [16, 32])
def test_tree_shaped_sharing_d128(bs):
    # an MCTS-like tree: root, 4 children, 16 grandchildren (Llama-3-8B heads)
    p = Kv4Pool(L=2, Hkv=8, d=128, bs=bs, nb=200)
    root = p.alloc()
    p.append([root], [300])
    level = [root]
    for _ in range(2):
        nxt = []
        for par in level:
            for _c in range(4):
                c = p.fork(par)
                nxt.append(c)
        p.append(nxt, [40] * len(nxt))
        level = nxt
    p.append(level, [1] * len(level))
    p.check_pages()
    got, got_l, want, want_l = p.decode(level, Hq=32, step=7)
    check_close(got, want)
    check_lse(got_l, want_l)
    p.close()


def test_scaled_rows_and_peaked_queries():
    # rows far from unit scale (exponents from about -40 to +30) and a
    # sharply peaked softmax
    p = Kv4Pool(L=1, Hkv=4, d=64, bs=16, nb=64)
    s = [p.alloc() for _ in range(3)]
    for sq, sc in zip(s, (1e-12, 1.0, 1e9)):
        p.append([sq], [70], scale=sc)
    p.check_pages()
    got, got_l, want, want_l = p.decode(s[1:2], Hq=32, step=3, q_scale=4.0)
    check_close(got, want, max_abs_tol=peaked_max_abs(want, p.v_absmax))
    check_lse(got_l, want_l)
    p.close()


def test_accept_moves_codes_and_exponents():
    w = W.verify_tree(2, layers=1, ctx=200, n_draft=24)
    p = Kv4Pool(L=1, Hkv=8, d=128, bs=16, nb=64)
    seqs = [p.alloc() for _ in range(2)]
    p.append(seqs, [224, 224])
    sib = p.fork(seqs[0])                          # shares every block: moves copy first
    parents = w.info["parents"]
    for b, sq in enumerate(seqs):
        acc = 23 if b == 0 else 10
        pm = p.m.accept_draft(sq, 200, [int(x) for x in parents[b]], acc)
        pl = kvp.seq_accept_draft(p.pool, sq, 200, parents[b], acc)
        assert list(pl) == pm
    p.check_pages()
    assert p.m.length(sib) == 224
    p.close()
