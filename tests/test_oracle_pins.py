"""Pins of the oracle's attention to things other than itself.

Brute force on tiny contiguous inputs, closed forms computed by hand from the
softmax definition, and invariants that any correct implementation
satisfies.  A dropped term, a wrong sign, a transposed index, a wrong head
mapping or a wrong scale in the oracle fails at least one of these.
"""
import math

import numpy as np
import pytest

import oracle
from workloads import f32_to_bf16_bits, bf16_bits_to_f32, normal_bf16

pytestmark = pytest.mark.filterwarnings("ignore")


def bf(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def up(b):
    return bf16_bits_to_f32(b).astype(np.float64)


def scatter_into_pool(seqs_k, seqs_v, Hkv, d, bs, NB, rng, L=1):
    """Place contiguous per-sequence K/V ([L][n][Hkv][d]) into a pool at random
    distinct block ids.  Returns pool arrays, tables, lens."""
    k_pool = np.zeros((L, NB, Hkv, bs, d), dtype=np.uint16)
    v_pool = np.zeros_like(k_pool)
    free = list(rng.permutation(NB))
    MB = max(-(-k.shape[1] // bs) for k in seqs_k)
    tables = np.full((len(seqs_k), MB), -1, dtype=np.int32)
    lens = np.zeros(len(seqs_k), dtype=np.int32)
    for s, (k, v) in enumerate(zip(seqs_k, seqs_v)):
        n = k.shape[1]
        lens[s] = n
        for j in range(-(-n // bs)):
            b = free.pop()
            tables[s, j] = b
            lo, hi = j * bs, min(n, (j + 1) * bs)
            k_pool[:, b, :, :hi - lo, :] = k[:, lo:hi].transpose(0, 2, 1, 3)
            v_pool[:, b, :, :hi - lo, :] = v[:, lo:hi].transpose(0, 2, 1, 3)
    return k_pool, v_pool, tables, lens


def brute(q, k, v, scale):
    """Contiguous attention, vectorised numpy: q [Hq][d], k/v [n][Hkv][d]."""
    Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    out = np.empty((Hq, d)); lse = np.empty(Hq)
    for h in range(Hq):
        z = (k[:, h // G, :] @ q[h]) * scale
        m = z.max()
        e = np.exp(z - m)
        out[h] = (e[:, None] * v[:, h // G, :]).sum(0) / e.sum()
        lse[h] = m + np.log(e.sum())
    return out, lse


@pytest.mark.parametrize("bs", [1, 4, 16])
def test_decode_matches_brute_force(bs):
    rng = np.random.default_rng(11 + bs)
    Hq, Hkv, d, L = 6, 2, 8, 2
    lens = [1, 5, 17, 40, 33]
    ks = [normal_bf16(1, 10 + i, (L, n, Hkv, d)) for i, n in enumerate(lens)]
    vs = [normal_bf16(1, 20 + i, (L, n, Hkv, d)) for i, n in enumerate(lens)]
    NB = sum(-(-n // bs) for n in lens) + 5
    kp, vp, tables, ln = scatter_into_pool(ks, vs, Hkv, d, bs, NB, rng, L)
    q = normal_bf16(1, 99, (L, len(lens), Hq, d))
    out, lse = oracle.decode_attention(q, kp, vp, tables, ln)
    for l in range(L):
        for s in range(len(lens)):
            bo, bl = brute(up(q[l, s]), up(ks[s][l]), up(vs[s][l]), 1 / math.sqrt(d))
            np.testing.assert_allclose(out[l, s], bo, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[l, s], bl, rtol=0, atol=1e-12)


def test_sampled_equals_full():
    rng = np.random.default_rng(3)
    ks = [normal_bf16(2, i, (2, n, 2, 8)) for i, n in enumerate([9, 30])]
    vs = [normal_bf16(2, 5 + i, (2, n, 2, 8)) for i, n in enumerate([9, 30])]
    kp, vp, t, ln = scatter_into_pool(ks, vs, 2, 8, 4, 20, rng, 2)
    q = normal_bf16(2, 50, (2, 2, 4, 8))
    out, lse = oracle.decode_attention(q, kp, vp, t, ln)
    samples = np.array([[1, 0, 3], [0, 1, 2], [1, 1, 0]], dtype=np.int32)
    so, sl = oracle.decode_attention(q, kp, vp, t, ln, samples=samples)
    for i, (l, r, h) in enumerate(samples):
        assert np.array_equal(so[i], out[l, r, h]) and sl[i] == lse[l, r, h]


def _one_seq(k, v, bs=4, NB=8, seed=0):
    """k, v: [n][Hkv][d] uint16 -> pool, table, len for one sequence, L=1."""
    return scatter_into_pool([k[None]], [v[None]], k.shape[1], k.shape[2], bs, NB,
                             np.random.default_rng(seed))


def test_single_key_returns_its_value():
    d = 16
    k = normal_bf16(3, 1, (1, 1, d)); v = normal_bf16(3, 2, (1, 1, d))
    q = normal_bf16(3, 3, (1, 1, 2, d))
    kp, vp, t, ln = _one_seq(k, v)
    out, lse = oracle.decode_attention(q, kp, vp, t, ln)
    np.testing.assert_array_equal(out[0, 0, 0], up(v[0, 0]))
    # lse of one key is its score
    z = float(up(q[0, 0, 0]) @ up(k[0, 0])) / math.sqrt(d)
    assert abs(lse[0, 0, 0] - z) < 1e-12


def test_zero_query_gives_mean_value_and_log_n():
    n, d = 13, 8
    k = normal_bf16(4, 1, (n, 1, d)); v = normal_bf16(4, 2, (n, 1, d))
    q = np.zeros((1, 1, 1, d), dtype=np.uint16)
    kp, vp, t, ln = _one_seq(k, v)
    out, lse = oracle.decode_attention(q, kp, vp, t, ln)
    np.testing.assert_allclose(out[0, 0, 0], up(v[:, 0]).mean(0), atol=1e-14)
    assert abs(lse[0, 0, 0] - math.log(n)) < 1e-14


def test_identical_keys_give_mean_value():
    n, d = 9, 8
    k = np.repeat(normal_bf16(5, 1, (1, 1, d)), n, axis=0)
    v = normal_bf16(5, 2, (n, 1, d))
    q = normal_bf16(5, 3, (1, 1, 1, d))
    kp, vp, t, ln = _one_seq(k, v)
    out, _ = oracle.decode_attention(q, kp, vp, t, ln)
    np.testing.assert_allclose(out[0, 0, 0], up(v[:, 0]).mean(0), atol=1e-14)


def test_two_keys_closed_form_pins_the_scale():
    # q = 2 e0, k1 = 4 e0, k2 = 0, d = 16: z1 = 8 / sqrt(16) = 2, z2 = 0.
    # out = sigmoid(2) v1 + sigmoid(-2) v2, lse = ln(e^2 + 1).
    d = 16
    q = np.zeros((1, 1, 1, d), dtype=np.float32); q[..., 0] = 2
    k = np.zeros((2, 1, d), dtype=np.float32); k[0, 0, 0] = 4
    v = np.zeros((2, 1, d), dtype=np.float32); v[0, 0, 0] = 1; v[1, 0, 1] = 1
    kp, vp, t, ln = _one_seq(bf(k), bf(v))
    out, lse = oracle.decode_attention(bf(q), kp, vp, t, ln)
    assert abs(out[0, 0, 0, 0] - 0.8807970779778823) < 1e-15
    assert abs(out[0, 0, 0, 1] - 0.11920292202211755) < 1e-15
    assert abs(lse[0, 0, 0] - 2.1269280110429727) < 1e-15
    # an explicit scale replaces 1/sqrt(d): scale 1 gives z1 = 8
    out1, lse1 = oracle.decode_attention(bf(q), kp, vp, t, ln, scale=1.0)
    assert abs(out1[0, 0, 0, 0] - 1 / (1 + math.exp(-8))) < 1e-15
    assert abs(lse1[0, 0, 0] - math.log(math.exp(8) + 1)) < 1e-13


def test_dominant_key_selects_its_value():
    n, d = 20, 8
    k = np.zeros((n, 1, d), dtype=np.float32)
    k[7, 0, 0] = 30.0          # score 30 * 16 / sqrt(8) ~ 170 above the rest
    v = normal_bf16(6, 2, (n, 1, d))
    q = np.zeros((1, 1, 1, d), dtype=np.float32); q[..., 0] = 16
    kp, vp, t, ln = _one_seq(bf(k), v, bs=8, NB=4)
    out, _ = oracle.decode_attention(bf(q), kp, vp, t, ln)
    np.testing.assert_array_equal(out[0, 0, 0], up(v[7, 0]))


def test_weights_sum_to_one_and_linearity():
    n, d = 37, 8
    k = normal_bf16(7, 1, (n, 2, d)); ones = bf(np.ones((n, 2, d)))
    q = normal_bf16(7, 3, (1, 1, 4, d))
    kp, vp, t, ln = _one_seq(k, ones, bs=16, NB=6)
    out, _ = oracle.decode_attention(q, kp, vp, t, ln)
    np.testing.assert_allclose(out, 1.0, atol=1e-14)
    # out is linear in V: V1 and V2 chosen so that V1 + V2 is exact in bf16
    v1 = bf(np.arange(n * 2 * d).reshape(n, 2, d) % 7)
    v2 = bf(np.arange(n * 2 * d).reshape(n, 2, d) % 5)
    v12 = bf(up(v1) + up(v2))
    res = []
    for vv in (v1, v2, v12):
        kp, vp, t, ln = _one_seq(k, vv, bs=16, NB=6)
        res.append(oracle.decode_attention(q, kp, vp, t, ln)[0])
    np.testing.assert_allclose(res[0] + res[1], res[2], atol=1e-12)


def test_gqa_head_mapping_is_consecutive_groups():
    # kv head g has V == g + 1 everywhere; q head h must read kv head h // G.
    n, Hkv, G, d = 6, 4, 3, 8
    k = normal_bf16(8, 1, (n, Hkv, d))
    v = bf(np.broadcast_to(np.arange(1, Hkv + 1, dtype=np.float32)[None, :, None], (n, Hkv, d)))
    q = normal_bf16(8, 2, (1, 1, Hkv * G, d))
    kp, vp, t, ln = _one_seq(k, v, bs=4, NB=4)
    out, _ = oracle.decode_attention(q, kp, vp, t, ln)
    for h in range(Hkv * G):
        np.testing.assert_allclose(out[0, 0, h], h // G + 1, atol=1e-14)
    # identical q within a group gives identical outputs
    q2 = q.copy(); q2[0, 0, :] = q[0, 0, 0]
    out2, _ = oracle.decode_attention(q2, kp, vp, t, ln)
    for h in range(Hkv * G):
        np.testing.assert_array_equal(out2[0, 0, h], out2[0, 0, (h // G) * G])


def test_lse_merge_of_a_key_partition_equals_whole():
    bs, n, d = 8, 45, 16
    k = normal_bf16(9, 1, (n, 1, d)); v = normal_bf16(9, 2, (n, 1, d))
    q = normal_bf16(9, 3, (1, 1, 1, d))
    kp, vp, t, ln = _one_seq(k, v, bs=bs, NB=9)
    whole, wl = oracle.decode_attention(q, kp, vp, t, ln)
    for a_blocks in (1, 3, 5):
        a = a_blocks * bs
        o1, l1 = oracle.decode_attention(q, kp, vp, t, np.array([a], np.int32))
        t2 = np.full_like(t, -1); t2[0, :t.shape[1] - a_blocks] = t[0, a_blocks:]
        o2, l2 = oracle.decode_attention(q, kp, vp, t2, np.array([n - a], np.int32))
        M = max(l1[0, 0, 0], l2[0, 0, 0])
        w1, w2 = math.exp(l1[0, 0, 0] - M), math.exp(l2[0, 0, 0] - M)
        merged = (w1 * o1[0, 0, 0] + w2 * o2[0, 0, 0]) / (w1 + w2)
        np.testing.assert_allclose(merged, whole[0, 0, 0], atol=1e-12)
        assert abs(M + math.log(w1 + w2) - wl[0, 0, 0]) < 1e-12


def test_errors_on_empty_sequence_and_bad_block():
    k = normal_bf16(1, 1, (4, 1, 8)); v = normal_bf16(1, 2, (4, 1, 8))
    kp, vp, t, ln = _one_seq(k, v)
    q = normal_bf16(1, 3, (1, 1, 1, 8))
    with pytest.raises(ValueError):
        oracle.decode_attention(q, kp, vp, t, np.array([0], np.int32))
    bad = t.copy(); bad[0, 0] = kp.shape[1]
    with pytest.raises(ValueError):
        oracle.decode_attention(q, kp, vp, bad, ln)


# ------------------------------------------------------------- tree verify

def _verify_setup(ctx, n, parents, d=8, Hq=4, Hkv=2, bs=4, seed=0, L=1):
    B = len(ctx)
    ks = [normal_bf16(seed, 100 + b, (L, ctx[b] + n, Hkv, d)) for b in range(B)]
    vs = [normal_bf16(seed, 200 + b, (L, ctx[b] + n, Hkv, d)) for b in range(B)]
    NB = sum(-(-(c + n) // bs) for c in ctx) + 3
    kp, vp, t, ln = scatter_into_pool(ks, vs, Hkv, d, bs, NB, np.random.default_rng(seed), L)
    q = normal_bf16(seed, 300, (L, B * n, Hq, d))
    return ks, vs, kp, vp, t, q


def test_verify_one_node_equals_decode():
    ctx, n = [13, 20], 1
    ks, vs, kp, vp, t, q = _verify_setup(ctx, n, None)
    par = np.full((2, 1), -1, np.int32)
    vo, vl = oracle.verify_attention(q, kp, vp, t, np.array(ctx, np.int32), par)
    do, dl = oracle.decode_attention(q, kp, vp, t, np.array(ctx, np.int32) + 1)
    np.testing.assert_allclose(vo, do, atol=1e-14)
    np.testing.assert_allclose(vl, dl, atol=1e-14)


def test_verify_chain_tree_is_causal_attention():
    ctx, n, d = [11, 4], 9, 8
    ks, vs, kp, vp, t, q = _verify_setup(ctx, n, None, d=d)
    par = np.tile(np.arange(-1, n - 1, dtype=np.int32), (2, 1))
    vo, vl = oracle.verify_attention(q, kp, vp, t, np.array(ctx, np.int32), par)
    for b in range(2):
        for i in range(n):
            bo, bl = brute(up(q[0, b * n + i]), up(ks[b][0, :ctx[b] + i + 1]),
                           up(vs[b][0, :ctx[b] + i + 1]), 1 / math.sqrt(d))
            np.testing.assert_allclose(vo[0, b * n + i], bo, atol=1e-12)
            np.testing.assert_allclose(vl[0, b * n + i], bl, atol=1e-12)


def test_verify_star_tree_and_forest():
    ctx, n, d = [7], 6, 8
    ks, vs, kp, vp, t, q = _verify_setup(ctx, n, None, d=d)
    # star: node 0 root, every other node a child of 0
    star = np.array([[-1, 0, 0, 0, 0, 0]], np.int32)
    vo, _ = oracle.verify_attention(q, kp, vp, t, np.array(ctx, np.int32), star)
    for i in range(n):
        keep = list(range(ctx[0])) + sorted({ctx[0], ctx[0] + i})
        bo, _ = brute(up(q[0, i]), up(ks[0][0, keep]), up(vs[0][0, keep]), 1 / math.sqrt(d))
        np.testing.assert_allclose(vo[0, i], bo, atol=1e-12)
    # forest: roots 0 and 3; node 4 under 3, node 5 under 4, nodes 1, 2 under 0
    forest = np.array([[-1, 0, 1, -1, 3, 4]], np.int32)
    anc = {0: [0], 1: [0, 1], 2: [0, 1, 2], 3: [3], 4: [3, 4], 5: [3, 4, 5]}
    vo, _ = oracle.verify_attention(q, kp, vp, t, np.array(ctx, np.int32), forest)
    for i in range(n):
        keep = list(range(ctx[0])) + [ctx[0] + j for j in anc[i]]
        bo, _ = brute(up(q[0, i]), up(ks[0][0, keep]), up(vs[0][0, keep]), 1 / math.sqrt(d))
        np.testing.assert_allclose(vo[0, i], bo, atol=1e-12)


def test_verify_mask_recovered_from_one_hot_values():
    # q = 0 gives uniform weights over the attended set; with V of draft token
    # j equal to e_j and context V = 0, out[j] = 1/|set| exactly when j is in
    # the set: the attended draft set of each node is read off the output.
    ctx, n, d = 5, 8, 8
    parents = np.array([[-1, 0, 0, 1, 3, 2, -1, 6]], np.int32)
    expect = {0: {0}, 1: {0, 1}, 2: {0, 2}, 3: {0, 1, 3}, 4: {0, 1, 3, 4},
              5: {0, 2, 5}, 6: {6}, 7: {6, 7}}
    k = normal_bf16(12, 1, (1, ctx + n, 1, d))
    v = np.zeros((1, ctx + n, 1, d), np.float32)
    for j in range(n):
        v[0, ctx + j, 0, j] = 1
    kp, vp, t, _ = scatter_into_pool([k], [bf(v)], 1, d, 4, 6, np.random.default_rng(0))
    q = np.zeros((1, n, 1, d), np.uint16)
    out, lse = oracle.verify_attention(q, kp, vp, t, np.array([ctx], np.int32), parents)
    for i in range(n):
        size = ctx + len(expect[i])
        want = np.array([1.0 / size if j in expect[i] else 0.0 for j in range(d)])
        np.testing.assert_allclose(out[0, i, 0], want, atol=1e-15)
        assert abs(lse[0, i, 0] - math.log(size)) < 1e-14


def test_verify_rejects_bad_parent():
    ks, vs, kp, vp, t, q = _verify_setup([4], 3, None)
    with pytest.raises(ValueError):
        oracle.verify_attention(q, kp, vp, t, np.array([4], np.int32),
                                np.array([[-1, 2, 0]], np.int32))
