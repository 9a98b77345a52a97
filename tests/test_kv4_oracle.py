"""Pins of the oracle's 4-bit KV format (oracle/kv4.py): the pages'
compression figure, the round-trip error bound, exact round trips of
representable rows, zero rows, sign symmetry, half-even ties, the scale being
the smallest that does not clip, and dequantised values being exact bf16
(so the fp64 bf16 attention oracle serves the 4-bit pool unchanged)."""
import os

import numpy as np
import pytest

import oracle
from oracle import kv4
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv4_compression.txt")


def test_compression_matches_the_pages_figure():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    for d, ratio in rows:
        assert round(kv4.compression_vs_bf16(int(d)), 2) == float(ratio)
    assert kv4.bits_per_value(64) == 4.125 and round(kv4.compression_vs_bf16(128), 2) == 3.94


@pytest.mark.parametrize("scale", [1e-30, 1e-3, 1.0, 37.0, 1e30])
def test_round_trip_error_is_at_most_half_a_step(scale):
    rng = np.random.default_rng(int(abs(np.log10(scale))) + 1)
    x = rng.standard_normal((50, 64)) * scale * rng.uniform(0.01, 10, (50, 1))
    codes, e = kv4.quantize(x)
    y = kv4.dequantize(codes, e)
    step = np.ldexp(1.0, e.astype(np.int64))[:, None]
    assert np.all(np.abs(codes) <= 7)
    assert np.all(np.abs(x - y) <= step / 2 * (1 + 1e-12))


def test_representable_rows_round_trip_exactly_and_scale_is_minimal():
    rng = np.random.default_rng(3)
    for _ in range(200):
        e = int(rng.integers(-100, 100))
        k = rng.integers(-7, 8, 64).astype(np.float64)
        k[0] = 7 * rng.choice([-1, 1])                      # the row's largest magnitude is 7 steps
        x = np.ldexp(k, e)
        codes, ee = kv4.quantize(x[None])
        assert ee[0] == e and np.array_equal(codes[0], k.astype(np.int8))
        assert np.array_equal(kv4.dequantize(codes, ee)[0], x)
    x = np.random.default_rng(4).standard_normal((100, 64))
    _, e = kv4.quantize(x)
    m = np.abs(x).max(1)
    assert np.all(m <= 7 * np.ldexp(1.0, e.astype(np.int64)))
    assert np.all(m > 7 * np.ldexp(1.0, e.astype(np.int64) - 1))


def test_zero_rows_sign_symmetry_and_ties():
    codes, e = kv4.quantize(np.zeros((2, 64)))
    assert np.all(codes == 0) and np.all(e == kv4.E_MIN)
    x = np.random.default_rng(5).standard_normal((30, 64))
    c1, e1 = kv4.quantize(x)
    c2, e2 = kv4.quantize(-x)
    assert np.array_equal(c2, -c1) and np.array_equal(e1, e2)
    c, e = kv4.quantize(np.array([[2.5, 3.5, -2.5, 7.0]]))   # max 7 -> step 1
    assert e[0] == 0 and list(c[0]) == [2, 4, -2, 7]


def test_dequantised_values_are_exact_bf16():
    x = np.random.default_rng(6).standard_normal((4, 3, 2, 16, 64)) * 3
    y = kv4.dequantize(*kv4.quantize(x))
    back = W.bf16_bits_to_f32(W.f32_to_bf16_bits(y.astype(np.float32))).astype(np.float64)
    assert np.array_equal(back, y)


def test_attention_over_a_4bit_pool_uses_the_bf16_oracle_exactly():
    # tiny pool: the bf16 oracle on the dequantised pool equals a direct fp64
    # softmax over the dequantised keys and values
    rng = np.random.default_rng(7)
    L, NB, Hkv, bs, d, Hq = 1, 4, 2, 4, 64, 4
    k = kv4.dequantize(*kv4.quantize(rng.standard_normal((L, NB, Hkv, bs, d))))
    v = kv4.dequantize(*kv4.quantize(rng.standard_normal((L, NB, Hkv, bs, d))))
    q = W.f32_to_bf16_bits(rng.standard_normal((L, 1, Hq, d)).astype(np.float32))
    table = np.array([[2, 0, 3]], np.int32)
    n = 10
    o, lse = oracle.decode_attention(q, W.f32_to_bf16_bits(k.astype(np.float32)),
                                     W.f32_to_bf16_bits(v.astype(np.float32)), table, np.array([n], np.int32))
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        keys = np.stack([k[0, table[0, t // bs], kv, t % bs] for t in range(n)])
        vals = np.stack([v[0, table[0, t // bs], kv, t % bs] for t in range(n)])
        z = keys @ qf[0, 0, h] / np.sqrt(d)
        p = np.exp(z - z.max())
        assert np.allclose(o[0, 0, h], p @ vals / p.sum(), rtol=1e-12, atol=1e-12)
        assert np.isclose(lse[0, 0, h], z.max() + np.log(p.sum()), rtol=1e-12)
