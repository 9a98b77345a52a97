"""Helpers shared by the GPU parity tests: tolerances and replaying one
workload through both the oracle and the library."""
import numpy as np

import oracle
import workloads as W

# Attention outputs (bf16 in, fp32 accumulate, bf16 out) must match the fp64
# oracle within max-abs 1e-2 and relative RMS 5e-3.  lse (fp32, natural log)
# carries fp32 score rounding (~1e-6 relative over |lse| < 20) plus the SFU
# exp2/log2 approximations (a few ulp): 1e-3 absolute leaves a wide margin.
MAX_ABS = 1e-2
REL_RMS = 5e-3
LSE_ABS = 1e-3


def bf16_absmax(bits):
    """max |x| over a uint16 bf16 bit-pattern array."""
    from workloads import bf16_bits_to_f32
    return float(np.abs(bf16_bits_to_f32(bits)).max())


def to_f64(t):
    """torch tensor (bf16 / fp32, any device) -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def peaked_max_abs(want, v_absmax):
    """Max-abs bound for sharply peaked softmax (queries scaled up): one or two
    keys carry the weight, so the bf16 rounding of P (unit roundoff 2^-8,
    relative to p) passes straight through to out as up to 2^-8 * |v|, and the
    bf16 rounding of out itself adds up to 2^-8 * |out|; the rounding errors no
    longer average out over many keys as they do for the N(0,1) workloads."""
    return 2.0 ** -8 * (float(np.abs(want).max()) + float(v_absmax)) + 1e-3


def check_close(got, want, what="out", max_abs_tol=MAX_ABS):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - want)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.sqrt((err ** 2).sum() / max((want ** 2).sum(), 1e-300)))
    assert max_abs <= max_abs_tol, f"{what}: max-abs {max_abs:.3e} > {max_abs_tol:.3e}"
    assert rel <= REL_RMS, f"{what}: rel-RMS {rel:.3e} > {REL_RMS}"
    return max_abs, rel


def check_lse(got, want):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    assert np.isfinite(got).all()
    assert float(err.max()) <= LSE_ABS, f"lse max-abs {float(err.max()):.3e}"


def oracle_side(w, alloc_seed, steps_kv=(), threads=0):
    """Replay the workload (and decode-step appends) through the oracle."""
    rw = oracle.replay(w, alloc_seed=alloc_seed)
    for k, v in steps_kv:
        oracle.replay_step(rw, w, k, v)
    return rw


def sample_triples(rng, L, nq, Hq, n):
    return np.stack([rng.integers(0, L, n), rng.integers(0, nq, n), rng.integers(0, Hq, n)],
                    axis=1).astype(np.int32)
