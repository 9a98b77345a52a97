"""paged_decode_attention_noalloc -- decode attention for callers that cannot
allocate device memory (their memory manager owns all device memory, or they
run inside a host program whose allocator they cannot reach).  It must give
the same results as paged_decode_attention with a caller workspace, on two
calls in a row (the library's static workspace keeps the previous call's
contents), and reject batches whose plan exceeds the static workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import workloads as W
from _util import check_close, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_prefix_shared_decode_gb300 as kvp  # noqa: E402
from paged_prefix_shared_decode_gb300.runner import PoolRunner, DecodeCall, bf16_tensor  # noqa: E402


def _noalloc(call, q, out, lse):
    """Call the entry point through the C ABI."""
    lib = kvp.load()
    t = np.ascontiguousarray(call.h_tables, np.int32)
    ln = np.ascontiguousarray(call.h_lens, np.int32)
    return lib.paged_decode_attention_noalloc(
        q.data_ptr(), call.r.k_pool.data_ptr(), call.r.v_pool.data_ptr(),
        t.ctypes.data_as(ctypes.c_void_p), ln.ctypes.data_as(ctypes.c_void_p), t.shape[0], t.shape[1],
        ctypes.byref(call.desc), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("make", [W.tiny_fork, lambda: W.dendrite(layers=4),
                                  lambda: W.trellis(0.5, layers=2)])
def test_noalloc_matches_workspace_entry_point_twice(make):
    w = make()
    r = PoolRunner(w, alloc_seed=1)
    r.run_ops()
    call = DecodeCall(r)
    if w.step_tokens:
        k, v = W.step_kv(w, 0)
        r.append_step(bf16_tensor(k), bf16_tensor(v))
    call.refresh()
    assert kvp.kvp_decode_workspace_size(call.desc, call.h_tables, call.h_lens) <= kvp.KVP_STATIC_WORKSPACE_BYTES
    for step in range(2):
        q = bf16_tensor(W.step_q(w, step))
        call(q)
        want_o, want_l = to_f64(call.out), to_f64(call.lse)
        out = torch.full_like(call.out, float("nan"))
        lse = torch.full_like(call.lse, float("nan"))
        assert _noalloc(call, q, out, lse) == kvp.KVP_OK
        torch.cuda.synchronize()
        check_close(to_f64(out), want_o)
        assert np.abs(to_f64(lse) - want_l).max() <= 1e-3
    r.close()


def test_noalloc_rejects_batches_beyond_the_static_workspace():
    w = W.tiny_fork()
    r = PoolRunner(w, alloc_seed=1)
    r.run_ops()
    call = DecodeCall(r)
    call.refresh()
    # the same tables planned for many more layers need far more than the
    # static workspace; the call must refuse before touching the device
    big = kvp.AttnDesc(4096, 32, 4, 64, 16, r.NB, 0.0, 1)
    assert kvp.kvp_decode_workspace_size(big, call.h_tables, call.h_lens) > kvp.KVP_STATIC_WORKSPACE_BYTES
    call.desc = big
    q = torch.zeros((1, 4, 32, 64), dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(call, q, torch.empty_like(q), torch.empty((1, 4, 32), device="cuda"))
    assert rc == kvp.KVP_ERR_INVALID
    r.close()
