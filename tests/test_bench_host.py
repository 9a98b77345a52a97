"""Host-side logic of bench.py: workload naming and sizing, the JSON
descriptors, peak lookup, and the max-over-ranks aggregation of the replica
runs (world size 2 over gloo on CPU)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("name", ["dendrite", "trellis0.0", "trellis0.9", "mcts", "verify1", "verify32", "tiny"])
def test_workloads_and_descriptions(name):
    w = bench.workload(name, 40)
    assert w.num_blocks > 0 and w.max_blocks_per_seq > 0
    assert isinstance(bench.describe(w), str) and w.shapes.bs in (16, 32)


def test_peaks_and_traffic_lookup():
    peak, kind = bench.peaks()
    assert peak > 1000 and kind in ("measured", "fallback")
    for name in ("dendrite", "trellis_phi0.9", "mcts", "no-such-workload"):
        t = bench.traffic_for(name)
        assert t is None or t["dram_bytes_per_launch"] > 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out[rank] = bench.max_over_ranks(10.0 + rank * 5.0, world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
    assert all(p.exitcode == 0 for p in ps)
    assert out[0] == out[1] == 15.0
    assert bench.max_over_ranks(3.0, 1) == 3.0


@pytest.mark.parametrize("phi,frac", [(0.0, 0.0), (0.5, 0.5), (0.9, 0.875)])
def test_prefix_cache_bench_runs_on_the_host(phi, frac):
    # the radix-cache sweep entry needs no GPU; it also checks that the
    # library and the oracle served the same number of prompt tokens
    import paged_prefix_shared_decode_gb300 as kvp
    r = bench.prefix_cache_bench(kvp, phi, with_oracle=True, reps=1)
    assert r["hit_frac"] == frac
    assert r["host_us_per_session"] > 0 and r["cpu_baseline"]["host_us_per_session"] > 0
