#!/usr/bin/env python
"""Benchmark: decode attention tokens/s and achieved HBM GB/s over a
block-paged, prefix-shared KV pool on GB300.

Default workload (one GPU): Dendrite-shaped fork decode -- TinyLlama-1.1B
attention shapes (22 layers, 32 query / 4 kv heads, d 64), block 16, a
4096-token prefix forked into 6 branches with U{0..512} private tokens each.
One step = the whole hot path for one decode token per branch: append its K/V
(batched scatter, copy-on-write where needed), export the block tables, plan,
and run paged attention over all 22 layers (work-item kernel + log-sum-exp
merge).  Inputs are resident in HBM; L2 is flushed (a write of 2x its size)
between timed steps, outside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dendrite|trellis0.5|mcts|verify8|...] [--no-sweep]
                    [--sweep-set a,b,...] [--cost-table]

Beside the headline the line carries (unless --no-sweep):
  sweep   short device-timed runs of the rest of the metric: the Trellis phi
          sweep (0, 0.25, 0.5, 0.75, 0.9), MCTS (32 layers) and tree verify
          (B 1, 8, 32), each with unique KV bytes, kernel time, fraction of the
          HBM roofline, the sharing-off time and a single-layer call; and
          host-timed runs of the radix prefix cache on the Trellis session
          pattern (radix0.5 / radix0.9, the oracle beside them);
  fork    host seq_fork + seq_free of the Dendrite parent (256 blocks),
          beside the device copy of that context's K/V that a fork avoids;
  memory  the Dendrite batch's KV blocks and bytes with and without sharing.
--cost-table prints the tree-verify cost f(B, c, n) (B 1-32, contexts
512-8192, drafts of 16-64 nodes) and exits.

N > 1 runs independent replicas, one per GPU (torchrun; no data-path
collective).  `--impl reference` times the fp64 CPU oracle on the host cores
on the same workload and prints the same JSON line with "impl": "reference".
Prints exactly one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "decode attention tokens/s and achieved HBM GB/s (% of GB300 peak) vs φ/branches"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dendrite")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the phi / MCTS / verify sweep, fork and memory")
    ap.add_argument("--sweep", action="store_true", help=argparse.SUPPRESS)   # the default; kept for old commands
    ap.add_argument("--sweep-set", default="", help="comma list of sweep workloads (default: all)")
    ap.add_argument("--no-sharing", action="store_true", help="ablation: every sequence reads its own blocks")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle CPU-baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cost-table", action="store_true",
                    help="print the verify cost table f(B, c, n) (one JSON line) and exit")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    return a


def workload(name: str, extra_steps: int, layers: int = 0):
    """Named workloads; `extra_steps` decode steps of headroom in the pool;
    `layers` > 0 overrides the layer count."""
    kw = {"layers": layers} if layers > 0 else {}
    if name == "dendrite":
        w = W.dendrite(**kw)
    elif name.startswith("trellis"):
        w = W.trellis(float(name[len("trellis"):] or 0.5), **kw)
    elif name == "mcts":
        w = W.mcts(**kw)
    elif name.startswith("verify"):
        w = W.verify_tree(int(name[len("verify"):] or 8), **kw)
    elif name == "tiny":
        w = W.tiny_fork()
    else:
        raise SystemExit(f"unknown workload {name}")
    bs = w.shapes.bs
    w.num_blocks += len(w.batch) * (extra_steps * w.step_tokens // bs + 3)
    w.max_blocks_per_seq += extra_steps * w.step_tokens // bs + 2
    return w


def describe(w) -> str:
    s = w.shapes
    base = f"{s.L} layers, {s.Hq}q/{s.Hkv}kv heads, d {s.d}, block {s.bs}, bf16"
    if w.name == "dendrite":
        return (f"Dendrite-shaped fork decode: TinyLlama-1.1B attention ({base}); 4096-token prefix "
                f"forked into 6 branches with private tokens {w.info['private']}; one decode token per "
                f"branch per step")
    if w.name.startswith("trellis"):
        return (f"Trellis-shaped prefix sweep: {base}; 64 sessions, L=512 prompt, phi={w.info['phi']} "
                f"(prefixBlocks={w.info['prefix_blocks']}), decode at length 576")
    if w.name == "mcts":
        return f"MCTS radix tree: Llama-3-8B attention ({base}); 2048-token root, 4-ary depth 4, 64/edge"
    if w.name.startswith("verify"):
        return (f"speculative tree verify: Llama-3-8B attention ({base}); B={len(w.batch)}, "
                f"context 2048, 64-node draft tree")
    return f"{w.name}: {base}"


# ---------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of x over all ranks (identity for one process).  NCCL reduces a
    device tensor; gloo (CPU tests) a host tensor."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def traffic_for(workload: str):
    """DRAM bytes per launch of the attention kernel(s) on `workload` from
    profiles/dram_traffic.json (ncu captures), if every kernel source it
    names still has the hash recorded there; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
        for e in data.get("entries", []):
            if e.get("workload") != workload:
                continue
            for src, sha in e.get("sources", {}).items():
                if hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest() != sha:
                    return None
            return e
    except (OSError, ValueError, KeyError, TypeError):
        pass
    return None


# ------------------------------------------------------------- our path

def run_ours(a, rank, world, local):
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    from paged_prefix_shared_decode_gb300.runner import PoolRunner, bf16_tensor

    kvp.load()   # fails loudly without the CUDA library
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    K, Wm = a.steps, a.warmup
    E2E = max(4, min(K, 10))
    w = workload(a.workload, Wm + 2 * K + 2 * E2E + 2, a.layers)
    if w.name.startswith("verify"):
        return run_verify_bench(a, w, rank, world, dev)
    s = w.shapes
    S = len(w.batch)
    r = PoolRunner(w, alloc_seed=1)
    r.run_ops()
    desc = r.attn_desc(use_sharing=not a.no_sharing)
    MB = w.max_blocks_per_seq

    # per-step inputs (host, generated once) and their device copies: warm-up,
    # the K timed steps, then K more steps that time the attention kernel
    nsteps = Wm + 2 * K
    host_kv = [W.step_kv(w, i) for i in range(nsteps + 2 * E2E)]
    host_q = [W.step_q(w, i) for i in range(nsteps + 2 * E2E)]
    kd = [bf16_tensor(k) for k, _ in host_kv[:nsteps]]
    vd = [bf16_tensor(v) for _, v in host_kv[:nsteps]]
    qd = [bf16_tensor(q) for q in host_q[:nsteps]]
    out = torch.empty((s.L, S, s.Hq, s.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s.L, S, s.Hq), dtype=torch.float32, device=dev)
    seqs = np.array([r.ids[n] for n in w.batch], np.int32)
    ntoks = np.full(S, w.step_tokens, np.int32)
    # workspace: twice what the starting state needs covers the growth of
    # the run (a few tokens per sequence)
    t0, l0 = kvp.kvp_gather_tables(r.pool, seqs, MB)
    ws_bytes = 2 * kvp.kvp_decode_workspace_size(desc, t0, l0) + (8 << 20)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e4 in ev:                       # materialise the CUDA events
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize(dev)

    # one step = kvp_decode_step on device buffers: append, plan from the
    # pool's tables, attention
    ios = [kvp.step_io(qd[i], out, lse, kd[i], vd[i]) for i in range(nsteps)]
    calls = [kvp.DecodeStep(r.pool, seqs, w.step_tokens, io, desc, ws, ws_bytes, stream=stream) for io in ios]

    def step(i, timed_events=None):
        if timed_events is not None:
            kvp.kvp_set_kernel_events(timed_events[2], timed_events[3])
        calls[i]()
        if timed_events is not None:
            kvp.kvp_set_kernel_events(None, None)

    for i in range(Wm):
        flush.fill_(i & 0xFF)
        step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = Clocks(local)
    clocks.start()
    # the timed steps: events around each whole step only, so that the step's
    # kernels follow one another directly in the stream (the attention kernel
    # may start while the append finishes, the merge while attention does)
    launches0 = kvp.kvp_kernel_launches()
    for j in range(K):
        flush.fill_(j & 0xFF)
        ev[j][0].record(stream)
        step(Wm + j)
        ev[j][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = kvp.kvp_kernel_launches() - launches0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [ev[j][0].elapsed_time(ev[j][1]) for j in range(K)]
    total_ms = max_over_ranks(float(sum(step_ms)), world)
    # K more steps with events right before and after the attention kernel
    # (which serialise it against its neighbours): its duration and the
    # unique bytes of each launch
    step_tables = []
    for j in range(K):
        flush.fill_(j & 0xFF)
        step(Wm + K + j, ev[j])
        step_tables.append(kvp.kvp_gather_tables(r.pool, seqs, MB))   # host only, between steps
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    kern_ms = [ev[j][2].elapsed_time(ev[j][3]) for j in range(K)]
    tokens = S * w.step_tokens * K * world
    value = tokens / (total_ms / 1e3)
    ub = [kvp.kvp_decode_plan_stats(desc, ht, hl)["unique_kv_bytes"] for ht, hl in step_tables]
    stats = kvp.kvp_decode_plan_stats(desc, *step_tables[-1])
    peak, peak_kind = peaks()
    bytes_per_launch = float(np.mean(ub))
    kern_avg = float(np.mean(kern_ms))
    achieved = bytes_per_launch / (kern_avg / 1e3) / 1e9
    tr = traffic_for(w.name)
    traffic = float(tr["dram_bytes_per_launch"]) if tr else None

    memory = memory_report(kvp, r, w, seqs, MB)
    # end to end through the public API with host buffers
    e2e = run_e2e(kvp, r, w, seqs, ntoks, desc, ws, ws_bytes, flush, stream, dev,
                  host_kv[nsteps:nsteps + E2E], host_q[nsteps:nsteps + E2E], MB, planned=True)
    e2e["single_call"] = run_e2e(kvp, r, w, seqs, ntoks, desc, ws, ws_bytes, flush, stream, dev,
                                 host_kv[nsteps + E2E:], host_q[nsteps + E2E:], MB, planned=False)

    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 K/V/Q, shapes of the workload)",
        "config": {"workload": describe(w), "name": w.name, "sequences": S,
                   "tokens_per_step": S * w.step_tokens, "use_sharing": not a.no_sharing,
                   "l2": "flushed between timed steps (write of 2x L2), outside the timed region",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "attn_item_kernel", "algorithmic_bytes_per_launch": bytes_per_launch,
                     "kernel_ms": kern_avg, "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "timing": f"CUDA events on the launching stream around the attention kernel, "
                               f"{K} steps run right after the timed ones"},
        "step_hbm": {"unique_kv_gb_per_s": bytes_per_launch / (total_ms / K / 1e3) / 1e9,
                     "frac_of_peak": bytes_per_launch / (total_ms / K / 1e3) / 1e9 / peak},
        "plan": stats,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
        "memory": memory,
    }
    return res, w


def run_e2e(kvp, r, w, seqs, ntoks, desc, ws, ws_bytes, flush, stream, dev, host_kv,
            host_q, MB, planned=True):
    """Same step through the public API from page-locked host buffers, wall
    clock per step with a stream synchronise at its end.

    planned: the decode loop in two halves (StepPlan): each step runs its
    planned device half (H2D of the step's K, V and Q in one copy kernel,
    plan upload, append, attention, out and lse written into host memory),
    then plans the next step (the append's bookkeeping and the attention plan)
    while the device works, then synchronises.  Steps 1 .. n-2 are counted:
    each holds one run and one plan.
    Otherwise one kvp_decode_step call per step (copies, bookkeeping, plan
    and launches in one call), first step dropped."""
    import torch
    s = w.shapes
    S = len(seqs)
    n = len(host_kv)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = [pin(k) for k, _ in host_kv]
    hv = [pin(v) for _, v in host_kv]
    hq = [pin(q) for q in host_q]
    kd = torch.empty_like(hk[0], device=dev)
    vd = torch.empty_like(hv[0], device=dev)
    qd = torch.empty_like(hq[0], device=dev)
    out = torch.empty((s.L, S, s.Hq, s.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s.L, S, s.Hq), dtype=torch.float32, device=dev)
    ho = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    hl_ = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    ios = [kvp.step_io(qd, out, lse, kd, vd, h_k_new=hk[i], h_v_new=hv[i], h_q=hq[i], h_out=ho, h_lse=hl_)
           for i in range(n)]
    times = []
    if planned:
        calls = [kvp.StepPlan(r.pool, seqs, w.step_tokens, io, desc, ws, ws_bytes, stream=stream) for io in ios]
        calls[0].plan()
        for i in range(n):
            flush.fill_(i & 0xFF)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            calls[i].run()
            if i + 1 < n:
                calls[i + 1].plan()
            stream.synchronize()
            times.append(time.perf_counter() - t0)
        for c in calls:
            c.close()
        counted = times[1:-1]
        how = ("wall clock per step: the planned device half of the step (one copy kernel for the H2D of "
               "k/v/q from page-locked host memory, plan upload, append, attention and merge writing out+lse "
               "into host memory), the host half of the next step (append bookkeeping, plan) while the "
               "device runs, and a stream synchronise; first and last step dropped")
    else:
        calls = [kvp.DecodeStep(r.pool, seqs, w.step_tokens, io, desc, ws, ws_bytes, stream=stream) for io in ios]
        for i in range(n):
            flush.fill_(i & 0xFF)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            calls[i]()
            stream.synchronize()
            times.append(time.perf_counter() - t0)
        counted = times[1:]
        how = ("wall clock per step: one kvp_decode_step call (H2D of k/v/q from page-locked host memory, "
               "append, host plan and its upload, attention, D2H of out+lse) and a stream synchronise; "
               "first step dropped")
    sec, cnt = float(np.sum(counted)), len(counted)
    h2d = hk[0].numel() * 2 * 2 + hq[0].numel() * 2
    d2h = out.numel() * 2 + lse.numel() * 4
    return {"value": S * w.step_tokens * cnt / sec, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": sec / cnt * 1e3, "how": how}


def run_verify_bench(a, w, rank, world, dev, single_layer=False):
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    from paged_prefix_shared_decode_gb300.runner import PoolRunner, VerifyCall

    g = torch.Generator(device=dev).manual_seed(w.seed)
    s = w.shapes

    def kv_dev(w_, i):
        n = w_.ops[i][2]
        shape = (s.L, n, s.Hkv, s.d)
        return (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16),
                torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))

    r = PoolRunner(w, alloc_seed=1)
    r.run_ops(kv_dev_fn=kv_dev)
    call = VerifyCall(r)
    B, n = call.B, call.n
    q = torch.randn((s.L, B * n, s.Hq, s.d), generator=g, device=dev).to(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    K = a.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e4 in ev:
        for e in e4:
            e.record(stream)
    for i in range(a.warmup):
        flush.fill_(i)
        call(q, stream=stream)
    torch.cuda.synchronize(dev)
    clocks = Clocks(dev.index)
    clocks.start()
    l0 = kvp.kvp_kernel_launches()
    for j in range(K):
        flush.fill_(j)
        ev[j][0].record(stream)
        kvp.kvp_set_kernel_events(ev[j][2], ev[j][3])
        call(q, stream=stream)
        kvp.kvp_set_kernel_events(None, None)
        ev[j][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = kvp.kvp_kernel_launches() - l0
    clk = clocks.stop()
    step_ms = [ev[j][0].elapsed_time(ev[j][1]) for j in range(K)]
    kern_ms = float(np.mean([ev[j][2].elapsed_time(ev[j][3]) for j in range(K)]))
    total = float(sum(step_ms))
    ub = sum((int(c) + n) for c in call.ctx) * s.token_bytes * s.L
    flops = 0
    for b in range(B):
        par = w.info["parents"][b]
        depth = np.zeros(n, int)
        for i in range(n):
            depth[i] = 1 if par[i] < 0 else depth[par[i]] + 1
        flops += 4 * s.d * s.Hq * s.L * int((call.ctx[b] * n + depth.sum()))
    peak, kind = peaks()
    achieved = ub / (kern_ms / 1e3) / 1e9
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        tpk = float(mp["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        tpk = 1900.0
    res = {
        "metric": METRIC, "value": B * n * K / (total / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": a.warmup, "ms_per_step": total / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (device-generated N(0,1) bf16 K/V/Q)",
        "config": {"workload": describe(w), "name": w.name, "query_tokens_per_step": B * n,
                   "l2": "flushed between timed steps, outside the timed region"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "attn_tc_kernel",
                     "algorithmic_bytes_per_launch": ub, "kernel_ms": kern_ms,
                     "tensor_tflops": flops / (kern_ms / 1e3) / 1e12, "tensor_peak_tflops": tpk,
                     "tensor_frac": flops / (kern_ms / 1e3) / 1e12 / tpk,
                     "peak_kind": f"{kind} hbm_gbs (copy); tensor: measured bf16_tflops (burst)"},
        "e2e": None, "gpu_launches": int(launches), "clocks": clk,
    }
    if single_layer:
        # one layer alone: the pools' layer 0, q / out / lse of layer 0
        d1 = kvp.AttnDesc(1, s.Hq, s.Hkv, s.d, s.bs, r.NB, 0.0, 1)
        w1 = kvp.kvp_verify_workspace_size(d1, call.h_tables, call.ctx, n)
        ws1 = torch.empty(w1, dtype=torch.uint8, device=dev)
        ms1, kms1 = _timed_calls(lambda: kvp.tree_verify_attention(
            q[:1], call.parent, n, r.k_pool, r.v_pool, call.h_tables, call.ctx, d1, call.out[:1], call.lse[:1],
            ws1, stream=stream), flush, stream)
        res["single_layer"] = {"ms_per_call": ms1, "kernel_ms": kms1}
    return res, w


def _timed_calls(call, flush, stream, reps=5, warm=3):
    """(ms per call, attention-kernel ms) over `reps` event-timed calls with L2
    flushed (outside the events) before each; `warm` untimed calls first."""
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for e4 in ev:
        for e in e4:
            e.record(stream)
    for _ in range(warm):
        call()
    for j in range(reps):
        flush.fill_(j & 0xFF)
        ev[j][0].record(stream)
        kvp.kvp_set_kernel_events(ev[j][2], ev[j][3])
        call()
        kvp.kvp_set_kernel_events(None, None)
        ev[j][1].record(stream)
    torch.cuda.synchronize()
    return (float(np.mean([e[0].elapsed_time(e[1]) for e in ev])),
            float(np.mean([e[2].elapsed_time(e[3]) for e in ev])))


def max_sm_mhz():
    """Maximum SM clock (MEASURED_PEAKS.json, else GB300's 2070 MHz)."""
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["sm_max_mhz"])
    except (OSError, KeyError, ValueError):
        return 2070.0


def tensor_peak():
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def sweep_decode(name, dev, alloc_seed=1):
    """One decode workload of the sweep: sharing on (the planned call) and off
    (every sequence reads its own blocks), and one layer alone.  alloc_seed 0:
    the pool hands out blocks in id order (the contiguous control)."""
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    from paged_prefix_shared_decode_gb300.runner import PoolRunner
    peak, _ = peaks()
    tpk, _ = tensor_peak()
    w = workload(name, 16)
    s = w.shapes
    g = torch.Generator(device=dev).manual_seed(1)

    def kv_dev(w_, i):
        n = w_.ops[i][2]
        shape = (s.L, n, s.Hkv, s.d)
        return (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16),
                torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))

    r = PoolRunner(w, alloc_seed=alloc_seed)
    r.run_ops(kv_dev_fn=kv_dev)
    S = len(w.batch)
    seqs = np.array([r.ids[n] for n in w.batch], np.int32)
    kv = torch.randn((s.L, S, s.Hkv, s.d), generator=g, device=dev).to(torch.bfloat16)
    r.append_step(kv, kv)
    ht, hl = kvp.kvp_gather_tables(r.pool, seqs, w.max_blocks_per_seq)
    q = torch.randn((s.L, S, s.Hq, s.d), generator=g, device=dev).to(torch.bfloat16)
    o = torch.empty((s.L, S, s.Hq, s.d), dtype=torch.bfloat16, device=dev)
    ls = torch.empty((s.L, S, s.Hq), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = kvp.kvp_decode_plan_stats(r.attn_desc(True), ht, hl)
    ub = st["unique_kv_bytes"]
    flops = 4 * s.d * s.Hq * int(hl.sum()) * s.L
    entry = {"workload": name + ("_contig" if alloc_seed == 0 else ""),
             "config": describe(w) + ("; blocks handed out in id order (alloc_seed 0)" if alloc_seed == 0 else ""),
             "sequences": S, "unique_kv_bytes": ub, "items": st["items"], "partial_rows": st["partial_rows"]}
    for sharing in (True, False):
        desc = r.attn_desc(use_sharing=sharing)
        wsb = kvp.kvp_decode_workspace_size(desc, ht, hl)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        ms, kms = _timed_calls(lambda: kvp.paged_decode_attention(q, r.k_pool, r.v_pool, ht, hl, desc, o, ls, ws,
                                                                  wsb, stream=stream), flush, stream)
        if sharing:
            entry.update({"kernel_ms": kms, "ms_per_call": ms, "tokens_per_s": S / (ms / 1e3),
                          "unique_gb_per_s": ub / (kms / 1e3) / 1e9, "frac": ub / (kms / 1e3) / 1e9 / peak,
                          "tensor_tflops": flops / (kms / 1e3) / 1e12,
                          "tensor_frac": flops / (kms / 1e3) / 1e12 / tpk})
            # one layer alone (the pools' layer 0, q / out / lse of layer 0)
            d1 = kvp.AttnDesc(1, s.Hq, s.Hkv, s.d, s.bs, r.NB, 0.0, 1)
            w1 = kvp.kvp_decode_workspace_size(d1, ht, hl)
            ws1 = torch.empty(w1, dtype=torch.uint8, device=dev)
            ms1, kms1 = _timed_calls(lambda: kvp.paged_decode_attention(q[:1], r.k_pool, r.v_pool, ht, hl, d1, o[:1],
                                                                        ls[:1], ws1, w1, stream=stream), flush, stream)
            entry["single_layer"] = {"ms_per_call": ms1, "kernel_ms": kms1}
        else:
            entry["sharing_off"] = {"kernel_ms": kms, "ms_per_call": ms,
                                    "unique_gb_per_s": ub / (kms / 1e3) / 1e9, "frac": ub / (kms / 1e3) / 1e9 / peak}
        del ws
    tr = traffic_for(w.name) if alloc_seed == 1 else None
    entry["traffic"] = float(tr["dram_bytes_per_launch"]) if tr else None
    r.close()
    del flush
    torch.cuda.empty_cache()
    return entry


def sweep_kv4(name, dev):
    """A decode workload on a pool of 4-bit pages: unique bytes in that format
    (d/2 code bytes + 1 exponent byte per row, K and V), kernel time, the HBM
    fraction of those bytes, tokens/s; the bf16 pool's figures are the
    matching entry without the suffix."""
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    from paged_prefix_shared_decode_gb300.runner import PoolRunner
    peak, _ = peaks()
    base = name[:-len("_kv4")]
    w = workload(base, 16)
    s = w.shapes
    g = torch.Generator(device=dev).manual_seed(1)

    def kv_dev(w_, i):
        n = w_.ops[i][2]
        shape = (s.L, n, s.Hkv, s.d)
        return (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16),
                torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))

    r = PoolRunner(w, alloc_seed=1, kv4=True)
    r.run_ops(kv_dev_fn=kv_dev)
    S = len(w.batch)
    seqs = np.array([r.ids[n] for n in w.batch], np.int32)
    kv = torch.randn((s.L, S, s.Hkv, s.d), generator=g, device=dev).to(torch.bfloat16)
    r.append_step(kv, kv)
    ht, hl = kvp.kvp_gather_tables(r.pool, seqs, w.max_blocks_per_seq)
    desc = r.attn_desc(True)
    st = kvp.kvp_decode_plan_stats(desc, ht, hl)
    ub4 = st["unique_kv_bytes"]   # in the 4-bit rows' bytes
    q = torch.randn((s.L, S, s.Hq, s.d), generator=g, device=dev).to(torch.bfloat16)
    o = torch.empty((s.L, S, s.Hq, s.d), dtype=torch.bfloat16, device=dev)
    ls = torch.empty((s.L, S, s.Hq), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    wsb = kvp.kvp_decode_workspace_size(desc, ht, hl)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ms, kms = _timed_calls(lambda: kvp.paged_decode_attention_kv4(q, r.k_pool, r.k_exp, r.v_pool, r.v_exp, ht, hl,
                                                                  desc, o, ls, ws, wsb, stream=stream), flush, stream)
    entry = {"workload": name, "config": describe(w) + "; 4-bit pages (codes + one exponent per row)",
             "sequences": S, "unique_kv_bytes": ub4, "bits_per_value": 4 + 8 / s.d,
             "kernel_ms": kms, "ms_per_call": ms, "tokens_per_s": S / (ms / 1e3),
             "unique_gb_per_s": ub4 / (kms / 1e3) / 1e9, "frac": ub4 / (kms / 1e3) / 1e9 / peak,
             "kernel": "attn_item_kernel<d, 4-bit> (and attn_tc_kernel<d, 4-bit> for items of more than "
                       "32 rows at head dim 128)", "traffic": None}
    tr = traffic_for(name)
    if tr:
        entry["traffic"] = float(tr["dram_bytes_per_launch"])
    r.close()
    del flush, ws
    torch.cuda.empty_cache()
    return entry


def sweep_trellis_loop(phi, dev, steps=64):
    """The Trellis benchmark's whole decode loop: from the sessions' prompts
    (length 512) through `steps` decode steps, each appending one token per
    session and attending over all layers (kvp_decode_step on device-resident
    inputs), timed as one block of steps with CUDA events."""
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    from paged_prefix_shared_decode_gb300.runner import PoolRunner
    w = W.trellis(phi, decode=1)   # the prompts only
    s = w.shapes
    g = torch.Generator(device=dev).manual_seed(1)

    def kv_dev(w_, i):
        n = w_.ops[i][2]
        shape = (s.L, n, s.Hkv, s.d)
        return (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16),
                torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))

    r = PoolRunner(w, alloc_seed=1)
    r.run_ops(kv_dev_fn=kv_dev)
    S = len(w.batch)
    seqs = np.array([r.ids[n] for n in w.batch], np.int32)
    desc = r.attn_desc(True)
    kd = torch.randn((steps, s.L, S, s.Hkv, s.d), generator=g, device=dev).to(torch.bfloat16)
    vd = torch.randn((steps, s.L, S, s.Hkv, s.d), generator=g, device=dev).to(torch.bfloat16)
    qd = torch.randn((steps, s.L, S, s.Hq, s.d), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty((s.L, S, s.Hq, s.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s.L, S, s.Hq), dtype=torch.float32, device=dev)
    t0, l0 = kvp.kvp_gather_tables(r.pool, seqs, w.max_blocks_per_seq)
    ws_bytes = 2 * kvp.kvp_decode_workspace_size(desc, t0, l0) + (8 << 20)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ios = [kvp.step_io(qd[i], out, lse, kd[i], vd[i]) for i in range(steps)]
    calls = [kvp.DecodeStep(r.pool, seqs, 1, io, desc, ws, ws_bytes, stream=stream) for io in ios]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for c in calls:
        c()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    _, ln = kvp.kvp_gather_tables(r.pool, seqs, w.max_blocks_per_seq)
    entry = {"workload": f"trellis{phi}_loop",
             "config": (f"Trellis-shaped decode loop: {s.L} layers, {s.Hq}q/{s.Hkv}kv heads, d {s.d}, block {s.bs}, "
                        f"bf16; 64 sessions from length 512 (phi={phi}, prefixBlocks={w.info['prefix_blocks']}) "
                        f"through {steps} decode steps (append one token per session, attention over all layers)"),
             "sequences": S, "steps": steps, "ms": ms, "ms_per_step": ms / steps,
             "tokens_per_s": S * steps / (ms / 1e3), "final_length": int(ln.max()),
             "how": "CUDA events around the block of steps (kvp_decode_step on device buffers: append, plan "
                    "from the pool's tables, attention, merge); no L2 flush between steps"}
    r.close()
    del ws, kd, vd, qd
    torch.cuda.empty_cache()
    return entry


def run_sweep(a, dev):
    """The rest of the metric beside the headline: the phi sweep, MCTS and
    verify on the device, the radix prefix cache on the host."""
    import torch
    import paged_prefix_shared_decode_gb300 as kvp
    out = []
    names = ["trellis0.0", "trellis0.25", "trellis0.5", "trellis0.75", "trellis0.9", "mcts",
             "verify1", "verify8", "verify32", "dendrite_kv4", "trellis0.0_kv4", "mcts_kv4",
             "radix0.5", "radix0.9", "dendrite_contig", "trellis0.0_loop", "trellis0.9_loop"]
    if a.sweep_set:
        names = [n for n in a.sweep_set.split(",") if n]
    for name in names:
        if name.startswith("radix"):
            out.append(prefix_cache_bench(kvp, float(name[len("radix"):]), with_oracle=not a.no_cpu_baseline))
            continue
        if name.endswith("_kv4"):
            out.append(sweep_kv4(name, dev))
            continue
        if name.endswith("_contig"):
            out.append(sweep_decode(name[:-len("_contig")], dev, alloc_seed=0))
            continue
        if name.endswith("_loop"):
            out.append(sweep_trellis_loop(float(name[len("trellis"):-len("_loop")]), dev))
            continue
        if name.startswith("verify"):
            sub = argparse.Namespace(**vars(a))
            sub.steps, sub.warmup = 5, 3
            res, w = run_verify_bench(sub, workload(name, 0), 0, 1, dev, single_layer=True)
            rf = res["roofline"]
            # third bound: one exp per (query row, key attended), at the
            # ex2.approx.ftz.f32 rate a probe measured on this GPU (about 60
            # results per clock per SM), at the maximum SM clock
            exps = rf["tensor_tflops"] * 1e12 * rf["kernel_ms"] / 1e3 / (4 * w.shapes.d)
            props = torch.cuda.get_device_properties(dev)
            exp_ms = exps / (60.0 * props.multi_processor_count * max_sm_mhz() * 1e6) * 1e3
            out.append({"workload": name, "config": describe(w), "query_tokens": res["config"]["query_tokens_per_step"],
                        "unique_kv_bytes": rf["algorithmic_bytes_per_launch"], "kernel_ms": rf["kernel_ms"],
                        "ms_per_call": res["ms_per_step"], "tokens_per_s": res["value"],
                        "unique_gb_per_s": rf["achieved"], "frac": rf["frac"],
                        "tensor_tflops": rf["tensor_tflops"], "tensor_frac": rf["tensor_frac"],
                        "exp_bound": {"exps": exps, "ms": exp_ms, "frac": exp_ms / rf["kernel_ms"],
                                      "rate": "60 ex2 results per clock per SM (probe on this GPU), max SM clock"},
                        "single_layer": res["single_layer"], "traffic": None})
            torch.cuda.empty_cache()
            continue
        out.append(sweep_decode(name, dev))
    return out


def fork_bench(kvp, reps: int = 100000):
    """Host cost of seq_fork + seq_free on the Dendrite parent (4096 tokens =
    256 blocks of 16) through the C ABI, next to the device copy of that
    context's K/V (all 22 layers) that a fork avoids."""
    import ctypes
    import torch
    from paged_prefix_shared_decode_gb300.runner import PoolRunner
    w = W.dendrite()
    r = PoolRunner(w, alloc_seed=1, device=False)
    r.run_ops(device_kv=False)
    parent = r.ids[0]
    lib = kvp.load()
    child = ctypes.c_int32()
    nb = ctypes.c_int32()
    tbl = np.zeros(w.max_blocks_per_seq, np.int32)
    lib.seq_block_table(r.pool, parent, tbl.ctypes.data_as(ctypes.c_void_p), len(tbl), ctypes.byref(nb))
    per = []
    for _ in range(reps // 1000):
        t0 = time.perf_counter_ns()
        for _ in range(1000):
            lib.seq_fork(r.pool, parent, ctypes.byref(child))
            lib.seq_free(r.pool, child.value)
        per.append((time.perf_counter_ns() - t0) / 1000 / 1e3)
    r.close()
    # the copy a fork avoids: the parent's K and V of every layer on the device
    nbytes = w.info["prefix"] * w.shapes.token_bytes * w.shapes.L
    src = torch.empty(nbytes // 2, dtype=torch.bfloat16, device="cuda")
    dst = torch.empty_like(src)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        dst.copy_(src)
    e0.record()
    for _ in range(10):
        dst.copy_(src)
    e1.record()
    torch.cuda.synchronize()
    return {"parent_tokens": w.info["prefix"], "parent_blocks": int(nb.value),
            "fork_plus_free_us_median": float(np.median(per)), "fork_plus_free_us_min": float(np.min(per)),
            "reps": reps, "api": "one ctypes call each for seq_fork and seq_free (call overhead included)",
            "device_copy_of_parent_kv_ms": e0.elapsed_time(e1) / 10, "parent_kv_bytes": int(nbytes),
            "pages_context": "Dendrite: ~3 us fork at 4K context vs 50-100 ms copying (other hardware)"}


def memory_report(kvp, r, w, seqs, MB):
    """KV blocks and bytes the batch holds with sharing, and what it would
    hold if every branch had its own copy of its blocks."""
    s = w.shapes
    t, ln = kvp.kvp_gather_tables(r.pool, seqs, MB)
    nblk = [(int(x) + s.bs - 1) // s.bs for x in ln]
    rows = [t[i, :nblk[i]] for i in range(len(seqs))]
    unique = len(set(np.concatenate(rows).tolist()))
    private = sum(nblk)
    block_bytes = s.L * s.Hkv * s.bs * s.d * 2 * 2
    res = {"blocks_shared": unique, "blocks_unshared": private, "block_bytes": block_bytes,
           "kv_bytes_shared": unique * block_bytes, "kv_bytes_unshared": private * block_bytes,
           "saved_frac": 1.0 - unique / private}
    if w.name == "dendrite":
        res["pages_context"] = "Dendrite: 1.1 GB vs 6 GB for a 4K prefix x 6 branches (>80% saved; model and " \
                               "precision unstated)"
    return res


# ------------------------------------------------- verify cost table (CAST)

def cost_table(a, dev):
    """Tree-verify cost f(B, c, n) on this GPU, the table CAST's tree-size
    choice consumes ("CAST", section on the verification cost model: the
    cost of verifying n draft tokens grows with batch size B, context c and
    n).  Llama-3-8B shapes, 32 layers, block 16, random draft trees of depth
    <= 8; per point the event-timed verify call (plan upload, tree masks,
    attention, merge) with L2 flushed between calls."""
    rows = []
    for B in (1, 4, 16, 32):
        for c in (512, 2048, 8192):
            for n in (16, 32, 64):
                sub = argparse.Namespace(**vars(a))
                sub.steps, sub.warmup = 5, 3
                w = W.verify_tree(B, layers=32, ctx=c, n_draft=n)
                res, _ = run_verify_bench(sub, w, 0, 1, dev)
                rows.append({"B": B, "c": c, "n": n, "ms": res["ms_per_step"],
                             "kernel_ms": res["roofline"]["kernel_ms"],
                             "tensor_tflops": res["roofline"]["tensor_tflops"],
                             "hbm_frac": res["roofline"]["frac"]})
                import torch
                torch.cuda.empty_cache()
    return rows


# ---------------------------------------------------- prefix cache (host)

def _prefix_cache_op(api, system, prompts, fulls, bs):
    """One pass of the Trellis session pattern through a prefix cache: warm
    the system prompt, then per session match its prompt, start from the
    cached blocks, take blocks for the rest of the prompt and the decoded
    tokens, cache the finished session (fulls: prompt + decoded tokens),
    unlock, free.  Returns (seconds, matched tokens)."""
    pool, cache = api["new"]()
    s = api["alloc"](pool)
    api["reserve"](pool, s, len(system))
    api["insert"](cache, system, api["table"](pool, s))
    api["free"](pool, s)
    matched = 0
    t0 = time.perf_counter()
    for prompt, full in zip(prompts, fulls):
        got, lock = api["match"](cache, prompt)
        matched += len(got) * bs
        s = api["alloc_prefix"](pool, got)
        api["reserve"](pool, s, len(full) - len(got) * bs)
        api["insert"](cache, full, api["table"](pool, s))
        api["unlock"](cache, lock)
        api["free"](pool, s)
    dt = time.perf_counter() - t0
    api["close"](pool, cache)
    return dt, matched


def prefix_cache_bench(kvp, phi: float, with_oracle: bool, reps: int = 5):
    """Host cost per session of the radix prefix cache through the public
    API (bookkeeping pool, no device K/V), on the Trellis benchmark's session
    pattern (64 sessions, 512-token prompts sharing 32 * round(phi * 512 / 32)
    tokens, 64 decoded tokens each, 32-token blocks); the oracle beside it."""
    import workloads as W
    bs, sessions = 32, 64
    system, prompts, generated = W.prefix_cache_sessions(phi, sessions=sessions)
    nb = sessions * (len(prompts[0]) + len(generated[0])) // bs + 64
    mb = (len(prompts[0]) + len(generated[0])) // bs + 2

    def lib_new():
        pool = kvp.kv_pool_create(kvp.PoolDesc(1, nb, bs, 1, 64, sessions + 2, mb, 1))
        return pool, kvp.kvp_radix_create(pool)

    def lib_close(pool, cache):
        kvp.kvp_radix_destroy(cache)
        kvp.kv_pool_destroy(pool)

    lib = {"new": lib_new, "close": lib_close, "alloc": kvp.seq_alloc, "free": kvp.seq_free,
           "reserve": lambda p, s, n: kvp.seq_reserve(p, s, n), "table": kvp.seq_block_table,
           "insert": kvp.kvp_radix_insert, "alloc_prefix": kvp.seq_alloc_prefix,
           "match": lambda c, t: kvp.kvp_radix_match(c, t), "unlock": kvp.kvp_radix_unlock}
    np_sys = np.asarray(system, np.int32)
    np_prompts = [np.asarray(p, np.int32) for p in prompts]
    np_fulls = [np.asarray(p + g, np.int32) for p, g in zip(prompts, generated)]
    runs = [_prefix_cache_op(lib, np_sys, np_prompts, np_fulls, bs) for _ in range(reps)]
    dt = float(np.median([r[0] for r in runs]))
    # one match + unlock through ctypes on preallocated buffers (the C call
    # itself, without the binding's array handling)
    import ctypes
    lib_ = kvp.load()
    pool, cache = lib_new()
    s = kvp.seq_alloc(pool)
    kvp.seq_reserve(pool, s, len(system))
    kvp.kvp_radix_insert(cache, np_sys, kvp.seq_block_table(pool, s))
    q = np_prompts[0]
    buf = np.zeros(len(q) // bs, np.int32)
    nb_, lk = ctypes.c_int32(), ctypes.c_int32()
    qp, bp = q.ctypes.data_as(ctypes.c_void_p), buf.ctypes.data_as(ctypes.c_void_p)
    t0 = time.perf_counter()
    for _ in range(2000):
        lib_.kvp_radix_match(cache, qp, len(q), bp, len(buf), ctypes.byref(nb_), ctypes.byref(lk))
        lib_.kvp_radix_unlock(cache, lk.value)
    match_us = (time.perf_counter() - t0) / 2000 * 1e6
    lib_close(pool, cache)
    res = {"workload": f"radix{phi}", "sessions": sessions, "block": bs,
           "match_unlock_us": match_us,
           "host_us_per_session": dt / sessions * 1e6,
           "hit_frac": runs[0][1] / sum(len(p) for p in prompts),
           "api": "Python binding over the C ABI, int32 token arrays (match, seq_alloc_prefix, "
                  "seq_reserve, insert, unlock, seq_free per session)"}
    if with_oracle:
        import oracle

        def or_new():
            m = oracle.PoolModel(nb, bs, sessions + 2, mb, alloc_seed=1)
            return m, oracle.RadixModel(m)

        orc = {"new": or_new, "close": lambda p, c: None, "alloc": lambda p: p.alloc(),
               "free": lambda p, s: p.free_seq(s), "reserve": lambda p, s, n: p.append(s, n),
               "table": lambda p, s: p.table(s), "insert": lambda c, t, b: c.insert(t, list(b)),
               "alloc_prefix": lambda p, b: p.alloc_prefix(b), "match": lambda c, t: c.match(t),
               "unlock": lambda c, lk: c.unlock(lk)}
        fulls = [p + g for p, g in zip(prompts, generated)]
        oruns = [_prefix_cache_op(orc, system, prompts, fulls, bs) for _ in range(2)]
        assert oruns[0][1] == runs[0][1]
        res["cpu_baseline"] = {"kind": "oracle", "cores": 1,
                               "host_us_per_session": float(np.median([r[0] for r in oruns])) / sessions * 1e6}
    return res


# -------------------------------------------------------- oracle timing

def oracle_time(w, seconds: float, max_steps: int | None = None):
    """The fp64 oracle, as it stands, on full decode steps of the workload
    (all layers, sequences and heads) on the host cores.  Returns
    (tokens/s, steps, cores, seconds)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    rw = oracle.replay(w, alloc_seed=1)
    steps = 0
    t_total = 0.0
    while True:
        if w.step_tokens:
            k, v = W.step_kv(w, steps)
            oracle.replay_step(rw, w, k, v)
        q = W.step_q(w, steps)
        t, ln = rw.tables(w.batch, w.max_blocks_per_seq)
        t0 = time.perf_counter()
        oracle.decode_attention(q, rw.k_pool, rw.v_pool, t, ln, threads=cores)
        t_total += time.perf_counter() - t0
        steps += 1
        if (max_steps is not None and steps >= max_steps) or (max_steps is None and t_total >= seconds):
            break
    tokens = steps * len(w.batch) * max(1, w.step_tokens)
    return tokens / t_total, steps, cores, t_total


def run_reference(a, rank, world):
    if rank != 0:
        return None
    w = workload(a.workload, a.warmup + a.steps + 2, a.layers)
    if w.name.startswith("verify"):
        print(json.dumps({"impl": "reference", "unavailable": "oracle arm times decode workloads only"}))
        return None
    import oracle
    cores = len(os.sched_getaffinity(0))
    rw = oracle.replay(w, alloc_seed=1)
    times = []
    for i in range(a.warmup + a.steps):
        if w.step_tokens:
            k, v = W.step_kv(w, i)
            oracle.replay_step(rw, w, k, v)
        q = W.step_q(w, i)
        t, ln = rw.tables(w.batch, w.max_blocks_per_seq)
        t0 = time.perf_counter()
        oracle.decode_attention(q, rw.k_pool, rw.v_pool, t, ln, threads=cores)
        if i >= a.warmup:
            times.append(time.perf_counter() - t0)
    total = float(np.sum(times))
    S = len(w.batch)
    value = S * max(1, w.step_tokens) * a.steps / total
    sample = (f"each step: one full decode step of the workload ({w.shapes.L} layers x {S} sequences x "
              f"{w.shapes.Hq} heads) by the fp64 oracle")
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": total / a.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": describe(w), "name": w.name},
           "cpu_baseline": {"kind": "oracle", "value": value, "unit": "tokens/s", "cores": cores,
                            "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return res


def main():
    a = parse()
    rank, world, local = dist_env()
    if a.impl == "reference":
        res = run_reference(a, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if a.cost_table:
        if rank == 0:
            import torch
            print(json.dumps({"cost_table": cost_table(a, torch.device("cuda", local)),
                              "unit": "ms per verify call"}), flush=True)
        return 0
    res, w = run_ours(a, rank, world, local)
    if rank == 0:
        import torch
        if not a.no_sweep:
            res["sweep"] = run_sweep(a, torch.device("cuda", local))
            import paged_prefix_shared_decode_gb300 as kvp
            res["fork"] = fork_bench(kvp)
        if not a.no_cpu_baseline and not w.name.startswith("verify"):
            v, steps, cores, sec = oracle_time(w, a.cpu_seconds)
            res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                   "sample": f"{steps} full decode steps of the same workload "
                                             f"({sec:.1f} s of oracle time)"}
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
