"""Throughput of the speculative-decoding verification cycle on GB300.

One step = one pass of the whole hot path over one batch of the throughput
workload (B = 64 requests, k = 4 drafts, V = 128256, bf16 target and draft
logits, T = 0.8, top-p 0.95 on p and q, paged KV with 16-slot blocks,
S_b ~ U[128, 8192]):
    bfl_reserve  (lookahead blocks for the verify pass)
    spec_verify  (accept / reject / correction or bonus per request)
    kv_commit_rollback (commit the accepted prefix, free the rejected tail)
The metric is verified rows per second (sum_b (k_b + 1) target rows per
step).  Inputs rotate over 4 independent batches (4 x 148 MB, larger than L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on this host as the reference arm
(a bounded sample of the same workload per step).  Under torchrun (N > 1)
every rank runs its own batch (the path shards by request; no collective on
the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = dict(workload="verify_b64_k4", B=64, k=4, V=128256, input_dtype="bf16",
                temperature=0.8, top_p=0.95, block_size=16, prefix="U[128,8192]")
METRIC = "verify rows/s & HBM GB/s vs 8 TB/s at B=64 k=4 V=128256 bf16"
N_SETS = 4


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.cmd = ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", str(period_ms)]
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def build_sets(n_sets):
    from speculative_decoding_verification_07_gb300 import workloads as W
    sets = []
    for s in range(n_sets):
        inp = W.verify_b64_k4(index=5 + 97 * s)
        inp["seed"] = 2005 + s
        sets.append(inp)
    return sets


def rows_per_step(inp):
    return int((inp["k"].astype(np.int64) + 1).sum())


def full_bytes(inp):
    """B_full: every target row (k_b + 1) and draft row (k_b) of the batch, plus
    the per-request metadata read and written (tokens, k, T, top_p, ids,
    seq_len, outputs)."""
    V = inp["target"].shape[-1]
    k = inp["k"].astype(np.int64)
    rows = ((k + 1) * V * 2 + k * V * 2).sum()
    meta = (4 * k + 4 * (k + 1) + 24).sum()
    return int(rows + meta)


def needed_bytes(inp, accepted):
    """B_min: the rows the method must read -- target rows 0..a_b and draft rows
    0..min(a_b, k_b - 1) (every row after the first rejection is discarded); a
    request refused at row 0 (a_b = -1) still had row 0 read."""
    V = inp["target"].shape[-1]
    k = inp["k"].astype(np.int64)
    a = np.maximum(np.asarray(accepted, np.int64), 0)
    return int(((a + 1) * V * 2 + np.minimum(a + 1, k) * V * 2).sum())


# --------------------------------------------------------------------------- #
# reference arm: the fp64 oracle on the host
# --------------------------------------------------------------------------- #
_REF_INP = None


def _ref_init():
    """Pool initializer of the reference arm: each process holds the workload."""
    global _REF_INP
    _REF_INP = build_sets(1)[0]


def _ref_walk(b):
    """One request walk of the oracle in a pool process; returns its rows."""
    from oracle import sampling as S
    inp = _REF_INP
    kb = int(inp["k"][b])
    S.verify_request(S.decode(inp["target"][b, :kb + 1], "bf16"),
                     S.decode(inp["draft"][b, :kb], "bf16"), inp["tokens"][b, :kb], kb,
                     inp["temperature"][b], inp["top_p"][b], "logits", inp["seed"],
                     int(inp["request_id"][b]), int(inp["seq_len"][b]))
    return kb + 1


def run_reference(args):
    """The oracle on the host's cores: one spawned process per core; a step is
    one request walk per process (nproc requests of the batch, in turn)."""
    import multiprocessing as mp
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    nproc = args.ref_procs if args.ref_procs > 0 else (os.cpu_count() or 1)
    B = 64
    with mp.get_context("spawn").Pool(nproc, initializer=_ref_init) as pool:
        def step(t):
            return sum(pool.map(_ref_walk, [(t * nproc + r) % B for r in range(nproc)], chunksize=1))

        t0 = time.perf_counter()
        step(0)
        per = time.perf_counter() - t0
        budget = 180.0
        steps = args.steps
        if (args.steps + args.warmup) * per > budget:
            steps = max(3, int(budget / per) - args.warmup)
        for t in range(args.warmup):
            step(t)
        rows = 0
        t0 = time.perf_counter()
        for t in range(steps):
            rows += step(t)
        el = time.perf_counter() - t0
    value = rows / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": ws, "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(WORKLOAD, sample=f"{nproc} requests of the batch per step, one per "
                                            f"process (k_b + 1 rows each)",
                           parallelism=f"{nproc} host processes"),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nproc, "kind": "oracle",
                             "sample": f"{steps} steps of {nproc} request walks of one "
                                       f"verify_b64_k4 batch"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(inp, seconds=12.0):
    """The oracle as it stands on this host, bounded to about `seconds`."""
    from oracle import sampling as S
    B = inp["k"].shape[0]
    rows = n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or n < 2:
        b = n % B  # cycles over the batch's requests
        kb = int(inp["k"][b])
        S.verify_request(S.decode(inp["target"][b, :kb + 1], "bf16"),
                         S.decode(inp["draft"][b, :kb], "bf16"), inp["tokens"][b, :kb], kb,
                         inp["temperature"][b], inp["top_p"][b], "logits", inp["seed"],
                         int(inp["request_id"][b]), int(inp["seq_len"][b]))
        rows += kb + 1
        n += 1
    el = time.perf_counter() - t0
    return {"value": rows / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} request walks cycling over the {B} requests of one verify_b64_k4 "
                      f"batch ({rows} rows, {el:.1f} s, numpy fp64, one thread)"}


def _oracle_worker(job):
    """One process of the all-cores oracle baseline: its own copy of the
    workload, then request walks (every nproc-th request) for about `seconds`."""
    rank, nproc, seconds = job
    from oracle import sampling as S
    inp = build_sets(1)[0]
    B = inp["k"].shape[0]
    rows = n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or n < 1:
        b = (rank + n * nproc) % B
        kb = int(inp["k"][b])
        S.verify_request(S.decode(inp["target"][b, :kb + 1], "bf16"),
                         S.decode(inp["draft"][b, :kb], "bf16"), inp["tokens"][b, :kb], kb,
                         inp["temperature"][b], inp["top_p"][b], "logits", inp["seed"],
                         int(inp["request_id"][b]), int(inp["seq_len"][b]))
        rows += kb + 1
        n += 1
    return rows, n, time.perf_counter() - t0


def cpu_baseline_all_cores(seconds=12.0):
    """The oracle on every host core: one spawned process per core (spawned,
    since the parent has used the GPU), each timing its own walks."""
    import multiprocessing as mp
    nproc = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(nproc) as pool:
        res = pool.map(_oracle_worker, [(r, nproc, seconds) for r in range(nproc)])
    rows = sum(r for r, _, _ in res)
    walks = sum(w for _, w, _ in res)
    el = max(t for _, _, t in res)
    return {"value": rows / el, "unit": "rows/s", "cores": nproc, "kind": "oracle",
            "sample": f"{nproc} processes, {walks} request walks of one verify_b64_k4 batch "
                      f"({rows} rows, {el:.1f} s each at most, numpy fp64)"}


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def run_ours(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_07_gb300 import binding, device_io, replicas

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if ws > 1:
            dist.barrier()

    sets = build_sets(N_SETS)
    B, k, V = 64, 4, 128256
    rows = rows_per_step(sets[0])
    ver = binding.Verifier(local)
    dsets = [device_io.to_device(s, dev) for s in sets]
    for d in dsets:
        d["request_id"] = replicas.rank_request_ids(d["request_id"], rank)
    BS = 16
    N_LONG = 2000  # steps of the longer (context) region below
    steps_total = args.warmup + args.steps + N_LONG + 64 * 6 + 64
    max_blocks = (8192 + (k + 1) * steps_total) // BS + 4
    pool = binding.BlockPool(ver.handle, B * max_blocks, BS)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32, device=dev)
    seq = torch.zeros(B, dtype=torch.int32, device=dev)
    S0 = torch.tensor(sets[0]["seq_len"], dtype=torch.int32, device=dev)
    pool.reserve(seq, S0 - 1, table)
    seq.copy_(S0)
    kk = dsets[0]["k"]
    outs = [ver.outputs(B, k) for _ in range(N_SETS)]
    ev = {}
    evs = {}

    def step(i, stream=None, timed_verify=False, top_p=None, timed_small=False):
        d = dsets[i % N_SETS]
        o = outs[i % N_SETS]
        if timed_small:
            torch.cuda._sleep(200_000)
            evs[i][0].record()
        pool.reserve(seq, kk, table, stream=stream)
        if timed_small:
            evs[i][1].record()
        a = binding.make_args(target=d["target"], draft=d["draft"], draft_tokens=d["draft_tokens"],
                              temperature=d["temperature"], k=d["k"],
                              top_p=d["top_p"] if top_p is None else top_p,
                              seed=d["seed"], request_id=d["request_id"], seq_len=seq,
                              draft_kind="logits", **o)
        wsp = ver.ensure_workspace(a)
        if timed_verify:
            # keep the stream busy while the host enqueues event, kernel, event,
            # so the events bracket the kernel alone
            torch.cuda._sleep(200_000)
            ev[i][0].record()
        binding.spec_verify(ver.handle, a, wsp, stream)
        if timed_verify:
            ev[i][1].record()
        if timed_small:
            evs[i][2].record()
        pool.commit_rollback(kk, o["accepted"], seq, table, stream=stream)
        if timed_small:
            evs[i][3].record()

    # warm-up (eager), then capture a graph of G steps cycling the input sets
    # and a graph of one step, so that exactly args.steps steps are timed
    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    assert ver.error() == 0, "device error during warm-up"
    G = 8
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    graph, graph1 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for i in range(G):
                step(i, stream=s)
        with torch.cuda.graph(graph1, stream=s):
            step(0, stream=s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(2):
            graph.replay()
    torch.cuda.synchronize()

    K = max(1, args.steps)
    reps, tail = K // G, K % G
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    nvtx = _Nvtx()
    nvtx.range_push("timed steps (graph replays)")
    with ClockSampler(local) as clk, torch.cuda.stream(s):
        t0e.record(s)
        for _ in range(reps):
            graph.replay()      # replays on the current stream, s
        for _ in range(tail):
            graph1.replay()
        t1e.record(s)
        torch.cuda.synchronize()
    barrier()
    ms = t0e.elapsed_time(t1e)
    assert ver.error() == 0, "device error in the timed region"
    value, ms = replicas.whole_job_rate(ms, rows * K, device=dev)
    # the same steps over a longer region (a steadier figure; context only)
    nlong = max(G, (N_LONG // G) * G)
    with torch.cuda.stream(s):
        t0e.record(s)
        for _ in range(nlong // G):
            graph.replay()
        t1e.record(s)
        torch.cuda.synchronize()
    long_ms = t0e.elapsed_time(t1e) / nlong
    nvtx.range_pop()
    # verify-kernel duration: CUDA events around each launch of G more steps
    nvtx.range_push("per-launch kernel timings")
    nv = 4 * G
    for i in range(nv):
        ev[i] = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for i in range(nv):
        step(i, timed_verify=True)
    torch.cuda.synchronize()
    vms = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) for i in range(nv)]))
    bfull = float(np.mean([full_bytes(sets[i % N_SETS]) for i in range(N_SETS)]))
    bmin = float(np.mean([needed_bytes(sets[i % N_SETS], outs[i % N_SETS]["accepted"].cpu().numpy())
                          for i in range(N_SETS)]))
    peak, peak_src = measured_peaks()
    achieved = bfull / (vms / 1e3) / 1e9
    # the same kernel with top_p = 1 on p and q (no nucleus filter)
    ones = torch.ones(B, dtype=torch.float32, device=dev)
    for i in range(nv):
        step(i, timed_verify=True, top_p=ones)
    torch.cuda.synchronize()
    vms1 = float(np.mean([ev[i][0].elapsed_time(ev[i][1]) for i in range(nv)]))
    # the step's two small kernels on their own
    for i in range(nv):
        evs[i] = tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
    for i in range(nv):
        step(i, timed_small=True)
    torch.cuda.synchronize()
    reserve_us = float(np.mean([evs[i][0].elapsed_time(evs[i][1]) for i in range(nv)])) * 1e3
    commit_us = float(np.mean([evs[i][2].elapsed_time(evs[i][3]) for i in range(nv)])) * 1e3
    assert ver.error() == 0, "device error in the kernel timings"
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "verify_traffic.json")
    if os.path.exists(tpath):
        try:
            tj = json.load(open(tpath))
            if tj.get("kernel_source_sha") == kernel_source_sha():
                traffic = tj.get("bytes_per_launch")
        except Exception:
            traffic = None

    # end to end through the public API with host buffers (pinned)
    nvtx.range_pop()
    nvtx.range_push("end to end with host buffers")
    e2e = e2e_run(ver, sets, dev, args, pool, table, seq, kk, B, k)
    nvtx.range_pop()
    nvtx.range_push("commit by copy")
    copy_line = commit_copy_run(ver, sets, outs, dev, peak)
    nvtx.range_pop()
    nvtx.range_push("token trees")
    tree_line = tree_run(ver, dev, peak)
    nvtx.range_pop()
    nvtx.range_push("configurations")
    legs = config_legs(ver, dev, peak) if not args.no_legs else {"skipped": "--no-legs"}
    nvtx.range_pop()

    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(WORKLOAD, parallelism=f"replicas x{ws} (requests shard, no collective)",
                           step="bfl_reserve + spec_verify + kv_commit_rollback",
                           launch=f"CUDA graphs of {G} steps and of 1 step (programmatic "
                                  f"dependent launches between the step's kernels)",
                           l2=f"inputs rotate over {N_SETS} batches of "
                              f"{full_bytes(sets[0]) / 1e6:.1f} MB (> L2)"),
            "gpu_launches": 3 * K,
            "ms_per_step_long": long_ms, "steps_long": nlong,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "verify_kernel<bf16,bf16>",
                         "kernel_ms": vms, "bytes_full_per_launch": bfull,
                         "bytes_needed_per_launch": bmin,
                         "achieved_needed": bmin / (vms / 1e3) / 1e9,
                         "peak_source": peak_src,
                         "frac_of_8tbs": achieved / 8000.0},
            "verify_top_p_1": {"kernel_ms": vms1, "achieved": bfull / (vms1 / 1e3) / 1e9,
                               "frac": bfull / (vms1 / 1e3) / 1e9 / peak},
            "small_kernels_us": {"bfl_reserve": reserve_us, "kv_commit_rollback": commit_us},
            "clocks": clk.summary(),
            "e2e": e2e,
            "kv_commit_copy": copy_line, "tree_verify": tree_line,
            "configs": legs}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sets[0])
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
    if rank == 0:
        print(json.dumps(line), flush=True)
    ver.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


def e2e_run(ver, sets, dev, args, pool, table, seq, kk, B, k):
    """rows/s through the public API with the step's inputs in pinned host
    memory: per step, the H2D copy of its inputs, reserve + verify + commit,
    and the D2H read of its outputs.  Two device input buffers let the H2D copy
    of step i+1 (on a copy stream) run while step i computes, as a serving loop
    would; every step still moves all of its own bytes inside the timed region."""
    import torch

    from speculative_decoding_verification_07_gb300 import device_io
    hsets = [device_io.to_device(s, None, pin=True) for s in sets]
    dbufs = [device_io.to_device(sets[0], dev) for _ in range(2)]
    o = ver.outputs(B, k)
    ho = {key: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for key, v in o.items()}
    keys = ("target", "draft", "draft_tokens", "k", "temperature", "top_p", "request_id")
    h2d = sum(hsets[0][key].numel() * hsets[0][key].element_size() for key in keys)
    d2h = sum(v.numel() * v.element_size() for v in ho.values())
    n = max(8, min(64, args.steps // 20))
    comp = torch.cuda.current_stream(dev)
    cps = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]

    def load(i):
        j = i % 2
        cps.wait_event(ev_free[j])          # step i-2 is done with buffer j
        with torch.cuda.stream(cps):
            h = hsets[i % N_SETS]
            for key in keys:
                dbufs[j][key].copy_(h[key], non_blocking=True)
        ev_in[j].record(cps)

    def run(i):
        j = i % 2
        d = dbufs[j]
        comp.wait_event(ev_in[j])
        pool.reserve(seq, d["k"], table)
        ver.verify(target=d["target"], draft=d["draft"], draft_tokens=d["draft_tokens"],
                   temperature=d["temperature"], k=d["k"], top_p=d["top_p"],
                   seed=hsets[i % N_SETS]["seed"], request_id=d["request_id"], seq_len=seq, out=o)
        pool.commit_rollback(d["k"], o["accepted"], seq, table)
        ev_free[j].record(comp)
        for key in o:
            ho[key].copy_(o[key], non_blocking=True)

    def steps(n0, count, e0=None):
        if e0 is not None:
            cps.wait_event(e0)
        load(n0)
        for i in range(n0, n0 + count):
            if i + 1 < n0 + count:
                load(i + 1)
            run(i)

    steps(0, 3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    steps(3, n, e0)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    rows = rows_per_step(sets[0])
    return {"value": rows * n / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n,
            "overlap": "H2D of step i+1 on a copy stream while step i computes (two input buffers)"}


def graph_us_per_call(fn, n_calls, replays, dev):
    """Microseconds per call of fn(i, stream), i = 0 .. n_calls - 1, captured
    once in a CUDA graph on a side stream and replayed `replays` times after
    two untimed replays: the host's launch cost stays out of the timed region."""
    import torch
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(n_calls):
                fn(i, s)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(2):
            g.replay()
        e0.record(s)
        for _ in range(replays):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / (replays * n_calls) * 1e3
    del g
    return us


def commit_copy_run(ver, sets, outs, dev, peak):
    """The commit-by-copy kernel at the workload's KV shape (32 layers x 8 KV
    heads x d128 bf16, block 16): entries 0..a_b of every request move from a
    staging buffer into their paged slots.  Four staging sets (> L2) rotate.
    Bytes per launch: sum_b (a_b + 1) x layers x 2 x heads x d x 2 B, read + written."""
    import torch

    from speculative_decoding_verification_07_gb300 import binding
    L, H, D, BS = 32, 8, 128, 16
    B, kmax = 64, 4
    # every request's positions S .. S + k lie in at most 2 blocks: give each its own two
    S = [torch.tensor(s["seq_len"], dtype=torch.int32, device=dev) for s in sets]
    max_blocks = (8192 + 2 * BS) // BS + 2
    tables = []
    for s_dev in S:
        t = torch.full((B, max_blocks), -1, dtype=torch.int32)
        for b, s0 in enumerate(s_dev.cpu().tolist()):
            t[b, s0 // BS] = 2 * b
            t[b, (s0 + kmax) // BS] = 2 * b + 1
        tables.append(t.to(dev))
    kv = torch.zeros(2 * B, L, 2, H, BS, D, dtype=torch.bfloat16, device=dev)
    stages = [torch.randn(B, kmax + 1, L, 2, H, D, device=dev).to(torch.bfloat16) for _ in sets]
    acc = [o["accepted"].clone() for o in outs]
    run = lambda i, st=None: binding.kv_commit_copy(ver.handle, acc[i % len(sets)], S[i % len(sets)],
                                                    tables[i % len(sets)], BS, 2 * B,
                                                    stages[i % len(sets)], kv, stream=st)
    for i in range(8):
        run(i)
    torch.cuda.synchronize()
    n = 64
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        run(i)
    e1.record()
    torch.cuda.synchronize()
    us_eager = e0.elapsed_time(e1) / n * 1e3
    # the launches one by one from Python are bound by the host's call rate:
    # the kernel's own time comes from a graph of the same 64 launches
    try:
        us, launch = graph_us_per_call(run, n, 4, dev), f"CUDA graph of {n} launches, 4 replays"
    except Exception as exc:  # keep the eager figure, say why
        torch.cuda.synchronize()
        us, launch = us_eager, f"eager ({type(exc).__name__}: graph capture failed)"
    assert ver.error() == 0, "device error in the commit-by-copy leg"
    per_tok = L * 2 * H * D * 2
    nbytes = float(np.mean([2 * ((a.cpu().numpy().astype(np.int64) + 1).clip(min=0).sum()) * per_tok
                            for a in acc]))
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": us, "bytes_per_launch": nbytes, "GB/s": gbs, "peak": peak, "frac": gbs / peak,
            "launch": launch, "us_eager_launches": us_eager,
            "shape": "32 layers x 8 KV heads x d128 bf16, block 16, staged entries 0..a_b"}


class _Nvtx:
    """NVTX ranges around the bench's phases, for a profiler's timeline; a
    no-op where this torch build has no NVTX."""

    def __init__(self):
        import torch
        try:
            torch.cuda.nvtx.range_push("probe")
            torch.cuda.nvtx.range_pop()
            self._n = torch.cuda.nvtx
        except Exception:
            self._n = None

    def range_push(self, msg):
        if self._n is not None:
            self._n.range_push(msg)

    def range_pop(self):
        if self._n is not None:
            self._n.range_pop()


def tree_run(ver, dev, peak):
    """Token-tree verification at the workload's vocabulary: B = 64 full binary
    trees of depth 3 (14 nodes), V = 128256 bf16, T = 0.8, top-p 0.95.  Bytes
    needed per call: the target row of every node on the walk and the draft
    row of every visited node with children."""
    import torch

    from speculative_decoding_verification_07_gb300 import device_io
    from speculative_decoding_verification_07_gb300 import workloads as W
    inp = W.tree_batch(B=64, V=128256, shape="binary:3")
    d = device_io.tree_to_device(inp, dev)
    out = ver.tree_outputs(64, inp["parent"].shape[1])
    for _ in range(3):
        ver.verify_tree(**d, out=out)
    torch.cuda.synchronize()
    n = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        ver.verify_tree(**d, out=out)
    e1.record()
    torch.cuda.synchronize()
    assert ver.error() == 0, "device error in the tree run"
    us = e0.elapsed_time(e1) / n * 1e3
    acc = out["accepted"].cpu().numpy()
    pth = out["path"].cpu().numpy()
    V = inp["V"]
    par = inp["parent"]
    nbytes = 0
    for b in range(64):
        visited = [0] + [int(x) for x in pth[b, :acc[b]]]
        for j in visited:
            nbytes += V * 2 + (V * 2 if (par[b] == j).any() else 0)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us": us, "requests_per_s": 64 / (us * 1e-6),
            "tokens_per_s": float((acc + 1).sum()) / (us * 1e-6),
            "mean_accepted": float(acc.mean()), "bytes_needed_per_call": float(nbytes),
            "GB/s": gbs, "peak": peak, "frac": gbs / peak,
            "shape": "64 binary trees of depth 3 (14 nodes), V=128256 bf16, T=0.8, top-p 0.95"}


CONFIG_LEGS = [
    # name, batch recipe, notes
    ("C1", dict(B=1, k=5, V=1024, target_sd=2.0, draft_sd=0.5, temperature=1.0,
                target_dtype="f32", draft_dtype="f32"), "fp32 logits, contiguous KV"),
    ("C2", dict(B=8, k=4, V=32000, target_sd=2.0, draft_sd=0.5, temperature="U[0.5,1.2]"),
     "bf16, T_b ~ U[0.5, 1.2]"),
    ("C3", dict(B=64, k="U{1..8}", V=128256, temperature=0.8, top_p=0.95, draft_kind="probs"),
     "bf16 target, fp32 draft probabilities, ragged k, top-p 0.95"),
    ("M", dict(B=64, k=4, V=128256, temperature=0.8, top_p=0.95), "the metric workload"),
    ("M_stream", dict(B=64, k=4, V=128256, temperature=0.8, top_p=0.95, stream=True),
     "the metric workload on the streaming kernel (SV_FLAG_STREAM_PATH)"),
    ("C4", dict(B=256, k=4, V=151936, temperature="half0"), "half the rows T = 0, half T = 1"),
] + [(f"C5_B{B}_V{V}", dict(B=B, k=8, V=V, temperature=1.0), "sweep point, sigma 1")
     for B in (64, 256, 1024) for V in (32000, 128256, 256000)]


def config_legs(ver, dev, peak, budget_s=90.0):
    """Throughput of spec_verify on every configuration of the benchmark set
    (device-generated inputs, rotated over enough sets to exceed L2): rows/s,
    GB/s of the full and of the needed bytes, and fractions of the measured
    peak and of 8 TB/s.  Per leg: CUDA-event time per call over replays of a
    graph of the calls (`us`), and over the same calls launched one by one from
    Python (`us_eager_calls`, bound by the host's call rate on small batches)."""
    import torch

    from speculative_decoding_verification_07_gb300 import binding
    from speculative_decoding_verification_07_gb300 import device_workloads as DW
    legs = {}
    t_start = time.perf_counter()
    for li, (name, r, note) in enumerate(CONFIG_LEGS):
        if time.perf_counter() - t_start > budget_s:
            legs[name] = {"skipped": "time budget"}
            continue
        B, V = r["B"], r["V"]
        g = torch.Generator(device="cpu")
        g.manual_seed(4000 + li)
        k = r["k"]
        if k == "U{1..8}":
            k = torch.randint(1, 9, (B,), generator=g)
        T = r.get("temperature", 1.0)
        if T == "U[0.5,1.2]":
            T = 0.5 + 0.7 * torch.rand(B, generator=g)
        elif T == "half0":
            T = torch.tensor([0.0 if b % 2 == 0 else 1.0 for b in range(B)])
        dt = {"f32": torch.float32, None: torch.bfloat16}
        kw = dict(target_sd=r.get("target_sd", 3.0), draft_sd=r.get("draft_sd", 1.0),
                  temperature=T, top_p=r.get("top_p", 1.0), draft_kind=r.get("draft_kind", "logits"),
                  target_dtype=dt[r.get("target_dtype")], draft_dtype=dt[r.get("draft_dtype")])
        one = DW.make_batch(B, k, V, device=dev, seed=5000 + 31 * li, **kw)
        per = DW.full_bytes(one)
        n_sets = DW.sets_for(per)
        sets = [one] + [DW.make_batch(B, k, V, device=dev, seed=5000 + 31 * li + s, **kw)
                        for s in range(1, n_sets)]
        kmax = one["kmax"]
        outs = [ver.outputs(B, kmax) for _ in sets]
        use_top_p = r.get("top_p", 1.0) < 1.0
        args = [binding.make_args(target=d["target"], draft=d["draft"], draft_tokens=d["draft_tokens"],
                                  temperature=d["temperature"], k=d["k"],
                                  top_p=d["top_p"] if use_top_p else None, seed=d["seed"],
                                  request_id=d["request_id"], seq_len=d["seq_len"],
                                  draft_kind=d["draft_kind"],
                                  flags=binding.FLAG_STREAM_PATH if r.get("stream") else 0, **o)
                for d, o in zip(sets, outs)]
        wsp = ver.ensure_workspace(max(args, key=lambda a: binding.sv_workspace_size(a)))

        def call(i):
            a = args[i % len(args)]
            binding.spec_verify(ver.handle, a, ver.ensure_workspace(a), None)

        for i in range(max(3, len(sets))):
            call(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call(0)
        e1.record()
        torch.cuda.synchronize()
        est = max(e0.elapsed_time(e1), 1e-3)
        n = int(min(200, max(10, 40.0 / est)))
        e0.record()
        for i in range(n):
            call(i)
        e1.record()
        torch.cuda.synchronize()
        assert ver.error() == 0, f"device error in config leg {name}"
        us_eager = e0.elapsed_time(e1) / n * 1e3
        # small configurations are bound by the host's call rate when launched
        # one by one: time a graph of the same calls (all sets, at least 8)
        n_calls = len(sets) * max(1, -(-8 // len(sets)))
        try:
            us = graph_us_per_call(lambda i, st: binding.spec_verify(ver.handle, args[i % len(args)],
                                                                      wsp, st),
                                   n_calls, max(1, -(-n // n_calls)), dev)
            launch = f"CUDA graph of {n_calls} calls"
        except Exception as exc:  # keep the eager figure, say why
            torch.cuda.synchronize()
            us, launch = us_eager, f"eager ({type(exc).__name__}: graph capture failed)"
        assert ver.error() == 0, f"device error in config leg {name} (graph)"
        rows = float(np.mean([(d["k"].long() + 1).sum().item() for d in sets]))
        bfull = float(np.mean([DW.full_bytes(d) for d in sets]))
        bneed = float(np.mean([DW.needed_bytes(d, o["accepted"]) for d, o in zip(sets, outs)]))
        gfull, gneed = bfull / (us * 1e-6) / 1e9, bneed / (us * 1e-6) / 1e9
        kern = "stream" if r.get("stream") else "cluster"
        legs[name] = {"B": B, "k": "U{1..8}" if r["k"] == "U{1..8}" else r["k"], "V": V,
                      "note": note, "kernel": kern, "us": us, "rows_per_s": rows / (us * 1e-6),
                      "bytes_full": bfull, "bytes_needed": bneed, "GBs_full": gfull,
                      "GBs_needed": gneed, "frac_full": gfull / peak, "frac_of_8tbs": gfull / 8000.0,
                      "l2": f"{len(sets)} input sets of {per / 1e6:.1f} MB rotate",
                      "launches": n, "launch": launch, "us_eager_calls": us_eager}
        del sets, outs, args, one
        torch.cuda.empty_cache()
    return legs


def kernel_source_sha():
    import hashlib
    h = hashlib.sha256()
    for f in ("verify_kernel.cuh", "verify.cu", "verify_bf16.cu", "common.cuh"):
        with open(os.path.join(ROOT, "speculative_decoding_verification_07_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-procs", type=int, default=0,
                    help="host processes of the reference arm (0: one per core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-legs", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
