"""The bench's reference arm (the fp64 oracle on the host cores) and its byte
accounting, on the CPU: the JSON line it prints keeps the contract, other
ranks of a multi-process launch exit without work, and the bench's byte
counts agree with the throughput-input module's."""

import json
import os
import subprocess
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_verification_07_gb300 import device_workloads as DW  # noqa: E402


def _run(args, env_extra=None, timeout=600):
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_line():
    r = _run(["--impl", "reference", "--steps", "2", "--warmup", "1", "--ref-procs", "2"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "rows/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["warmup"] == 1 and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "verify_b64_k4"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
             {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_bench_and_device_byte_counts_agree():
    rng = np.random.default_rng(4)
    V = 97
    k = rng.integers(0, 9, size=12)
    kmax = int(k.max())
    inp = {"target": np.zeros((12, kmax + 1, V), np.uint16), "k": k}
    tb = {"target": torch.zeros(12, kmax + 1, V, dtype=torch.bfloat16),
          "draft": torch.zeros(12, max(kmax, 1), V, dtype=torch.bfloat16),
          "k": torch.tensor(k, dtype=torch.int32)}
    assert bench.full_bytes(inp) == DW.full_bytes(tb)
    acc = np.minimum(rng.integers(-1, 9, size=12), k)
    assert bench.needed_bytes(inp, acc) == DW.needed_bytes(tb, torch.tensor(acc))
