"""The replica bookkeeping of runs over several GPUs, as two gloo ranks on CPU.

Each rank owns its own requests; the only cross-rank steps are distinct request
ids (distinct Philox streams) and the whole-job rate (units of all ranks over
the slowest rank's time).  A rank's oracle walk with its own ids must also
differ from the other rank's, showing that the replicas do not draw the same
random numbers.
"""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_07_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = 10.0 * (rank + 1)             # rank 1 is the slower one
        units = 100.0 * (rank + 1)
        rate, ms_max = replicas.whole_job_rate(ms, units)
        ids = replicas.rank_request_ids(torch.arange(4, dtype=torch.int64), rank)
        gathered = [torch.zeros(4, dtype=torch.int64) for _ in range(ws)]
        dist.all_gather(gathered, ids)
        q.put((rank, rate, ms_max, [g.tolist() for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_rate_and_ids():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, ms_max, ids in res:
        assert ms_max == 20.0                          # the slowest rank's time
        assert rate == (100.0 + 200.0) / 0.020         # all units over that time
        flat = sum(ids, [])
        assert len(set(flat)) == len(flat)             # no id shared between ranks


def test_single_rank_is_identity():
    rate, ms = replicas.whole_job_rate(4.0, 10.0)
    assert ms == 4.0 and rate == 10.0 / 0.004


def test_rank_ids_give_distinct_walks():
    from oracle import sampling as S
    from speculative_decoding_verification_07_gb300 import workloads as W
    inp = W.tiny(V=64, k=3, B=32, T=1.0)
    ref = S.verify_batch(inp)
    other = dict(inp)
    other["request_id"] = replicas.rank_request_ids(torch.from_numpy(
        inp["request_id"].astype(np.int64)), 1).numpy().astype(np.uint32)
    out = S.verify_batch(other)
    assert (ref["out_tokens"] != out["out_tokens"]).any()
