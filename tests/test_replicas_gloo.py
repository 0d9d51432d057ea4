"""The replica path of bench.py (--gpus N, one process per GPU): every rank
times its own independent replica, the job's time is the slowest rank's and
its throughput is all ranks' bytes over that time.  The rank reduction is
checked with two gloo ranks on the CPU; the per-rank inputs and the one-copy
input staging on the host."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from paged_kv_decode_varlen_gb300 import workloads as W


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's step and end-to-end times: the job takes the slowest of each
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], torch.device("cpu"))
        queue.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == {0: [2.0, 10.0], 1: [2.0, 10.0]}


def test_single_process_needs_no_group():
    assert bench.max_over_ranks([3.5, 4.5], torch.device("cpu")) == [3.5, 4.5]


def test_whole_job_throughput():
    # 1 GB per rank, 2 ranks, 1 s for the slowest rank -> 2 GB/s
    assert bench.whole_job_gbs(1e9, 2, 1000.0) == pytest.approx(2.0)
    assert bench.whole_job_gbs(5e8, 1, 0.5) == pytest.approx(1000.0)


def test_replicas_get_their_own_batches():
    a = W.workload_batch("tiny", seed_offset=0)
    b = W.workload_batch("tiny", seed_offset=1)
    assert a.q.shape == b.q.shape and np.array_equal(a.seq_lens, b.seq_lens)
    assert not np.array_equal(a.q, b.q)            # independent data per rank
    assert W.step_bytes(a)["unique"] == W.step_bytes(b)["unique"]   # the same work per rank (weak scaling)


def test_input_staging_layout_round_trips():
    t = {"q": torch.randn(3, 5).to(torch.bfloat16), "slots": torch.arange(7, dtype=torch.int64),
         "lens": torch.tensor([1, 2, 3], dtype=torch.int32)}
    layout, n = bench.stage_layout(t)
    offs = [o for o, _, _ in layout.values()]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    assert n >= offs[-1] + 3 * 4
    buf = torch.zeros(n, dtype=torch.uint8)
    views = bench.stage_views(buf, layout)
    for k, v in t.items():
        views[k].copy_(v)
    again = bench.stage_views(buf.clone(), layout)
    for k, v in t.items():
        assert again[k].dtype == v.dtype and torch.equal(again[k], v)
