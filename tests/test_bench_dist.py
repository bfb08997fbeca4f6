"""The multi-rank side of bench.py on CPU: two gloo ranks on 127.0.0.1.

Weak scaling: each rank runs its own batch (own seed, same shapes); the only
collective is the max over ranks of the step time, and the job value is the
work of all ranks over that time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import WORKLOADS, make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ws_, r, local = bench._dist()
        slowest = bench.max_over_ranks(times[rank], ws_)
        w = bench.rank_workload(WORKLOADS["tiny"], r)
        first = make_inputs(w)["q"].flatten()[:8].tolist()
        q.put((rank, ws_, local, slowest, bench.job_tflops(2.0e12, slowest, ws_), w.seed, first))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [3.0, 5.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, l0, s0, v0, seed0, q0), (r1, ws1, l1, s1, v1, seed1, q1) = res
    assert (ws0, ws1, l0, l1) == (2, 2, 0, 1)
    assert s0 == s1 == 5.0                      # max over ranks
    assert v0 == v1 == pytest.approx(2 * 2.0e12 / 5e-3 / 1e12)  # both ranks' work
    assert seed1 == seed0 + 1 and q0 != q1      # each rank its own batch


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_tflops(1.0e12, 1.0, 1) == pytest.approx(1000.0)
    w = bench.rank_workload(WORKLOADS["gqa32k"], 0)
    assert (w.L, w.Hq, w.Hkv, w.seed, w.backward) == (32768, 32, 8, WORKLOADS["gqa32k"].seed, True)
