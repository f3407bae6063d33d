"""The N > 1 path of bench.py on the CPU: two gloo ranks (spawned processes).

The codec shards by micro-batch (each rank its own tokens, no collective on
the data path); the process group carries only the barrier and the
max-over-ranks timing, and rank 0 alone reports.  These tests run that host
logic with world size 2 on the gloo backend.
"""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        import torch.distributed as dist
        import bench
        from pipeline_activation_compression_gb300 import synth
        ws_, rank_ = bench.dist_setup(backend="gloo")
        # each rank "measures" a different time; every rank must see the max
        t_max = bench.max_over_ranks(10.0 * (rank_ + 1), ws_)
        bench.barrier(ws_)
        b = synth.make_boundary("tiny_d64_r16", seed=bench.rank_seed(rank_), n_tokens=64)
        q.put((rank_, ws_, t_max, b["tids"].tolist(), float(np.asarray(b["X"]).sum())))
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put(("error", rank, repr(e)))


def _run(ws=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    errs = [o for o in out if o[0] == "error"]
    assert not errs, errs
    return sorted(out)


def test_two_rank_max_and_sharding():
    out = _run(2)
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    # max over ranks: both see the slower rank's time
    assert all(o[2] == 20.0 for o in out)
    # each rank works on its own tokens (weak scaling, no duplicated work)
    assert out[0][3] != out[1][3] and out[0][4] != out[1][4]


def test_whole_job_rate():
    import bench
    # two ranks of 32768 tokens x 10 steps in 5 ms (the slower rank's time)
    assert bench.whole_job_rate(32768 * 10, 2, 5.0) == pytest.approx(2 * 327680 / 5e-3)
    assert bench.whole_job_rate(100, 1, 1.0) == pytest.approx(1e5)


def test_reference_arm_only_rank0_reports():
    import argparse
    import bench
    args = argparse.Namespace(workload="vq_d1024_r128", steps=1, warmup=0)
    assert bench.run_reference(args, 2, 1) is None
