"""Multi-rank host logic of the benchmark (gloo, world size 2, CPU): the
max-over-ranks timing, the whole-job value, each rank's own batch, and the
reference arm printing only on rank 0. The data path itself has no
collective: (segment, head) units are independent, so ranks shard the job by
batches."""
import argparse
import io
import os
import socket
import contextlib

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank
        m = bench.reduce_max(local_ms, torch.device("cpu"))
        results[rank] = (m, bench.job_tflops(1e12, world, m))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        got = dict(results)
    assert got[0][0] == got[1][0] == 15.0
    assert got[0][1] == pytest.approx(2e12 / 15e-3 / 1e12)


def test_reduce_max_without_process_group_is_identity():
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    assert bench.job_tflops(2e12, 1, 1000.0) == pytest.approx(2.0)


def test_reference_arm_is_silent_off_rank_zero():
    args = argparse.Namespace(config=1, steps=1, warmup=3, ref_rows=4)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank=1, world=2)
    assert buf.getvalue() == ""


def test_each_rank_processes_its_own_batch():
    from vision_encoder_varlen_gb300 import workloads as wl
    w = wl.make_config(1)
    a, b = bench.rank_inputs(w, 0), bench.rank_inputs(w, 1)
    assert a["q"].shape == b["q"].shape
    assert not torch.equal(a["q"], b["q"]) and not torch.equal(a["v"], b["v"])
    assert torch.equal(bench.rank_inputs(w, 1)["k"], b["k"])          # seeded: the same every run
