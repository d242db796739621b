"""The multi-GPU path of the benchmark (replicas): one process per GPU, no data-path collective,
the job timed by its slowest rank and its throughput summed over ranks.  Checked here with two gloo
ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # every rank reports its own time; the job's time is the slowest
    t = bench.max_over_ranks(1.0 + 0.25 * rank, world, torch.device("cpu"))
    rate = bench.whole_job_rate(1000, 10, world, t)
    out[rank] = (t, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_and_summed_rate():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 1.25           # the slowest rank's time
    assert res[0][1] == pytest.approx(1000 * 2 * 10 / 1.25)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_rate(10, 4, 1, 2.0) == 20.0


def test_reference_arm_prints_once_on_rank_zero(capsys):
    """The reference arm (the CPU oracle on samples of the workload) runs and prints on rank 0
    only; the other ranks return without work or output."""
    import argparse
    import json
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(steps=1, warmup=1, gpus=2, impl="reference")
    bench.run_reference(args, 1, 2)
    assert capsys.readouterr().out == ""
    bench.run_reference(args, 0, 2)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    from speculative_decoding_verification_token_gb300 import synth
    assert line["config"] == bench.token_config(synth.TOKEN_LARGE, 2)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
