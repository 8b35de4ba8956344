"""The multi-rank host logic of bench.py on two gloo ranks on the CPU: under
torchrun every rank runs the whole workload (replicas, weak scaling), the
job's step time is the slowest rank's, and rank 0's line counts every rank's
tokens; the reference arm runs on rank 0 only."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    import ssd_inputs as si
    cfg = si.CONFIGS["mamba2_2p7b"]
    ms = 0.25 + 0.1 * rank            # the last rank is the slowest
    slowest = bench.max_over_ranks(ms, world)
    line = bench.bench_line(cfg, world, 5, 3, slowest, {"gpu_launches": 5})
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "line": line}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_slowest_time_and_whole_job_tokens(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert res[0]["slowest"] == res[1]["slowest"] == pytest.approx(0.35)
    sys.path.insert(0, ROOT)
    import ssd_inputs as si
    cfg = si.CONFIGS["mamba2_2p7b"]
    line = res[0]["line"]
    assert line["n_gpus"] == world and line["scaling"] == "weak"
    assert line["ms_per_step"] == pytest.approx(0.35)
    assert line["value"] == pytest.approx(cfg.tokens * world / 0.35e-3)
    assert line["config"]["global_batch"] == cfg.batch * world
    assert line["config"]["parallelism"] == "replicas x2"
    assert line["gpu_launches"] == 5


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    import ssd_inputs as si
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(argparse.Namespace(gpus=2, steps=1, warmup=0), si.CONFIGS["tiny"])
    assert capsys.readouterr().out == ""   # ranks other than 0 exit without work
