"""The multi-GPU path's host logic, as two gloo ranks on the CPU.

Several GPUs run independent replicas of the step (attention heads and
sequences need no exchange): each rank seeds its own inputs, the ranks meet
at barriers around the timed region and take the maximum of their times, and
rank 0 alone reports.  These tests run exactly that logic (the module the
benchmark uses) in a world of two processes over gloo, with no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mass_adaptive_sparse_gb300 import replicas, synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = replicas.rank_env()
        ranks = replicas.Ranks(dist, torch.device("cpu"))
        ranks.barrier()
        # each rank's own time; every rank must see the largest
        t_max = ranks.max(10.0 + 5.0 * rank)
        # each rank's own inputs
        cfg = synthetic.CONFIGS["tiny_fp32"]
        x = synthetic.prefill_inputs(cfg, L=64, seed=replicas.replica_seed(cfg.seed, r))
        digest = float(x["q"].double().sum())
        ranks.barrier()
        res = {"rank": r, "world": w, "local": local, "max": t_max, "reports": ranks.reports,
               "digest": digest, "group_rank": ranks.rank, "group_world": ranks.world}
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert (x["rank"], x["world"], x["local"]) == (r, world, r)
        assert (x["group_rank"], x["group_world"]) == (r, world)
        assert x["max"] == 15.0
        assert x["reports"] == (r == 0)
    # rank 0 draws the single-process inputs; the other rank draws its own
    cfg = synthetic.CONFIGS["tiny_fp32"]
    alone = float(synthetic.prefill_inputs(cfg, L=64, seed=cfg.seed)["q"].double().sum())
    assert res[0]["digest"] == alone
    assert res[1]["digest"] != res[0]["digest"]


def test_single_process_defaults(monkeypatch):
    for n in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(n, raising=False)
    assert replicas.rank_env() == (0, 1, 0)
    ranks = replicas.Ranks()
    calls = []
    ranks.sync = lambda: calls.append(1)
    ranks.barrier()
    assert calls == [1]
    assert ranks.max(3.5) == 3.5 and ranks.reports
    assert replicas.replica_seed(7, 0) == 7 and replicas.replica_seed(7, 3) == 10


def test_reference_arm_other_ranks_exit_without_work():
    """bench.py --impl reference on rank 1 of 2: exits 0, prints nothing, runs no oracle."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
