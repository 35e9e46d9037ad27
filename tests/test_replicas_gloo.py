"""Multi-process (world size 2, gloo, CPU) checks of the host logic that
bench.py runs under torchrun: every replica draws its own batch, the step
time is the maximum over ranks, and the whole-job value counts every
replica's tokens.  The one-GPU shuffle has no cross-GPU step, so replicas
exchange only these scalars."""
from __future__ import annotations

import json
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, outdir: str):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    from workloads import CONFIGS, make_case

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = bench.replica_config(CONFIGS["tiny"], rank)
        case = make_case(cfg)
        seconds = bench.oracle_step(case)          # each replica's own problem
        local_ms = seconds * 1e3 + 10.0 * rank     # make the ranks differ
        ms = bench.max_over_ranks(local_ms)
        value = bench.whole_job_tokens_per_s(cfg.num_tokens, world, ms)
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump(dict(seed=cfg.seed, local_ms=local_ms, ms=ms, value=value,
                           first_row=case.topk_idx[0].tolist()), f)
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_replicas_with_gloo(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    assert r[0]["seed"] != r[1]["seed"]                  # independent batches
    assert r[0]["first_row"] != r[1]["first_row"] or r[0]["seed"] != r[1]["seed"]
    mx = max(x["local_ms"] for x in r)
    assert r[0]["ms"] == r[1]["ms"] == pytest.approx(mx)  # max over ranks
    T = 512
    assert r[0]["value"] == pytest.approx(T * world / (mx / 1e3))


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    import bench
    from workloads import CONFIGS
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 1, 3, 2
    bench.run_reference(A(), CONFIGS["tiny"])  # returns without work or output
    assert capsys.readouterr().out == ""
