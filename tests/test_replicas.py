"""bench.py's host logic on CPU.  The N>1 path: replicas over gloo, world
size 2.  Each rank runs its own sequences; the step time is the max over
ranks and the whole-job throughput counts every rank's tokens (no data-path
collective).  And the reference arm's JSON line."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    ms_local = [120.0, 150.0][rank]
    ms, value = bench.reduce_over_ranks(ms_local, tokens_per_step=1000, world=world)
    # weak scaling: each rank draws its own sequences from its own seed
    seqs = synth.rollout_sequences(synth.TINY, prompts=2, responses=2, seed=1 + rank)
    first = torch.tensor([int(seqs[0].tokens[0])], dtype=torch.int64)
    gathered = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(gathered, first)
    out[rank] = (ms, value, [int(g.item()) for g in gathered])
    dist.destroy_process_group()


def test_two_rank_replicas_max_time_and_whole_job_value():
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    for r in range(2):
        ms, value, firsts = out[r]
        assert ms == 150.0
        assert value == pytest.approx(2 * 1000 / 0.150)
        assert firsts[0] != firsts[1]          # different sequences per rank


def test_reference_arm_line(monkeypatch, capsys):
    """The reference arm (the CPU oracle on the host's cores) prints one JSON
    line with the contract's keys; rank 0 alone runs it."""
    import json
    import types
    import bench
    calls = []

    def fake_sample(layers):
        calls.append(layers)
        return 96 / 2.0, 2.0, 96
    monkeypatch.setattr(bench, "oracle_sample", fake_sample)
    args = types.SimpleNamespace(gpus=1, steps=2, warmup=3, layers=28)
    bench.run_reference(args, rank=1)
    assert calls == [] and capsys.readouterr().out == ""
    bench.run_reference(args, rank=0)
    assert calls == [28] * 5
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] == 48.0 and line["unit"] == bench.UNIT
    assert line["metric"] == bench.METRIC and line["steps"] == 2 and line["warmup"] == 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == 48.0 and cb["cores"] >= 1 and "28-layer" in cb["sample"]
    assert line["e2e"] == {"value": 48.0, "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
