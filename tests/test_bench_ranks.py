"""The benchmark's multi-rank host logic on CPU: two gloo ranks, launched the
way torchrun sets them up (RANK / WORLD_SIZE / LOCAL_RANK / MASTER_* on
127.0.0.1).  Each replica's time is reduced to the slowest rank's, the
whole-job rate counts every replica's steps, and only rank 0 of the reference
arm does any work."""
import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench

TIMEOUT_S = 120


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import datetime

    import torch.distributed as dist
    import bench as b
    dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=60))
    try:
        w, r, local = b.dist_setup()
        slowest = b.max_over_ranks(1.0 + 0.5 * r, w)      # rank 1 takes 1.5 s
        q.put((r, w, local, slowest, b.replica_value(w, 300, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(TIMEOUT_S)
    alive = [p for p in procs if p.is_alive()]
    for p in alive:
        p.kill()
    assert not alive, "a rank did not finish"
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get() for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for rank, world, local, slowest, value in got:
        assert world == 2 and local == rank
        assert slowest == 1.5                  # every rank sees the slowest time
        assert value == pytest.approx(2 * 300 / 1.5)


def test_single_rank_is_its_own_maximum():
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.replica_value(1, 10, 0.5) == 20.0


def test_reference_arm_other_ranks_do_nothing(capsys):
    args = argparse.Namespace(steps=3, warmup=3, gpus=2, impl="reference")
    assert bench.run_reference(args, world=2, rank=1, local=1) is None
    assert capsys.readouterr().out == ""


def test_stored_traffic_only_for_the_captured_sources(monkeypatch):
    """The committed DRAM figure is reported while the pass's sources hash to
    the value recorded with it, and withheld (None) once they differ."""
    import json
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    entry = rec["e2b_pass_step"]
    assert entry["dram_bytes_per_unit"] == entry["dram_bytes_read"] + entry["dram_bytes_write"]
    if entry["source_hash"] == bench.source_hash():          # captured on the current sources
        assert bench.stored_traffic("e2b_pass_step") == entry["dram_bytes_per_unit"]
    else:                                                     # the kernel changed since the capture
        assert bench.stored_traffic("e2b_pass_step") is None
    monkeypatch.setattr(bench, "source_hash", lambda names=bench.PASS_SOURCES: entry["source_hash"])
    assert bench.stored_traffic("e2b_pass_step") == entry["dram_bytes_per_unit"]
    monkeypatch.setattr(bench, "source_hash", lambda names=bench.PASS_SOURCES: "f" * 16)   # a changed kernel
    assert bench.stored_traffic("e2b_pass_step") is None
    assert bench.stored_traffic("no_such_kernel") is None
