"""bench.py's multi-rank path on the CPU: world size 2 over gloo (replicas, no data exchange).

Each rank runs its own replica; the job's step time is the max over ranks and the reported
value aggregates all ranks' bytes.  Only rank 0 prints; the oracle's reference arm runs on
rank 0 alone.
"""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist_env()
        assert (ws, r, local) == (world, rank, rank)
        # rank r measured (step, attention) = (1 + r, 10 - r) ms: the job takes the slowest
        step_ms, attn_ms = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
        out.put((rank, step_ms, attn_ms, bench.whole_job_gbs(ws, 1_000_000, step_ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_take_the_max_over_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(out.get() for _ in range(2))
    for rank, step_ms, attn_ms, gbs in got:
        assert step_ms == 2.0 and attn_ms == 10.0
        assert gbs == pytest.approx(2 * 1_000_000 / 2e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(config="tiny", steps=3, warmup=3, impl="reference")
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_single_process_keeps_its_own_timings():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.25]) == [3.5, 1.25]
    assert bench.whole_job_gbs(1, 2_000_000_000, 1000.0) == pytest.approx(2.0)


def test_both_arms_describe_the_same_config(monkeypatch, capsys):
    """The reference arm prints the config dict the GPU arm builds from the same arguments
    (config_dict(workload, args)): the workload and the timing protocol, nothing arm-specific."""
    sys.path.insert(0, ROOT)
    import json

    import bench
    from paged_kv_decode_slot_gb300 import inputs as gen
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--config", "tiny", "--steps", "1",
                                          "--warmup", "3"]))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    ours = bench.config_dict(gen.make_config("tiny"), bench.parse_args(["--config", "tiny"]))
    assert line["config"] == ours
