"""Multi-rank host logic of bench.py on CPU: two gloo ranks, 127.0.0.1 rendezvous.

The path shards with no collective (independent sequences and heads): each rank runs
its own batch, the job time is the slowest rank's, and the job rate counts every
rank's tokens.  This checks that aggregation without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    ws, r, _ = bench.dist_setup("gloo")
    seconds = 0.5 + 0.25 * r                      # rank 1 is the slower one
    t = bench.max_over_ranks(seconds, ws, device="cpu")
    rate = bench.job_rate(4096, t, ws)
    bench.barrier(ws, cuda=False)
    queue.put((r, ws, t, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    out = sorted(queue.get(timeout=5) for _ in range(2))
    for r, ws, t, rate in out:
        assert ws == 2
        assert t == pytest.approx(0.75)
        assert rate == pytest.approx(2 * 4096 / 0.75)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_rate(100, 2.0, 1) == 50.0


def test_measured_traffic_is_dropped_when_the_kernel_source_changes(tmp_path, monkeypatch):
    # the roofline's traffic comes from a committed ncu summary only while the profiled
    # source is unchanged
    import bench
    prof = tmp_path / "profiles"
    src = tmp_path / "gated_deltanet_mixer_delta_gb300" / "csrc"
    prof.mkdir()
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    import hashlib
    h = hashlib.sha256(b"kernel v1\n").hexdigest()
    (prof / "k.md").write_text(f"summary\n\ntraffic_bytes_per_call 12345\nsource_sha256 {h}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("k.md", "k.cu") == 12345
    (src / "k.cu").write_text("kernel v2\n")
    assert bench.measured_traffic("k.md", "k.cu") is None
    assert bench.measured_traffic("missing.md", "k.cu") is None
