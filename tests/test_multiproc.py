"""Replica plumbing of bench.py across processes (gloo, world size 2, CPU only).

The staged path shards over requests with no data exchange, so several GPUs run independent
replicas; the only cross-rank operations are a barrier and the max of the timed durations.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist(want_gpu=False)
    try:
        d.barrier()
        mx = d.max(1.5 + rank)
        ref = bench.run_reference(type("A", (), {"alias": 1, "threads": 1, "warmup": 0, "steps": 1})(), d) \
            if rank == 1 else "skipped"
        q.put((rank, mx, ref))
    finally:
        d.close()


def test_two_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [2.5, 2.5]   # every rank sees the slowest rank's time
    assert got[1][2] is None                   # the reference arm runs on rank 0 only


def test_ranks_share_the_host():
    """Under torchrun the ranks on one host split its pinned KV buffers and its cores."""
    import bench
    assert bench.rank_host_share(16, 0, 1) == (16, 0)
    assert bench.rank_host_share(16, 0, 2)[0] == 8
    assert bench.rank_host_share(16, 0, 8)[0] == 2
    assert bench.rank_host_share(16, 0, 16)[0] == 2
    assert bench.rank_host_share(16, 3, 4) == (4, 3)
    assert bench.rank_host_share(16, 0, 4)[1] >= 1


def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    """bench.py reports an ncu traffic figure only while the sources it names still hash as
    recorded (a changed kernel makes the figure null)."""
    import hashlib
    import bench
    (tmp_path / "profiles").mkdir()
    srcs = ["a.cu", "b.h"]
    for n, text in zip(srcs, ("kernel v1\n", "header\n")):
        (tmp_path / n).write_text(text)
    h = hashlib.sha256()
    for n in srcs:
        h.update((tmp_path / n).read_bytes())
    (tmp_path / "profiles" / "k.md").write_text(
        f"notes\n    bench: traffic_bytes_per_launch=12345 source={','.join(srcs)} sha256_16={h.hexdigest()[:16]}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md") == 12345
    (tmp_path / "b.h").write_text("header, changed\n")
    assert bench.profiled_traffic("k.md") is None
    assert bench.profiled_traffic("missing.md") is None
