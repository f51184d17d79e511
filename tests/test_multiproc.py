"""Replica plumbing of bench.py across processes (gloo, world size 2, CPU only).

The staged path shards over requests with no data exchange, so several GPUs run independent
replicas; the only cross-rank operations are a barrier and the max of the timed durations.
`--gpus N` launches the ranks itself, and each rank places its threads and pinned host KV on
its GPU's NUMA node (sysfs read here from a fake tree).
"""
import json
import os
import socket
import subprocess
import sys

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
        args = bench.parse_args(["--impl", "reference", "--alias", "1", "--threads", "1", "--warmup", "0",
                                 "--steps", "1"])
        ref = bench.run_reference(args, d) if rank == 1 else "skipped"
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


def test_committed_traffic_lines_match_the_kernels():
    """Every ncu traffic line committed under profiles/ names sources that still hash as recorded,
    so the bench line carries the measured DRAM traffic of the kernels as they stand (a kernel
    changed after its capture needs a new capture, or its line is stale and this fails)."""
    import bench
    lines = 0
    for name in sorted(os.listdir(os.path.join(bench.ROOT, "profiles"))):
        text = open(os.path.join(bench.ROOT, "profiles", name)).read()
        if "bench: traffic_bytes_per_launch=" in text:
            lines += 1
            assert bench.profiled_traffic(name) is not None, name
    assert lines >= 2  # the attention and the staging kernels


def test_gpus_flag_launches_the_ranks():
    """`bench.py --gpus 2` with no torchrun environment starts two ranks (torchrun, 127.0.0.1); they
    join one process group and rank 0 alone prints the line (the reference arm on the CPU)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0", "--batch", "2", "--layers", "1", "--alias", "1",
                        "--threads", "2", "--oracle-requests", "1"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_numa_placement_from_sysfs(tmp_path):
    import bench
    dev = tmp_path / "bus" / "pci" / "devices" / "0009:01:00.0"
    dev.mkdir(parents=True)
    (dev / "numa_node").write_text("1\n")
    assert bench.pci_numa_node(9, 1, 0, str(tmp_path)) == 1
    assert bench.pci_numa_node(9, 2, 0, str(tmp_path)) == -1
    allowed = sorted(os.sched_getaffinity(0))
    node = tmp_path / "devices" / "system" / "node" / "node1"
    node.mkdir(parents=True)
    (node / "cpulist").write_text(",".join(str(c) for c in allowed) + "\n")
    (tmp_path / "devices" / "system" / "node" / "node2").mkdir()
    (tmp_path / "devices" / "system" / "node" / "node2" / "cpulist").write_text("0-3,8,10-11\n")
    assert bench.node_cpus(2, str(tmp_path)) == {0, 1, 2, 3, 8, 10, 11}

    class FakeLibc:
        def __init__(self):
            self.calls = []

        def syscall(self, nr, mode, mask, maxnode):
            self.calls.append((nr, mode, [mask[i] for i in range(16)], maxnode.value))
            return 0

    libc = FakeLibc()
    done = bench.place_on_node(1, str(tmp_path), libc=libc)
    assert done["numa_node"] == 1 and done["cpus"] == len(allowed)
    assert sorted(os.sched_getaffinity(0)) == allowed
    if libc.calls:  # x86_64 or aarch64: set_mempolicy(MPOL_PREFERRED, {node 1})
        nr, mode, mask, maxnode = libc.calls[0]
        assert mode == 1 and mask[0] == 2 and not any(mask[1:]) and maxnode == 1024
        assert done["memory"] == "preferred"
    assert bench.place_on_node(-1, str(tmp_path), libc=libc) == {"numa_node": None}
