#!/usr/bin/env python3
"""Benchmark of the lookahead sparse KV staging + sparse decode attention path on GB300.

Metric: sparse-decode tok/s at Qwen3-8B attention shapes (36 layers, 32 query / 8 KV heads,
head_dim 128, bf16), batch 128, 16K context, block 16, 2048-token budget, fetch cap 0.05, with
the HBM and host-link roofline fractions of the kernels that carry it.

One step = one decode step of the whole hot path over all layers: per layer, sparse attention
of the step's query over the resident slot pool, then staging from the draft query (block
scoring against the min/max summaries, per-head top-K, capped diff/evict, host->HBM gather of
the admitted blocks), the staging overlapped with the later layers' attention.
`value` = batch * steps / device time of the timed steps (inputs resident in HBM), the median
of `--repeats` timed regions of exactly `--steps` steps each (`repeats` gives all of them);
`e2e` = the same through the C ABI with the step's queries and drafts copied from pinned host
memory and the step's attention outputs copied back, inside the timed region (the copies of
the neighbouring steps overlap the compute, on their own streams).

Full KV lives in page-locked host memory. The 288 GiB of the full batch do not fit the host,
so requests alias `--alias` distinct host buffers (request r reads buffer r mod alias); every
request still has its own summaries, selections, slot pool and queries, so device work and
host-link traffic per step are those of the full batch.

`--workload gqa32b_32k_b32` runs the 32B-class GQA workload (64 layers, 64/8 heads, 32K,
batch 32) through the same path. The default run also carries a compact fetch-cap sweep
(`capsweep`: the batch-90 sweep workload, a few steps per cap).

`--impl reference` times the CPU oracle (binary64 C, the host cores) on the same workload:
each step is one full decode step (every layer, attention and staging) of a few of the
batch's requests, measured, not extrapolated.
Multi-GPU: `--gpus N` without a torchrun environment launches N ranks itself (torchrun,
127.0.0.1); each rank runs its own replica of the workload (requests shard with no data
exchange), its pinned host KV and threads placed on its GPU's NUMA node; timing is the max over
ranks, `value` sums all ranks' tokens.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import platform
import socket
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-decode tok/s, Qwen3-8B attn 16K b128; % of HBM & host-link roofline"
WORKLOAD = "qwen3_8b_16k_b128"


def log(*a):
    print("[bench]", *a, file=sys.stderr, flush=True)


# per workload: distinct host KV buffers the batch aliases by default (the host's memory), and
# the model the shapes come from
WORKLOAD_DEFAULTS = {
    "qwen3_8b_16k_b128": {"alias": 16, "model": "Qwen3-8B attention"},      # 16 x 2.25 GiB
    "gqa32b_32k_b32": {"alias": 8, "model": "32B-class GQA attention"},     # 8 x 8 GiB
    "qwen3_8b_capsweep_b90": {"alias": 16, "model": "Qwen3-8B attention"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=64)
    p.add_argument("--warmup", type=int, default=4)
    p.add_argument("--repeats", type=int, default=3, help="timed regions of --steps steps; value = their median")
    p.add_argument("--impl", choices=["okv", "reference"], default="okv")
    p.add_argument("--alias", type=int, default=0, help="distinct host KV buffers the batch aliases (0: per workload)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-capsweep", action="store_true", help="leave the compact fetch-cap sweep out of the line")
    p.add_argument("--threads", type=int, default=0)
    p.add_argument("--batch", type=int, default=0, help="override the batch (smaller profiling cases)")
    p.add_argument("--layers", type=int, default=0, help="override the layer count (smaller profiling cases)")
    p.add_argument("--oracle-requests", type=int, default=8,
                   help="requests in each full decode step the CPU oracle times (cpu_baseline and the reference arm)")
    p.add_argument("--report", choices=["bench", "capsweep", "agreement", "dense", "partial", "append"], default="bench",
                   help="capsweep: bytes per step and tok/s per fetch cap (batch-90 sweep workload); "
                        "agreement: draft vs previous-token top-K agreement with the true next query; "
                        "dense: dense decode attention over the full KV in HBM vs the sparse path, same shapes; "
                        "partial: admission-time partial staging traffic, occupancy and tok/s at 24K and 32K; "
                        "append: the mixed-length workload with one appended token per request and layer")
    p.add_argument("--workload", default=None, help="synthetic workload name (default: the metric's)")
    args = p.parse_args(argv)
    name = args.workload or WORKLOAD
    if args.alias <= 0:
        args.alias = WORKLOAD_DEFAULTS.get(name, {"alias": 16})["alias"]
    return args


# ---- replica launch and placement ------------------------------------------------------------

def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def self_launch(argv, n: int) -> int:
    """Run this script as n ranks under torchrun on this node (127.0.0.1), the way a multi-GPU
    run is launched by hand; returns torchrun's exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def pci_numa_node(domain: int, bus: int, device: int, sysfs: str = "/sys") -> int:
    """numa_node of PCI function domain:bus:device.0 in sysfs, or -1 if unknown."""
    try:
        with open(os.path.join(sysfs, "bus", "pci", "devices", f"{domain:04x}:{bus:02x}:{device:02x}.0",
                               "numa_node")) as f:
            return int(f.read().strip())
    except (OSError, ValueError):
        return -1


def gpu_numa_node(device: int, sysfs: str = "/sys") -> int:
    """NUMA node of CUDA device `device`, or -1 if unknown."""
    try:
        import torch
        pr = torch.cuda.get_device_properties(device)
        return pci_numa_node(pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id, sysfs)
    except Exception:
        return -1


def node_cpus(node: int, sysfs: str = "/sys") -> set:
    """CPUs of a NUMA node (its cpulist: "0-71,144-215")."""
    cpus = set()
    try:
        with open(os.path.join(sysfs, "devices", "system", "node", f"node{node}", "cpulist")) as f:
            for part in f.read().strip().split(","):
                if "-" in part:
                    a, b = part.split("-")
                    cpus.update(range(int(a), int(b) + 1))
                elif part:
                    cpus.add(int(part))
    except OSError:
        pass
    return cpus


def place_on_node(node: int, sysfs: str = "/sys", libc=None) -> dict:
    """Run this process's threads on the CPUs of `node` that it may use, and prefer that node's
    memory for its pages, before any host KV buffer is allocated: page-locked buffers are then
    backed by the GPU's own host memory (on Grace-based nodes each GPU's host link ends on its own
    CPU socket). Returns what was done; nothing changes when the node is unknown."""
    if node < 0:
        return {"numa_node": None}
    done = {"numa_node": node}
    allowed = os.sched_getaffinity(0)
    cpus = node_cpus(node, sysfs) & allowed
    if cpus:
        os.sched_setaffinity(0, cpus)
        done["cpus"] = len(cpus)
    nr = {"x86_64": 238, "aarch64": 237}.get(platform.machine())  # set_mempolicy(2)
    if nr is not None and node < 1024:
        try:
            libc = libc or ctypes.CDLL(None, use_errno=True)
            mpol_preferred = 1
            mask = (ctypes.c_ulong * 16)()
            mask[node // 64] = 1 << (node % 64)
            if libc.syscall(nr, mpol_preferred, mask, ctypes.c_ulong(16 * 64)) == 0:
                done["memory"] = "preferred"
        except (AttributeError, OSError):
            pass
    return done


# ---- distributed plumbing (replicas: barrier and max-over-ranks only) -------------------------

class Dist:
    def __init__(self, want_gpu: bool):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if want_gpu and torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist
            self.backend = backend

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---- measurement helpers ---------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples (every 100 ms), kept for the windows marked with
    mark_start() / mark_stop() (the timed regions)."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="okv_clocks_", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.windows.append([time.time(), None])

    def mark_stop(self):
        if self.windows and self.windows[-1][1] is None:
            self.windows[-1][1] = time.time()

    @staticmethod
    def _stamp(text: str):
        from datetime import datetime
        try:
            return datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        in_window = [r for r in rows if (t := self._stamp(r[0])) is not None
                     and any(a - 0.05 <= t <= (b or a) + 0.05 for a, b in self.windows)]
        use = in_window or rows  # (if the stamps cannot be read, every sample)
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use),
                "window": "timed regions" if in_window else "whole run"}


def profiled_traffic(profile: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, or None once the kernel's
    sources have changed since the capture: the line names them (comma-separated) with the
    sha256 prefix of their concatenated contents."""
    import hashlib
    import re
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        m = re.search(r"bench: traffic_bytes_per_launch=(\d+) source=(\S+) sha256_16=([0-9a-f]{16})", text)
        if not m:
            return None
        h = hashlib.sha256()
        for path in m.group(2).split(","):
            h.update(open(os.path.join(ROOT, path), "rb").read())
        return int(m.group(1)) if h.hexdigest()[:16] == m.group(3) else None
    except OSError:
        return None


def pinned_h2d_gbs(nbytes=1 << 30, reps=5) -> float:
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    h.fill_(1)
    for _ in range(2):
        d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    best = 1e30
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        b.synchronize()
        best = min(best, a.elapsed_time(b))
    del h, d
    return nbytes / (best / 1e3) / 1e9


class PlainBuffer:
    """Ordinary (pageable) host memory with the .ptr / .free() of a HostBuffer."""

    def __init__(self, nbytes: int):
        import numpy as np
        self.a = np.empty(nbytes + 256, dtype=np.uint8)
        self.ptr = (self.a.ctypes.data + 255) // 256 * 256
        self.nbytes = nbytes

    def free(self):
        self.a = None


# ---- workload setup ----------------------------------------------------------------------------

class Workload:
    def __init__(self, alias: int, threads: int, batch: int = 0, layers: int = 0, name: str | None = None):
        import numpy as np
        import synth
        self.np = np
        self.synth = synth
        self.name = name or WORKLOAD
        self.w = synth.WORKLOADS[self.name]
        if batch:
            self.w = self.w.scaled(batch=batch)
        if layers:
            self.w = self.w.scaled(layers=layers)
        w = self.w
        self.B, self.L, self.Hq, self.Hkv, self.d = w.batch, w.layers, w.q_heads, w.kv_heads, w.head_dim
        self.n_tok = w.context
        self.nb = -(-w.context // w.block_size)
        self.kb = w.budget_tokens // w.block_size
        self.alias = max(1, min(alias, self.B))
        self.ids = np.arange(self.B, dtype=np.int32)
        self.keys = (self.ids % self.alias).astype(np.int32)
        self.threads = threads or os.cpu_count() or 1

    def config(self):
        from sparse_kv_cache_draft_gb300 import BF16, Config
        w = self.w
        return Config(w.layers, w.q_heads, w.kv_heads, w.head_dim, w.block_size, w.budget_tokens, w.batch,
                      self.nb, w.fetch_cap, BF16)

    def host_kv(self, pinned: bool = True, n_buffers: int | None = None):
        """The aliased host KV buffers (the first n_buffers of them), filled by the generator.
        pinned=False gives plain host memory (the CPU oracle needs nothing else)."""
        cfg = self.config()
        n = self.alias if n_buffers is None else min(n_buffers, self.alias)
        t0 = time.time()
        if pinned:
            from sparse_kv_cache_draft_gb300 import HostBuffer
            bufs = [HostBuffer(cfg.host_bytes(self.nb)) for _ in range(n)]
        else:
            bufs = [PlainBuffer(cfg.host_bytes(self.nb)) for _ in range(n)]
        t1 = time.time()
        for k, b in enumerate(bufs):
            self.synth.fill_kv(b.ptr, self.w, k, 0, self.n_tok, self.nb, n_threads=self.threads)
        log(f"host KV: {n} x {cfg.host_bytes(self.nb) / 2**30:.2f} GiB allocated in {t1 - t0:.1f}s, "
            f"generated in {time.time() - t1:.1f}s")
        return bufs

    def step_bytes(self):
        """Algorithmic bytes of one decode step: HBM (summaries and draft rows read by the
        scoring; slots, q and out rows and slot tables of the attention) and, per admitted
        block, the host-link read and the HBM write of its slot."""
        w = self.w
        elem = 2
        summ = self.B * self.Hkv * self.nb * 2 * self.d * elem + self.B * self.Hq * self.d * elem
        attend_fixed = 2 * self.B * self.Hq * self.d * elem + self.B * self.Hkv * self.kb * 4
        return {"score_per_layer": summ, "attend_fixed_per_layer": attend_fixed,
                "slot_bytes": 2 * w.block_size * self.d * elem}

    def queries(self, layer, step, kind, out=None):
        return self.synth.queries(self.w, layer, step, kind, self.ids, self.keys, out=out, n_threads=self.threads)

    def config_json(self):
        w = self.w
        ref = self.synth.WORKLOADS[self.name]
        full = (self.B, self.L) == (ref.batch, ref.layers)
        sb = self.step_bytes()
        working = self.L * (sb["score_per_layer"] + self.B * self.Hkv * self.kb * sb["slot_bytes"])
        return {"workload": self.name if full else f"{self.name} (batch {self.B}, {self.L} layers)",
                "model_shapes": WORKLOAD_DEFAULTS.get(self.name, {}).get("model", "Qwen3-8B attention"),
                "batch": self.B, "seq_len": self.n_tok,
                "layers": self.L, "q_heads": self.Hq, "kv_heads": self.Hkv, "head_dim": self.d,
                "block_size": w.block_size, "budget_tokens": w.budget_tokens, "fetch_cap": w.fetch_cap,
                "host_kv_buffers": self.alias, "parallelism": "replicas",
                "l2": f"no flush: per-step working set ({working / 2**30:.0f} GiB of summaries and slot pool) "
                      ">> 129 MB L2"}


# ---- CPU oracle timing (cpu_baseline leg and the reference arm) -------------------------------

class OracleSample:
    """The oracle as it stands, on the host cores: full decode steps (every layer: attention of
    the step's query over the resident set, then staging from its draft) of the first n requests
    of the workload, after the same bootstrap staging the GPU run makes. Per request the work of
    a step is that of the full batch, so tok/s = n / seconds per step."""

    def __init__(self, wl: "Workload", bufs, n_req: int):
        import oracle
        self.oracle = oracle
        self.wl = wl
        w = wl.w
        self.n = max(1, min(n_req, wl.B))
        self.ids, self.keys = wl.ids[:self.n], wl.keys[:self.n]
        self.model = oracle.OracleModel(layers=w.layers, q_heads=w.q_heads, kv_heads=w.kv_heads,
                                        head_dim=w.head_dim, block_size=w.block_size,
                                        budget_tokens=w.budget_tokens, dtype=w.dtype,
                                        req_ptrs=[bufs[int(k)].ptr for k in self.keys], cap_blocks=[wl.nb] * self.n,
                                        n_tok=wl.n_tok, n_threads=wl.threads)
        self.C = oracle.fetch_cap_blocks(w.fetch_cap, wl.kb)
        t0 = time.time()
        boot = oracle.fetch_cap_blocks(1.0, wl.kb)
        for l in range(w.layers):
            self.model.build_summaries(l)
            self.model.stage(l, self.queries(l, -1, 1), boot, 0)
        self.prepare_s = time.time() - t0

    def queries(self, layer, step, kind):
        return self.wl.synth.queries(self.wl.w, layer, step, kind, self.ids, self.keys, n_threads=self.wl.threads)

    def step(self, t: int, threads: int | None = None) -> float:
        """Seconds of decode step t (inputs generated before the clock starts)."""
        L = self.wl.w.layers
        qs = [(self.queries(l, t, 0), self.queries(l, t, 1)) for l in range(L)]
        keep = self.model.n_threads
        if threads:
            self.model.n_threads = threads
        t0 = time.perf_counter()
        for l in range(L):
            self.model.attend(l, qs[l][0])
            self.model.stage(l, qs[l][1], self.C, t + 1)
        dt = time.perf_counter() - t0
        self.model.n_threads = keep
        return dt


def cpu_baseline(wl: "Workload", bufs, n_req: int, n_steps: int = 2):
    """The oracle's tok/s over n_steps full decode steps of n_req requests on all the threads,
    and over one more step on one thread."""
    t0 = time.time()
    o = OracleSample(wl, bufs, n_req)
    secs = [o.step(t) for t in range(n_steps)]
    one = o.step(n_steps, threads=1)
    per_step = statistics.mean(secs)
    return {"value": round(o.n / per_step, 3), "unit": "tok/s", "cores": wl.threads, "nproc": os.cpu_count(),
            "kind": "oracle",
            "one_thread": {"value": round(o.n / one, 3), "unit": "tok/s", "cores": 1},
            "sample": f"{n_steps} full decode steps (all {wl.L} layers: attention, then staging of the draft) of "
                      f"requests 0..{o.n - 1} of the {wl.B}-request batch, {per_step:.2f} s per step on "
                      f"{wl.threads} threads, measured (bootstrap and summaries {o.prepare_s:.1f} s, untimed); "
                      f"tok/s = requests / seconds per step; one_thread: one more step on 1 thread "
                      f"({one:.2f} s); {time.time() - t0:.1f} s in all"}


# ---- the okv arm -------------------------------------------------------------------------------

def rank_host_share(alias: int, threads: int, world: int) -> tuple[int, int]:
    """Host KV buffers and generator threads of one rank when `world` ranks share a host: each
    rank aliases its share of the buffers (at least 2) and uses its share of the cores. Aliasing
    changes neither the device work nor the host-link bytes of a step."""
    if world <= 1:
        return alias, threads
    return max(2, alias // world), threads or max(1, (os.cpu_count() or 1) // world)


def run_okv(args, dist: Dist):
    import numpy as np
    import torch
    from sparse_kv_cache_draft_gb300 import Context, HostBuffer, load_library

    load_library()
    torch.cuda.set_device(dist.local)
    placement = place_on_node(gpu_numa_node(dist.local))
    alias, threads = rank_host_share(args.alias, args.threads, dist.world)
    wl = Workload(alias, threads, args.batch, args.layers, args.workload)
    cfg = wl.config()
    B, L, Hq, d = wl.B, wl.L, wl.Hq, wl.d
    K, W, NR = args.steps, args.warmup, max(1, args.repeats)
    bufs = wl.host_kv()
    t0 = time.time()
    ctx = Context(cfg)
    for r in range(B):
        ctx.add_request(r, bufs[int(wl.keys[r])].ptr, wl.nb, wl.n_tok)
    log(f"context + {B} requests registered in {time.time() - t0:.1f}s")

    # inputs for the bootstrap, W warm-up steps, NR timed regions of K steps and the e2e steps
    # (pinned host copies for e2e)
    n_steps = W + NR * K
    qshape = (L, B, Hq, d)
    per_step = L * B * Hq * d
    t0 = time.time()
    q_host = HostBuffer(n_steps * per_step * 2)
    d_host = HostBuffer((n_steps + 1) * per_step * 2)
    qh = q_host.numpy(np.uint16, (n_steps,) + qshape)
    dh = d_host.numpy(np.uint16, (n_steps + 1,) + qshape)  # dh[t + 1] = draft of step t
    for t in range(-1, n_steps):
        for l in range(L):
            if t >= 0:
                wl.queries(l, t, 0, out=qh[t, l])
            wl.queries(l, t, 1, out=dh[t + 1, l])
    log(f"inputs for {n_steps} steps generated in {time.time() - t0:.1f}s")

    def as_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)

    q_dev = as_bf16(qh).to("cuda")
    d_dev = as_bf16(dh).to("cuda")
    out = torch.empty(qshape, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(dist.local)
    sampler.start()

    # bootstrap staging from the draft of step -1 at fetch cap 1.0 (fills the empty pools)
    for l in range(L):
        ctx.stage(l, d_dev[0, l], 0, 1.0)
    for t in range(W):
        ctx.step(q_dev[t], d_dev[t + 1], out, t + 1)
    torch.cuda.synchronize()
    assert ctx.sync(60_000) == 0

    # timed regions: NR x K decode steps, inputs resident in HBM; the library's per-launch events
    # (timing) cover all of them
    ctx.set_timing(True)
    launches0 = ctx.launch_count()
    region_ms = []
    for rep in range(NR):
        torch.cuda.synchronize()
        dist.barrier()
        sampler.mark_start()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for t in range(W + rep * K, W + (rep + 1) * K):
            ctx.step(q_dev[t], d_dev[t + 1], out, t + 1)
        ctx.join(stream)
        ev1.record(stream)
        ev1.synchronize()
        sampler.mark_stop()
        dist.barrier()
        region_ms.append(dist.max(ev0.elapsed_time(ev1)))
    launches = (ctx.launch_count() - launches0) / NR
    timing = ctx.read_timing()
    ctx.set_timing(False)
    assert ctx.sync(60_000) == 0
    ms_max = statistics.median(region_ms)

    # e2e: the same steps through the C ABI from pinned host inputs, outputs copied back. The
    # copies overlap the compute as a caller would run them: step i+1's queries and drafts are
    # copied in on one stream and step i's outputs copied out on another while step i computes
    # (double-buffered device tensors, events guarding every reuse).
    out_host = HostBuffer(2 * per_step * 2)
    oh = as_bf16(out_host.numpy(np.uint16, (2,) + qshape))
    q_in = [torch.empty(qshape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    d_in = [torch.empty(qshape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    o_dev = [torch.empty(qshape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_loaded = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_saved = [torch.cuda.Event() for _ in range(2)]
    qh_t, dh_t = as_bf16(qh), as_bf16(dh)

    def load(i):
        b, t = i % 2, W + i
        if i >= 2:
            s_in.wait_event(ev_done[b])  # step i-2 has finished reading this buffer
        with torch.cuda.stream(s_in):
            q_in[b].copy_(qh_t[t], non_blocking=True)
            d_in[b].copy_(dh_t[t + 1], non_blocking=True)
        ev_loaded[b].record(s_in)

    torch.cuda.synchronize()
    dist.barrier()
    sampler.mark_start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    load(0)
    for i in range(K):
        b = i % 2
        if i + 1 < K:
            load(i + 1)
        stream.wait_event(ev_loaded[b])
        if i >= 2:
            stream.wait_event(ev_saved[b])  # step i-2's output has left this buffer
        ctx.step(q_in[b], d_in[b], o_dev[b], W + NR * K + i + 1)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            oh[b].copy_(o_dev[b], non_blocking=True)
        ev_saved[b].record(s_out)
    ctx.join(stream)
    stream.wait_stream(s_out)
    e1.record(stream)
    e1.synchronize()
    sampler.mark_stop()
    e2e_ms = dist.max(e0.elapsed_time(e1))
    assert ctx.sync(60_000) == 0
    clocks = sampler.stop()

    # the same gather with only staging beside it (no attention): a few steps of okv_stage calls
    # after the timed regions, on drafts of earlier steps (so the cap binds); the state they leave
    # is not used again
    ctx.set_timing(True)
    n_alone = min(K, 4)
    for i in range(n_alone):
        for l in range(L):
            ctx.stage(l, d_dev[W + i + 1, l], W + NR * K + K + 1 + i)
    ctx.join(stream)
    torch.cuda.synchronize()
    alone = ctx.read_timing()
    ctx.set_timing(False)
    assert ctx.sync(60_000) == 0
    # the same attention launches with nothing else running: two passes over every layer
    ctx.set_timing(True)
    for _ in range(2):
        for l in range(L):
            ctx.attend(l, q_dev[W, l], out[l])
    torch.cuda.synchronize()
    att_alone = ctx.read_timing()
    ctx.set_timing(False)
    assert ctx.sync(60_000) == 0
    ctx.close()
    del q_dev, d_dev, out, q_in, d_in, o_dev
    torch.cuda.empty_cache()

    # rooflines
    hbm_peak, peak_src = measured_peaks()
    h2d_peak = pinned_h2d_gbs()
    sb = wl.step_bytes()
    slot_bytes = sb["slot_bytes"]
    n_steps_timed = NR * K
    n_att_calls = L * n_steps_timed
    att_ms = timing["ms"]["attend"] / n_att_calls
    att_bytes = (timing["attended_slots"] / n_att_calls) * slot_bytes + sb["attend_fixed_per_layer"]
    att_gbs = att_bytes / (att_ms / 1e3) / 1e9
    sc_ms = timing["ms"]["score_topk"] / n_att_calls
    sc_bytes = sb["score_per_layer"]
    sc_gbs = sc_bytes / (sc_ms / 1e3) / 1e9
    gather_bytes = timing["fetched_blocks"] * slot_bytes
    gather_ms = timing["ms"]["gather"]
    gather_gbs = gather_bytes / (gather_ms / 1e3) / 1e9 if gather_ms > 0 else 0.0
    alone_ms = alone["ms"]["gather"]
    alone_gbs = alone["fetched_blocks"] * slot_bytes / (alone_ms / 1e3) / 1e9 if alone_ms > 0 else 0.0
    sc_alone_ms = alone["ms"]["score_topk"] / (n_alone * L)
    att_alone_ms = att_alone["ms"]["attend"] / (2 * L)
    att_alone_bytes = (att_alone["attended_slots"] / (2 * L)) * slot_bytes + sb["attend_fixed_per_layer"]
    att_alone_gbs = att_alone_bytes / (att_alone_ms / 1e3) / 1e9 if att_alone_ms > 0 else 0.0
    sc_alone_gbs = sc_bytes / (sc_alone_ms / 1e3) / 1e9 if sc_alone_ms > 0 else 0.0
    step_ms = ms_max / K
    link_step_bytes = gather_bytes / n_steps_timed
    # HBM per step: the scoring's and the attention's reads, and the slots the gather writes
    hbm_step_bytes = L * (att_bytes + sc_bytes) + link_step_bytes
    ideal_hbm_ms = hbm_step_bytes / (hbm_peak * 1e9) * 1e3
    ideal_link_ms = link_step_bytes / (h2d_peak * 1e9) * 1e3
    ideal_ms = max(ideal_hbm_ms, ideal_link_ms)

    def tok_s(ms):
        return dist.world * B * K / (ms / 1e3)

    value = tok_s(ms_max)
    e2e_value = tok_s(e2e_ms)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tok/s", "n_gpus": dist.world, "steps": K,
        "warmup": W, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": wl.config_json(),
        "repeats": {"n": NR, "steps_each": K, "median": round(value, 1),
                    "min": round(tok_s(max(region_ms)), 1), "max": round(tok_s(min(region_ms)), 1),
                    "tok_s": [round(tok_s(m), 1) for m in region_ms]},
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 1), "unit": "tok/s", "h2d_bytes_per_step": 2 * per_step * 2,
                "d2h_bytes_per_step": per_step * 2},
        "gpu_launches": int(round(launches)),
        "roofline": {"bound": "hbm", "kernel": "sparse GQA decode attention (okv_attend)",
                     "achieved": round(att_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(att_gbs / hbm_peak, 4),
                     "traffic": profiled_traffic("attend_mma_qwen3_8b_16k.md") if (wl.name, B, L) == (WORKLOAD, 128, 36)
                     else None,
                     "peak_source": f"hbm_gbs, {peak_src}",
                     "bytes_per_launch": int(att_bytes), "ms_per_launch": round(att_ms, 5),
                     "without_staging": {"achieved": round(att_alone_gbs, 1),
                                         "frac": round(att_alone_gbs / hbm_peak, 4),
                                         "ms_per_launch": round(att_alone_ms, 5),
                                         "note": "the same attention launches with nothing else running, two "
                                                 "passes over every layer after the timed regions"}},
        "scoring_roofline": {"bound": "hbm", "kernel": "block scoring + top-K", "achieved": round(sc_gbs, 1),
                             "peak": hbm_peak, "unit": "GB/s", "frac": round(sc_gbs / hbm_peak, 4),
                             "traffic": profiled_traffic("stage_kernel_qwen3_8b_16k.md")
                             if (wl.name, B) == (WORKLOAD, 128) else None,
                             "bytes_per_launch": int(sc_bytes), "ms_per_launch": round(sc_ms, 5),
                             "note": "in the step the kernel runs on a least-priority stream: its event time "
                                     "includes waiting for SMs the attention holds",
                             "without_attention": {"achieved": round(sc_alone_gbs, 1),
                                                   "frac": round(sc_alone_gbs / hbm_peak, 4),
                                                   "ms_per_launch": round(sc_alone_ms, 5)}},
        "host_link": {"kernel": "host->HBM block gather", "achieved": round(gather_gbs, 1),
                      "peak": round(h2d_peak, 1), "unit": "GB/s", "frac": round(gather_gbs / h2d_peak, 4),
                      "peak_source": "pinned cudaMemcpy H2D of 1 GiB measured in this run",
                      "bytes_per_step": int(link_step_bytes),
                      "without_attention": {"achieved": round(alone_gbs, 1), "frac": round(alone_gbs / h2d_peak, 4),
                                            "note": f"the same gather beside staging only, {n_alone} steps of "
                                                    "okv_stage after the timed regions"}},
        "step_roofline": {"hbm_bytes": int(hbm_step_bytes), "hbm_peak_gbs": hbm_peak,
                          "link_bytes": int(link_step_bytes), "link_peak_gbs": round(h2d_peak, 1),
                          "ideal_ms": round(ideal_ms, 4), "bound": "hbm" if ideal_hbm_ms >= ideal_link_ms else "link",
                          "ideal_hbm_ms": round(ideal_hbm_ms, 4), "ideal_link_ms": round(ideal_link_ms, 4),
                          "ms_per_step": round(step_ms, 4), "frac": round(ideal_ms / step_ms, 4),
                          "note": "ideal step = max(HBM bytes / measured HBM peak, host-link bytes / in-run H2D "
                                  "peak); HBM bytes = scoring and attention reads plus the gather's slot writes"},
        "kernel_ms_per_step": {k: round(v / n_steps_timed, 4) for k, v in timing["ms"].items() if v > 0},
        "attention_ms_per_layer": round(att_ms, 5),
        "placement": placement,
    }
    if dist.rank == 0 and not args.no_capsweep and not args.batch and not args.layers and wl.name == WORKLOAD:
        t0 = time.time()
        res["capsweep"] = capsweep_compact(args, dist, threads)
        log(f"cap sweep took {time.time() - t0:.1f}s")
    if not args.no_cpu_baseline and dist.rank == 0 and dist.world == 1:
        t0 = time.time()
        res["cpu_baseline"] = cpu_baseline(wl, bufs, args.oracle_requests)
        log(f"cpu baseline sample took {time.time() - t0:.1f}s")
    for b in bufs:
        b.free()
    return res


def run_reference(args, dist: Dist):
    """The oracle on the host cores: each of the W + K steps is one full decode step of the first
    --oracle-requests requests; the K timed steps give the line (rank 0 only)."""
    if dist.rank != 0:
        return None
    wl = Workload(args.alias, args.threads, args.batch, args.layers, args.workload)
    n = min(args.oracle_requests, wl.B)
    bufs = wl.host_kv(pinned=False, n_buffers=n)
    o = OracleSample(wl, bufs, n)
    for t in range(args.warmup):
        o.step(t)
    secs = [o.step(t) for t in range(args.warmup, args.warmup + args.steps)]
    total = sum(secs)
    value = o.n * args.steps / total
    for b in bufs:
        b.free()
    sample = (f"each step: one full decode step (all {wl.L} layers: attention, then staging of the draft) of "
              f"requests 0..{o.n - 1} of the {wl.B}-request batch, measured (no extrapolation); tok/s = requests x "
              f"steps / seconds; bootstrap and summaries {o.prepare_s:.1f} s, untimed")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wl.config_json(),
            "cpu_baseline": {"value": round(value, 3), "unit": "tok/s", "cores": wl.threads, "nproc": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _setup_context(wl, bufs, cap=None):
    from sparse_kv_cache_draft_gb300 import Context
    cfg = wl.config()
    if cap is not None:
        cfg.fetch_cap = cap
    ctx = Context(cfg)
    for r in range(wl.B):
        ctx.add_request(r, bufs[int(wl.keys[r])].ptr, wl.nb, wl.n_tok)
    return ctx


def _device_inputs(wl, steps):
    """bf16 device tensors q[t] (steps 0..steps-1) and dr[t + 1] = draft of step t (t = -1..steps-1)."""
    import numpy as np
    import torch
    shape = (wl.L, wl.B, wl.Hq, wl.d)
    qh = np.empty((steps,) + shape, np.uint16)
    dh = np.empty((steps + 1,) + shape, np.uint16)
    for t in range(-1, steps):
        for l in range(wl.L):
            if t >= 0:
                wl.queries(l, t, 0, out=qh[t, l])
            wl.queries(l, t, 1, out=dh[t + 1, l])
    conv = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to("cuda")
    return conv(qh), conv(dh)


def _sweep_caps(wl, bufs, K, W, dist):
    """Per fetch cap: a fresh context, the bootstrap staging at cap 1.0, W warm-up and K timed
    decode steps; bytes moved host->HBM per step and tok/s."""
    import torch
    q, dr = _device_inputs(wl, W + K)
    out = torch.empty(q.shape[1:], dtype=torch.bfloat16, device="cuda")
    rows = []
    for cap in wl.w.caps:
        ctx = _setup_context(wl, bufs, cap)
        for l in range(wl.L):
            ctx.stage(l, dr[0, l], 0, 1.0)
        for t in range(W):
            ctx.step(q[t], dr[t + 1], out, t + 1)
        torch.cuda.synchronize()
        ctx.set_timing(True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for t in range(W, W + K):
            ctx.step(q[t], dr[t + 1], out, t + 1)
        ctx.join()
        e1.record()
        e1.synchronize()
        ms = dist.max(e0.elapsed_time(e1))
        tm = ctx.read_timing()
        assert ctx.sync(60_000) == 0
        gb = tm["fetched_blocks"] * 2 * wl.w.block_size * wl.d * 2 / K / 1e9
        rows.append({"fetch_cap": cap, "C_blocks": max(1, int(cap * wl.kb)), "gb_per_step": round(gb, 4),
                     "tok_s": round(dist.world * wl.B * K / (ms / 1e3), 1), "ms_per_step": round(ms / K, 4),
                     "gather_gbs": round(gb * K / (tm["ms"]["gather"] / 1e3), 1) if tm["ms"]["gather"] else None})
        ctx.close()
    del q, dr, out
    torch.cuda.empty_cache()
    return rows


def capsweep_compact(args, dist: Dist, threads: int):
    """The fetch-cap sweep workload (batch 90, 100 directions, 5 active, one replaced per step),
    2 warm-up and 4 timed steps per cap, for the bench line."""
    name = "qwen3_8b_capsweep_b90"
    wl = Workload(8, threads, 0, 0, name)
    bufs = wl.host_kv()
    try:
        rows = _sweep_caps(wl, bufs, 4, 2, dist)
    finally:
        for b in bufs:
            b.free()
    return {"workload": name, "batch": wl.B, "steps_per_cap": 4, "warmup_per_cap": 2, "host_kv_buffers": wl.alias,
            "note": "bytes moved host->HBM per step and decode tok/s per fetch cap (C = floor(cap x 128) blocks "
                    "per KV head per layer and step); the pages' ablation is context, not a target",
            "caps": rows}


def run_capsweep(args, dist: Dist):
    """Fetch-cap sweep: bytes moved host->HBM per step and decode tok/s per cap."""
    name = args.workload or "qwen3_8b_capsweep_b90"
    wl = Workload(args.alias, args.threads, args.batch, args.layers, name)
    bufs = wl.host_kv()
    K, W = args.steps, args.warmup
    rows = _sweep_caps(wl, bufs, K, W, dist)
    for b in bufs:
        b.free()
    return {"report": "capsweep", "metric": "sparse-decode tok/s and host->HBM GB/step per fetch cap",
            "unit": "tok/s", "n_gpus": dist.world, "steps": K, "warmup": W, "data": "synthetic",
            "config": wl.config_json(), "caps": rows}


def run_agreement(args, dist: Dist):
    """Per layer: overlap of the top-K the staging selects from the draft of step t with the top-K of
    the true query of step t+1, against the previous-token proxy (the query of step t)."""
    import numpy as np
    import torch
    wl = Workload(args.alias, args.threads, args.batch, args.layers, args.workload)
    bufs = wl.host_kv()
    K = args.steps
    q, dr = _device_inputs(wl, K + 1)
    ctx = _setup_context(wl, bufs)
    out = torch.empty(q.shape[1:], dtype=torch.bfloat16, device="cuda")
    counts = torch.zeros((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
    ids = torch.zeros((wl.B, wl.Hkv, wl.kb), dtype=torch.int32, device="cuda")

    def overlap(a_cnt, a_ids, b_cnt, b_ids):
        tot = hit = 0
        for r in range(wl.B):
            for h in range(wl.Hkv):
                n = int(a_cnt[r, h])
                hit += len(set(a_ids[r, h, :n].tolist()) & set(b_ids[r, h, :int(b_cnt[r, h])].tolist()))
                tot += n
        return hit / max(tot, 1)

    for l in range(wl.L):
        ctx.stage(l, dr[0, l], 0, 1.0)
    draft_agree = np.zeros((K, wl.L))
    proxy_agree = np.zeros((K, wl.L))
    for t in range(K):
        for l in range(wl.L):
            ctx.attend(l, q[t, l], out[l])
            ctx.stage(l, dr[t + 1, l], t + 1)
            torch.cuda.synchronize()
            d_cnt, d_ids, _ = ctx.read_selection(l)
            ctx.predict(l, q[t + 1, l], counts, ids)
            true_cnt, true_ids = counts.cpu().numpy().copy(), ids.cpu().numpy().copy()
            ctx.predict(l, q[t, l], counts, ids)
            prev_cnt, prev_ids = counts.cpu().numpy(), ids.cpu().numpy()
            draft_agree[t, l] = overlap(d_cnt, d_ids, true_cnt, true_ids)
            proxy_agree[t, l] = overlap(prev_cnt, prev_ids, true_cnt, true_ids)
    ctx.close()
    for b in bufs:
        b.free()
    return {"report": "agreement", "metric": "top-K agreement with the true next query", "unit": "fraction",
            "steps": K, "data": "synthetic", "config": wl.config_json(),
            "draft_mean": round(float(draft_agree.mean()), 4), "draft_min_layer": round(float(draft_agree.mean(0).min()), 4),
            "proxy_mean": round(float(proxy_agree.mean()), 4), "proxy_min_layer": round(float(proxy_agree.mean(0).min()), 4),
            "draft_per_layer": [round(float(x), 4) for x in draft_agree.mean(0)],
            "proxy_per_layer": [round(float(x), 4) for x in proxy_agree.mean(0)]}


def run_dense(args, dist: Dist):
    """Dense decode attention over the full KV held in HBM (the attention kernel over an identity slot
    table of every block) against the sparse path at the same shapes and batch."""
    import numpy as np
    import torch
    from sparse_kv_cache_draft_gb300 import BF16, binding
    wl = Workload(args.alias, args.threads, args.batch or 64, args.layers, args.workload)
    bufs = wl.host_kv()
    K, W = args.steps, args.warmup
    L, B, Hkv, nb, d = wl.L, wl.B, wl.Hkv, wl.nb, wl.d
    bs = wl.w.block_size
    unit_bytes = nb * 2 * bs * d * 2
    kv = torch.empty((L, B, Hkv, nb, 2, bs, d), dtype=torch.bfloat16, device="cuda")
    for k, b in enumerate(bufs):
        host = torch.from_numpy(b.numpy(np.int16, (L, Hkv, nb, 2, bs, d))).view(torch.bfloat16)
        for r in range(B):
            if int(wl.keys[r]) == k:
                for l in range(L):
                    kv[l, r].copy_(host[l])
    sb = torch.arange(nb, dtype=torch.int32, device="cuda").repeat(B, Hkv, 1).contiguous()
    lens = torch.full((B,), wl.n_tok, dtype=torch.int32, device="cuda")
    q, dr = _device_inputs(wl, W + K)
    out = torch.empty(q.shape[1:], dtype=torch.bfloat16, device="cuda")

    def dense_step(t):
        for l in range(L):
            binding.attend_static(kv[l], sb, lens, q[t, l], out[l], q_heads=wl.Hq, kv_heads=Hkv, head_dim=d,
                                  block_size=bs, slots=nb, dtype=BF16)

    for t in range(W):
        dense_step(t)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(W, W + K):
        dense_step(t)
    e1.record()
    e1.synchronize()
    dense_ms = dist.max(e0.elapsed_time(e1))
    del kv
    torch.cuda.empty_cache()
    # the sparse path at the same batch
    ctx = _setup_context(wl, bufs)
    for l in range(L):
        ctx.stage(l, dr[0, l], 0, 1.0)
    for t in range(W):
        ctx.step(q[t], dr[t + 1], out, t + 1)
    torch.cuda.synchronize()
    e0.record()
    for t in range(W, W + K):
        ctx.step(q[t], dr[t + 1], out, t + 1)
    ctx.join()
    e1.record()
    e1.synchronize()
    sparse_ms = dist.max(e0.elapsed_time(e1))
    ctx.close()
    for b in bufs:
        b.free()
    dense_tok = dist.world * B * K / (dense_ms / 1e3)
    sparse_tok = dist.world * B * K / (sparse_ms / 1e3)
    hbm_peak, src = measured_peaks()
    dense_bytes = L * B * Hkv * unit_bytes
    return {"report": "dense", "metric": "decode attention tok/s, dense (full KV in HBM) vs sparse staging",
            "unit": "tok/s", "n_gpus": dist.world, "steps": K, "warmup": W, "data": "synthetic",
            "config": wl.config_json(), "dense_tok_s": round(dense_tok, 1), "sparse_tok_s": round(sparse_tok, 1),
            "sparse_over_dense": round(sparse_tok / dense_tok, 3),
            "dense_ms_per_step": round(dense_ms / K, 3), "sparse_ms_per_step": round(sparse_ms / K, 3),
            "dense_hbm_gbs": round(dense_bytes / (dense_ms / K / 1e3) / 1e9, 1),
            "dense_hbm_frac": round(dense_bytes / (dense_ms / K / 1e3) / 1e9 / hbm_peak, 4),
            "peak_source": f"hbm_gbs, {src}"}


def run_partial(args, dist: Dist):
    """Admission-time partial staging: bytes that cross from the full copy (the prefill side's
    host memory) to the decode side at admission and during decoding, the decode side's host
    occupancy, and decode tok/s against the same steps on requests that hold their full KV."""
    import torch
    from sparse_kv_cache_draft_gb300 import Context, HostBuffer
    names = [args.workload] if args.workload else ["qwen3_8b_pd_24k_b8", "qwen3_8b_pd_32k_b8"]
    S = args.steps
    marks = sorted({m for m in (16, 64, 256) if m < S} | {S})
    results = []
    for name in names:
        # the full copies are only read: a few buffers stand for the batch's prefill-side memory
        wl = Workload(min(args.alias, 4), args.threads, args.batch, args.layers, name)
        bufs = wl.host_kv()
        L, B, Hkv, nb, kb, d, bs = wl.L, wl.B, wl.Hkv, wl.nb, wl.kb, wl.d, wl.w.block_size
        block_bytes = 2 * bs * d * 2
        full_bytes = L * Hkv * nb * block_bytes      # one request's KV: what a full admission moves
        summ_bytes = L * Hkv * nb * 2 * d * 2        # its min/max summaries
        q, dr = _device_inputs(wl, S)
        out = torch.empty(q.shape[1:], dtype=torch.bfloat16, device="cuda")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rows = []
        for cap in wl.w.caps:
            C = max(1, min(kb, int(cap * kb)))
            lcap = min(nb, kb + C * S)  # room for every block the run can demand: nothing bypasses
            cfg = wl.config()
            cfg.fetch_cap = cap
            local = [HostBuffer(cfg.host_bytes(lcap)) for _ in range(B)]
            ctx = Context(cfg)
            for r in range(B):
                ctx.add_request_partial(r, bufs[int(wl.keys[r])].ptr, nb, local[r].ptr, lcap, wl.n_tok)
            ctx.set_timing(True)
            for l in range(L):
                ctx.stage(l, dr[0, l], 0, 1.0)
            adm = ctx.read_timing()
            ctx.set_timing(True)
            ms, done, curve = 0.0, 0, []
            for m in marks:
                e0.record()
                for t in range(done, m):
                    ctx.step(q[t], dr[t + 1], out, t + 1)
                done = m
                ctx.join()
                e1.record()
                e1.synchronize()
                ms += e0.elapsed_time(e1)
                tm = ctx.read_timing()
                dec_bytes = tm["full_reads"] * block_bytes / B
                total = summ_bytes + adm["full_reads"] * block_bytes / B + dec_bytes
                curve.append({"steps": m, "decode_gb_per_request": round(dec_bytes / 1e9, 4),
                              "total_reduction": round(full_bytes / total, 3),
                              "local_hit_frac": round(tm["local_hits"] / max(1, tm["fetched_blocks"]), 4)})
            kept = sum(int(ctx.read_local(l)[0][:B].sum()) for l in range(L))
            passed = tm["full_reads"] - tm["local_fills"] + adm["full_reads"] - adm["local_fills"]
            ctx.close()
            for b in local:
                b.free()
            partial_tok = B * S / (ms / 1e3)
            # the same steps with every request holding its full KV
            ctx = _setup_context(wl, bufs, cap)
            ctx.set_timing(True)
            for l in range(L):
                ctx.stage(l, dr[0, l], 0, 1.0)
            torch.cuda.synchronize()
            e0.record()
            for t in range(S):
                ctx.step(q[t], dr[t + 1], out, t + 1)
            ctx.join()
            e1.record()
            e1.synchronize()
            full_tok = B * S / (e0.elapsed_time(e1) / 1e3)
            ctx.close()
            adm_bytes = summ_bytes + adm["full_reads"] * block_bytes / B
            rows.append({
                "fetch_cap": cap, "C_blocks": C, "decode_steps": S, "decode_side_entries_per_unit": lcap,
                "full_kv_gb_per_request": round(full_bytes / 1e9, 4),
                "admission_gb_per_request": round(adm_bytes / 1e9, 4),
                "admission_summary_gb": round(summ_bytes / 1e9, 4),
                "admission_reduction": round(full_bytes / adm_bytes, 3),
                "curve": curve,
                "decode_side_occupancy_gb_per_request": round(kept * block_bytes / B / 1e9, 4),
                "occupancy_reduction": round(full_bytes / max(1, kept * block_bytes / B), 3),
                "bypassed_blocks": int(passed),
                "partial_tok_s": round(partial_tok, 1), "full_kv_tok_s": round(full_tok, 1)})
        for b in bufs:
            b.free()
        del q, dr, out
        torch.cuda.empty_cache()
        results.append({"workload": name, "context": wl.n_tok, "batch": B, "rows": rows})
    return {"report": "partial", "metric": "admission-time partial staging: full-copy -> decode-side traffic, "
            "decode-side occupancy and tok/s", "unit": "GB per request", "n_gpus": dist.world, "steps": S,
            "data": "synthetic", "workloads": results}


def run_append(args, dist: Dist):
    """Decode steps that append one token per request and layer: the mixed-length workload
    (contexts ~ U[1K, 32K], one token per step), through okv_step with k_new / v_new. Appends go
    to each request's own host buffer (requests sharing a buffer cannot append): at batch 64 and
    256 steps that is 150 GB of page-locked host memory (a 199 GB GB300 host holds it)."""
    import numpy as np
    import torch
    import synth
    from sparse_kv_cache_draft_gb300 import BF16, Config, Context, HostBuffer
    name = args.workload or "qwen3_8b_mixed_b64"
    w = synth.WORKLOADS[name]
    if args.batch:
        w = w.scaled(batch=args.batch)
    if args.layers:
        w = w.scaled(layers=args.layers)
    B, L, Hq, Hkv, d, bs = w.batch, w.layers, w.q_heads, w.kv_heads, w.head_dim, w.block_size
    K, W = args.steps, args.warmup
    n_steps = W + K
    grow = max(1, w.grow_per_step)
    ctx0 = w.contexts().astype(np.int64)
    caps = [-(-(int(c) + grow * (n_steps + 1)) // bs) for c in ctx0]
    cfg = Config(L, Hq, Hkv, d, bs, w.budget_tokens, B, max(caps), w.fetch_cap, BF16)
    ids = np.arange(B, dtype=np.int32)
    threads = args.threads or os.cpu_count() or 1
    t0 = time.time()
    bufs = [HostBuffer(cfg.host_bytes(caps[r])) for r in range(B)]
    for r in range(B):
        synth.fill_kv(bufs[r].ptr, w, r, 0, int(ctx0[r]), caps[r], n_threads=threads)
    host_gb = sum(cfg.host_bytes(c) for c in caps) / 1e9
    log(f"host KV: {B} own buffers, {host_gb:.1f} GB, in {time.time() - t0:.1f}s")
    ctx = Context(cfg)
    for r in range(B):
        ctx.add_request(r, bufs[r].ptr, caps[r], int(ctx0[r]))
    shape_q, shape_kv = (L, B, Hq, d), (L, B, Hkv, d)
    # every step's inputs go straight to device memory, one step at a time on the host (the
    # host's memory holds the requests' KV)
    q = torch.empty((n_steps,) + shape_q, dtype=torch.bfloat16, device="cuda")
    dr = torch.empty((n_steps + 1,) + shape_q, dtype=torch.bfloat16, device="cuda")
    kn = torch.empty((n_steps,) + shape_kv, dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    qh = np.empty(shape_q, np.uint16)
    kh = np.empty(shape_kv, np.uint16)
    vh = np.empty_like(kh)

    def conv(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)

    t0 = time.time()
    for t in range(-1, n_steps):
        for l in range(L):
            synth.queries(w, l, t, 1, ids, ids, out=qh[l], n_threads=threads)
        dr[t + 1].copy_(conv(qh))
        if t >= 0:
            for l in range(L):
                synth.queries(w, l, t, 0, ids, ids, out=qh[l], n_threads=threads)
                kh[l], vh[l] = synth.token_kv(w, l, ids, ctx0 + t * grow)
            q[t].copy_(conv(qh))
            kn[t].copy_(conv(kh))
            vn[t].copy_(conv(vh))
    log(f"inputs for {n_steps} steps generated in {time.time() - t0:.1f}s")
    out = torch.empty(shape_q, dtype=torch.bfloat16, device="cuda")
    for l in range(L):
        ctx.stage(l, dr[0, l], 0, 1.0)
    for t in range(W):
        ctx.step(q[t], dr[t + 1], out, t + 1, k_new=kn[t], v_new=vn[t])
    torch.cuda.synchronize()
    assert ctx.sync(60_000) == 0
    ctx.set_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for t in range(W, n_steps):
        ctx.step(q[t], dr[t + 1], out, t + 1, k_new=kn[t], v_new=vn[t])
    ctx.join()
    e1.record()
    e1.synchronize()
    ms = dist.max(e0.elapsed_time(e1))
    tm = ctx.read_timing()
    assert ctx.sync(60_000) == 0
    lens = ctx.read_lengths(0)[:B]
    assert (lens == ctx0 + grow * n_steps).all(), "every request grew by one token per step"
    hbm_peak, src = measured_peaks()
    slot_bytes = 2 * bs * d * 2
    nb_end = -(-(ctx0 + grow * n_steps) // bs)
    summ_bytes = L * Hkv * int(nb_end.sum()) * 2 * d * 2  # per step, at the final lengths
    att_bytes = tm["attended_slots"] / K * slot_bytes
    step_ms = ms / K
    ctx.close()
    for b in bufs:
        b.free()
    return {"report": "append", "metric": "sparse-decode tok/s with one appended token per request and layer",
            "unit": "tok/s", "n_gpus": dist.world, "steps": K, "warmup": W, "data": "synthetic",
            "workload": f"{name} (batch {B}, {L} layers)", "contexts": {"min": int(ctx0.min()), "mean": float(ctx0.mean()),
                                                                     "max": int(ctx0.max())},
            "host_kv_gb": round(host_gb, 1),
            "tok_s": round(dist.world * B * K / (ms / 1e3), 1), "ms_per_step": round(step_ms, 4),
            "append_us_per_layer": round(tm["ms"]["append"] / (L * K) * 1e3, 2),
            "append_share_of_step": round(tm["ms"]["append"] / K / step_ms, 4),
            "step_hbm_gbs": round((att_bytes + summ_bytes) / (step_ms / 1e3) / 1e9, 1),
            "step_hbm_frac": round((att_bytes + summ_bytes) / (step_ms / 1e3) / 1e9 / hbm_peak, 4),
            "gather_gb_per_step": round(tm["fetched_blocks"] * slot_bytes / K / 1e9, 4),
            "kernel_ms_per_step": {k: round(v / K, 4) for k, v in tm["ms"].items() if v > 0},
            "peak_source": f"hbm_gbs, {src}"}


def main():
    args = parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one rank per GPU, launched here the way the multi-GPU runs are launched
        sys.exit(self_launch(sys.argv[1:], args.gpus))
    dist = Dist(want_gpu=args.impl == "okv")
    try:
        if args.report == "capsweep":
            res = run_capsweep(args, dist) if dist.rank == 0 else None
        elif args.report == "agreement":
            res = run_agreement(args, dist) if dist.rank == 0 else None
        elif args.report == "dense":
            res = run_dense(args, dist) if dist.rank == 0 else None
        elif args.report == "partial":
            res = run_partial(args, dist) if dist.rank == 0 else None
        elif args.report == "append":
            res = run_append(args, dist) if dist.rank == 0 else None
        else:
            res = run_okv(args, dist) if args.impl == "okv" else run_reference(args, dist)
        if res is not None and dist.rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
