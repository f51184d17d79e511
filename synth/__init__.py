"""Seeded synthetic workload (host KV, queries, drafts, appended tokens).

A module of its own: it generates inputs only and holds none of the method's
arithmetic, so the CPU oracle and the GPU path both read its output without
sharing any computation. The C source is ``synth.c`` (definitions in ``synth.h``);
this file compiles it on first use and wraps it with ctypes.

Workload presets (:data:`WORKLOADS`) restate the evaluation shapes of OasisKV
(paperlayer.ai/abs/2608.08097v1, "5 Evaluation"; agihunt.info/papers/2608.08097
throughput table): Qwen3-8B attention shapes at 16K context and batch 128, a mixed
1K-32K reasoning-length batch that grows one token per step, the 32B-class GQA
shape from "2 Background" (256 KiB of KV per token), and the fetch-cap sweep.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libokvsynth.so")
_SRC = [os.path.join(_HERE, "synth.c")]
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
PLANT_MOD, PLANT_COUNT = 0, 1


def build(force: bool = False) -> str:
    """Compile libokvsynth.so next to its source (plain C, no arch flags)."""
    newest = max(os.path.getmtime(p) for p in _SRC + [os.path.join(_HERE, "synth.h")])
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-Wall", "-o", tmp] + _SRC + ["-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class SynthParams(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("layers", ctypes.c_int32), ("q_heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("plant_mode", ctypes.c_int32), ("n_dirs", ctypes.c_int32),
        ("n_plant", ctypes.c_int32), ("plant_blocks", ctypes.c_int32),
        ("n_active", ctypes.c_int32), ("active_period", ctypes.c_int32),
        ("amplitude", ctypes.c_double), ("sigma_q", ctypes.c_double), ("sigma_d", ctypes.c_double),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.POINTER(SynthParams)
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            L.synth_fill_kv.argtypes = [vp, P, i32, i32, i32, i32, i32]
            L.synth_fill_kv_layer.argtypes = [vp, P, i32, i32, i32, i32, i32, i32]
            L.synth_queries.argtypes = [vp, P, i32, i32, i32, i32, vp, vp, i32]
            L.synth_token_kv.argtypes = [vp, vp, P, i32, i32, vp, vp]
            L.synth_direction.argtypes = [vp, P, i32, i32, i32, i32]
            L.synth_block_direction.argtypes = [P, i32, i32, i32, i32]
            L.synth_block_direction.restype = i32
            L.synth_normals.argtypes = [vp, i64, ctypes.c_uint64, ctypes.c_uint64,
                                        ctypes.c_uint64, ctypes.c_uint64]
            for f in (L.synth_fill_kv, L.synth_fill_kv_layer, L.synth_queries, L.synth_token_kv,
                      L.synth_direction, L.synth_normals):
                f.restype = ctypes.c_int
            _lib = L
    return _lib


@dataclass
class Workload:
    """Shapes, method parameters and generator recipe of one synthetic workload."""
    name: str
    seed: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    batch: int
    context: int                 # tokens per request (or the mean, for mixed lengths)
    block_size: int = 16
    budget_tokens: int = 2048
    fetch_cap: float = 0.05
    dtype: int = BF16
    steps: int = 1
    plant_mode: int = PLANT_MOD
    n_dirs: int = 20
    plant_frac: float = 0.05     # PLANT_COUNT: fraction of blocks planted
    n_active: int = 1
    active_period: int = 1
    amplitude: float = 3.0
    sigma_q: float = 0.5
    sigma_d: float = 0.1
    ctx_min: int = 0             # mixed lengths: per-request context ~ U[ctx_min, ctx_max]
    ctx_max: int = 0
    grow_per_step: int = 0       # tokens appended per request per decode step
    caps: tuple = field(default_factory=tuple)  # fetch-cap sweep values

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def contexts(self) -> np.ndarray:
        """Per-request initial context lengths (seeded, independent of the method)."""
        if self.ctx_max > 0:
            rng = np.random.default_rng(self.seed * 7919 + 11)
            return rng.integers(self.ctx_min, self.ctx_max + 1, size=self.batch).astype(np.int32)
        return np.full(self.batch, self.context, dtype=np.int32)

    def max_tokens(self) -> int:
        return int(self.contexts().max()) + self.grow_per_step * self.steps

    def params(self, n_blocks_plant: int | None = None) -> SynthParams:
        nb = n_blocks_plant if n_blocks_plant is not None else -(-self.context // self.block_size)
        n_plant = int(round(self.plant_frac * nb)) if self.plant_mode == PLANT_COUNT else 0
        return SynthParams(self.seed, self.layers, self.q_heads, self.kv_heads, self.head_dim,
                           self.block_size, self.dtype, self.plant_mode, self.n_dirs, n_plant, nb,
                           self.n_active, self.active_period, self.amplitude, self.sigma_q,
                           self.sigma_d)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # batch 2, GQA 8/2, d 64, 4096 tokens, budget 512 (32 blocks), cap 1.0, fp32, 5% of blocks
    # planted with one direction u, query = u + N(0, 0.5^2), draft = query + N(0, 0.1^2)
    "tiny": Workload("tiny", seed=1, layers=1, q_heads=8, kv_heads=2, head_dim=64, batch=2,
                     context=4096, budget_tokens=512, fetch_cap=1.0, dtype=F32, steps=1,
                     plant_mode=PLANT_COUNT, n_dirs=1, plant_frac=0.05),
    # Qwen3-8B attention shapes, 16K context, batch 128, 64 steps, heavy set = blocks
    # b = t (mod 20): 5% of the blocks, moving one block index per step
    "qwen3_8b_16k_b128": Workload("qwen3_8b_16k_b128", seed=2, layers=36, q_heads=32,
                                  kv_heads=8, head_dim=128, batch=128, context=16384, steps=64,
                                  n_dirs=20),
    # reasoning-style mixed lengths U[1K, 32K], +1 token per step over 256 steps, heavy
    # direction changes every 32 steps
    "qwen3_8b_mixed_b64": Workload("qwen3_8b_mixed_b64", seed=3, layers=36, q_heads=32,
                                   kv_heads=8, head_dim=128, batch=64, context=16896,
                                   ctx_min=1024, ctx_max=32768, grow_per_step=1, steps=256,
                                   n_dirs=20, active_period=32),
    # 32B-class GQA (64 layers, 64/8 heads, d 128): 256 KiB of KV per token, 32K context
    "gqa32b_32k_b32": Workload("gqa32b_32k_b32", seed=4, layers=64, q_heads=64, kv_heads=8,
                               head_dim=128, batch=32, context=32768, steps=32, n_dirs=33),
    # fetch-cap sweep: 100 directions at 1% of blocks each, 5 active, one replaced per step
    "qwen3_8b_capsweep_b90": Workload("qwen3_8b_capsweep_b90", seed=5, layers=36, q_heads=32,
                                      kv_heads=8, head_dim=128, batch=90, context=16384,
                                      steps=16, n_dirs=100, n_active=5,
                                      caps=(0.01, 0.02, 0.05, 0.1, 0.25, 1.0)),
    # admission-time partial staging at the disaggregated-serving contexts (24K and 32K): the
    # cap-sweep structure (100 directions at 1% of blocks, 5 active, one replaced per step), so
    # decode-time demand keeps drifting to blocks the admission did not stage
    "qwen3_8b_pd_24k_b8": Workload("qwen3_8b_pd_24k_b8", seed=6, layers=36, q_heads=32, kv_heads=8,
                                   head_dim=128, batch=8, context=24576, steps=256, n_dirs=100,
                                   n_active=5, caps=(0.05, 1.0)),
    "qwen3_8b_pd_32k_b8": Workload("qwen3_8b_pd_32k_b8", seed=7, layers=36, q_heads=32, kv_heads=8,
                                   head_dim=128, batch=8, context=32768, steps=256, n_dirs=100,
                                   n_active=5, caps=(0.05, 1.0)),
}


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def np_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def fill_kv(buf_ptr: int, w: Workload, req_key: int, tok_begin: int, tok_end: int,
            cap_blocks: int, n_threads: int | None = None, plant_blocks: int | None = None) -> None:
    """Fill one request's host KV buffer (layout [L][Hkv][cap_blocks][2][bs][d])."""
    p = w.params(plant_blocks)
    nt = n_threads or os.cpu_count() or 1
    rc = lib().synth_fill_kv(ctypes.c_void_p(buf_ptr), ctypes.byref(p), req_key, tok_begin,
                             tok_end, cap_blocks, nt)
    if rc != 0:
        raise ValueError("synth_fill_kv: bad arguments")


def fill_kv_layer(out: np.ndarray, w: Workload, req_key: int, layer: int, tok_begin: int, tok_end: int,
                  n_threads: int | None = None, plant_blocks: int | None = None) -> None:
    """Fill one layer of one request into `out`, a C-contiguous [Hkv][cap_blocks][2][bs][d] array
    of the storage dtype: the bytes fill_kv writes for that layer."""
    assert out.flags["C_CONTIGUOUS"] and out.dtype == np_dtype(w.dtype)
    assert out.shape[0] == w.kv_heads and out.shape[2:] == (2, w.block_size, w.head_dim)
    p = w.params(plant_blocks)
    nt = n_threads or os.cpu_count() or 1
    rc = lib().synth_fill_kv_layer(ctypes.c_void_p(_ptr(out)), ctypes.byref(p), req_key, layer, tok_begin,
                                   tok_end, out.shape[1], nt)
    if rc != 0:
        raise ValueError("synth_fill_kv_layer: bad arguments")


def queries(w: Workload, layer: int, step: int, kind: int, req_ids, req_keys,
            out: np.ndarray | None = None, n_threads: int | None = None,
            plant_blocks: int | None = None) -> np.ndarray:
    """Query (kind 0) or draft query (kind 1) of one layer: [batch][Hq][d] storage dtype."""
    ids = np.ascontiguousarray(req_ids, dtype=np.int32)
    keys = np.ascontiguousarray(req_keys, dtype=np.int32)
    if out is None:
        out = np.empty((len(ids), w.q_heads, w.head_dim), dtype=np_dtype(w.dtype))
    p = w.params(plant_blocks)
    nt = n_threads or min(len(ids), os.cpu_count() or 1)
    rc = lib().synth_queries(ctypes.c_void_p(_ptr(out)), ctypes.byref(p), layer, step, kind,
                             len(ids), ctypes.c_void_p(_ptr(ids)), ctypes.c_void_p(_ptr(keys)), nt)
    if rc != 0:
        raise ValueError("synth_queries: bad arguments")
    return out


def token_kv(w: Workload, layer: int, req_keys, positions, plant_blocks: int | None = None):
    """K and V of one appended token per request: two [batch][Hkv][d] arrays."""
    keys = np.ascontiguousarray(req_keys, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    k = np.empty((len(keys), w.kv_heads, w.head_dim), dtype=np_dtype(w.dtype))
    v = np.empty_like(k)
    p = w.params(plant_blocks)
    rc = lib().synth_token_kv(ctypes.c_void_p(_ptr(k)), ctypes.c_void_p(_ptr(v)), ctypes.byref(p),
                              layer, len(keys), ctypes.c_void_p(_ptr(keys)),
                              ctypes.c_void_p(_ptr(pos)))
    if rc != 0:
        raise ValueError("synth_token_kv: bad arguments")
    return k, v


def direction(w: Workload, layer: int, req_key: int, kv_head: int, j: int) -> np.ndarray:
    out = np.empty(w.head_dim, dtype=np.float64)
    p = w.params()
    lib().synth_direction(ctypes.c_void_p(_ptr(out)), ctypes.byref(p), layer, req_key, kv_head, j)
    return out


def block_direction(w: Workload, layer: int, req_key: int, kv_head: int, block: int,
                    plant_blocks: int | None = None) -> int:
    p = w.params(plant_blocks)
    return int(lib().synth_block_direction(ctypes.byref(p), layer, req_key, kv_head, block))


def normals(n: int, seed: int, stream: int = 0, a: int = 0, b: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_normals(ctypes.c_void_p(_ptr(out)), n, seed, stream, a, b)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def to_f64(a: np.ndarray, dtype: int) -> np.ndarray:
    return (a if dtype == F32 else bf16_to_f32(a)).astype(np.float64)
