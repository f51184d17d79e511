"""ORACLE: test infrastructure, not product code.

Plain CPU restatement (binary64) of OasisKV's per-decode-step path, written from
"4 System Design" of paperlayer.ai/abs/2608.08097v1. The arithmetic lives in
``okv_oracle.c``; this module compiles it and exposes:

* per-unit functions (one (layer, request, kv head) at a time) for the pins, and
* :class:`OracleModel`, the same state machine the GPU library keeps (summaries,
  resident map, slot table, stamps, selections, fetch lists), over whole layers,
  driven through the threaded C driver.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against a
closed form, a brute-force or library computation, or a hand-worked case
(``tests/test_oracle_*.py``, ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libokv_oracle.so")
_SRC = [os.path.join(_HERE, "okv_oracle.c")]
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
DO_SUMMARY, DO_SCORE, DO_SELECT, DO_ATTEND, DO_DENSE = 1, 2, 4, 8, 16


def build(force: bool = False, out_path: str | None = None, sources=None) -> str:
    """Compile the oracle (plain C, binary64, no FMA contraction) next to its source."""
    srcs = sources or _SRC
    path = out_path or _LIB_PATH
    newest = max(os.path.getmtime(p) for p in srcs + [os.path.join(_HERE, "okv_oracle.h")])
    if force or not os.path.exists(path) or os.path.getmtime(path) < newest:
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-Wall", "-I", _HERE, "-o", tmp] + list(srcs) + ["-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


class Unit(ctypes.Structure):
    _fields_ = [
        ("host_unit", ctypes.c_void_p), ("summ", ctypes.c_void_p), ("q", ctypes.c_void_p),
        ("n_tok", ctypes.c_int32), ("n_sel_override", ctypes.c_int32),
        ("sel_override", ctypes.c_void_p), ("resident", ctypes.c_void_p),
        ("slot_block", ctypes.c_void_p), ("stamp", ctypes.c_void_p), ("scores", ctypes.c_void_p),
        ("sel_ids", ctypes.c_void_p), ("sel_scores", ctypes.c_void_p), ("n_sel", ctypes.c_void_p),
        ("fetch", ctypes.c_void_p), ("n_fetch", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("local_cap", ctypes.c_int32), ("local_of", ctypes.c_void_p), ("local_used", ctypes.c_void_p),
        ("route", ctypes.c_void_p),
    ]


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("dtype", "bs", "d", "g", "kb", "cap_blocks", "step")]


def _load(path: str):
    L = ctypes.CDLL(path)
    i32, i64, vp, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    L.oracle_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
    L.oracle_kv_bytes_per_token.restype = i64
    L.oracle_fetch_cap_blocks.argtypes = [f32, i32]
    L.oracle_fetch_cap_blocks.restype = i32
    L.oracle_block_summary.argtypes = [vp, i32, i32, i32, i32, vp]
    L.oracle_block_scores.argtypes = [vp, i32, i32, i32, vp, i32, vp]
    L.oracle_topk.argtypes = [vp, i32, i32, vp]
    L.oracle_topk.restype = i32
    L.oracle_select_update.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, vp]
    L.oracle_select_update.restype = i32
    L.oracle_local_route.argtypes = [vp, vp, i32, vp, i32, vp]
    L.oracle_local_route.restype = i32
    L.oracle_attend.argtypes = [vp, i32, vp, i32, i32, i32, i32, vp, i32, vp]
    L.oracle_dense_attend.argtypes = [vp, i32, i32, i32, i32, vp, i32, vp]
    L.oracle_append.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp]
    L.oracle_run_units.argtypes = [ctypes.POINTER(Unit), i32, ctypes.POINTER(Dims), i32, i32]
    L.oracle_run_units.restype = ctypes.c_int
    for f in (L.oracle_block_summary, L.oracle_block_scores, L.oracle_attend,
              L.oracle_dense_attend, L.oracle_append):
        f.restype = None
    return L


def lib(path: str | None = None):
    """The oracle library; `path` loads another build of it (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _load(path)
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


def _p(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("storage arrays are float32 or uint16 (bfloat16 bits)")


# ---- per-unit functions ----------------------------------------------------------------------

def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int, L=None) -> int:
    return int((L or lib()).oracle_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes))


def fetch_cap_blocks(cap: float, budget_blocks: int, L=None) -> int:
    return int((L or lib()).oracle_fetch_cap_blocks(cap, budget_blocks))


def block_summary(host_unit: np.ndarray, n_tok: int, bs: int, d: int, L=None) -> np.ndarray:
    """host_unit: [cap_blocks][2][bs][d] storage -> [nb][2][d] storage (min, max)."""
    nb = -(-n_tok // bs)
    out = np.zeros((nb, 2, d), dtype=host_unit.dtype)
    (L or lib()).oracle_block_summary(_p(host_unit), _dt(host_unit), n_tok, bs, d, _p(out))
    return out


def block_scores(summ: np.ndarray, q: np.ndarray, L=None) -> np.ndarray:
    """summ: [nb][2][d]; q: [g][d] (same storage type) -> float32 [nb]."""
    nb, _, d = summ.shape
    q = np.ascontiguousarray(q, dtype=summ.dtype)
    out = np.zeros(nb, dtype=np.float32)
    (L or lib()).oracle_block_scores(_p(summ), _dt(summ), nb, d, _p(q), q.shape[0], _p(out))
    return out


def topk(scores: np.ndarray, kb: int, L=None) -> np.ndarray:
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    ids = np.zeros(max(1, min(kb, len(scores))), dtype=np.int32)
    n = (L or lib()).oracle_topk(_p(scores), len(scores), kb, _p(ids))
    return ids[:n].copy()


def select_update(resident: np.ndarray, slot_block: np.ndarray, stamp: np.ndarray, sel,
                  cap_blocks: int, step: int, L=None) -> np.ndarray:
    """Updates resident / slot_block / stamp (int32 arrays) in place; returns fetch [n][2]."""
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    kb = len(slot_block)
    fetch = np.zeros((kb, 2), dtype=np.int32)
    n = (L or lib()).oracle_select_update(_p(resident), _p(slot_block), _p(stamp), kb,
                                          _p(sel), len(sel), cap_blocks, step, _p(fetch))
    return fetch[:n].copy()


def local_route(local_of: np.ndarray, local_used: np.ndarray, local_cap: int, fetch,
                L=None) -> tuple[np.ndarray, int]:
    """Routes a fetch list ([n][2] (block, slot)) through a request's decode-side tier.

    Updates local_of ([nb] int32) and local_used (int32 array of one element) in place; returns
    (route [n] int32, number of entries read from the full copy)."""
    fetch = np.ascontiguousarray(np.asarray(fetch, dtype=np.int32).reshape(-1, 2))
    route = np.full(max(1, len(fetch)), -1, dtype=np.int32)
    n = (L or lib()).oracle_local_route(_p(local_of), _p(local_used), local_cap, _p(fetch),
                                        len(fetch), _p(route))
    return route[:len(fetch)].copy(), int(n)


def attend(host_unit: np.ndarray, slot_block: np.ndarray, n_tok: int, bs: int, d: int,
           q: np.ndarray, L=None) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=host_unit.dtype)
    slot_block = np.ascontiguousarray(slot_block, dtype=np.int32)
    out = np.zeros((q.shape[0], d), dtype=np.float64)
    (L or lib()).oracle_attend(_p(host_unit), _dt(host_unit), _p(slot_block), len(slot_block),
                               n_tok, bs, d, _p(q), q.shape[0], _p(out))
    return out


def dense_attend(host_unit: np.ndarray, n_tok: int, bs: int, d: int, q: np.ndarray,
                 L=None) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=host_unit.dtype)
    out = np.zeros((q.shape[0], d), dtype=np.float64)
    (L or lib()).oracle_dense_attend(_p(host_unit), _dt(host_unit), n_tok, bs, d, _p(q),
                                     q.shape[0], _p(out))
    return out


def append(host_unit: np.ndarray, summ: np.ndarray, n_tok: int, bs: int, d: int,
           k: np.ndarray, v: np.ndarray, L=None) -> None:
    k = np.ascontiguousarray(k, dtype=host_unit.dtype)
    v = np.ascontiguousarray(v, dtype=host_unit.dtype)
    (L or lib()).oracle_append(_p(host_unit), _p(summ), _dt(host_unit), n_tok, bs, d, _p(k), _p(v))


# ---- whole-layer model -----------------------------------------------------------------------

class OracleModel:
    """The oracle's copy of the staging state for every (layer, request, kv head).

    Host KV comes in one of two ways:

    * ``host_fill`` (what the parity tests use): the oracle keeps a private copy of every kept
      layer of every distinct content, ``req_keys[r]`` naming request r's content. The copy of
      (layer, key) is a [kv_heads][cap_blocks][2][bs][d] array of the storage type that
      ``host_fill(layer, key, array)`` fills from the seeded generator. Requests with the same
      key share it. Nothing the CUDA library writes reaches these bytes: appends are applied
      to them by :meth:`append`.
    * ``req_ptrs`` (timing only): request r's buffer at a raw address, laid out
      [layers][kv_heads][cap_blocks[r]][2][bs][d].

    Summaries and the per-unit tables live in numpy arrays here.

    ``local_cap[r]`` >= 0 marks request r as partially staged: its fetch lists are also routed
    through a decode-side tier of that many entries per unit (``local_of``, ``local_used``,
    ``route``); -1 (the default) marks a request that holds its full KV.
    """

    def __init__(self, *, layers, q_heads, kv_heads, head_dim, block_size, budget_tokens,
                 dtype, cap_blocks, n_tok, req_ptrs=None, host_fill=None, req_keys=None,
                 n_threads=None, layers_kept=None, local_cap=None):
        self.L, self.Hq, self.Hkv, self.d, self.bs = layers, q_heads, kv_heads, head_dim, block_size
        self.g = q_heads // kv_heads
        self.kb = budget_tokens // block_size
        self.dtype = dtype
        self.elem = 4 if dtype == F32 else 2
        self.sdt = np.float32 if dtype == F32 else np.uint16
        if (req_ptrs is None) == (host_fill is None):
            raise ValueError("give either req_ptrs or host_fill")
        self.B = len(req_ptrs) if req_ptrs is not None else len(req_keys)
        self.req_ptrs = [int(p) for p in req_ptrs] if req_ptrs is not None else None
        self.cap_blocks = np.asarray(cap_blocks, dtype=np.int64)
        self.n_tok = np.array(np.broadcast_to(np.asarray(n_tok, dtype=np.int32),
                                              (layers, self.B)))
        self.nb_max = int(self.cap_blocks.max())
        self.layers_kept = list(range(layers)) if layers_kept is None else list(layers_kept)
        self.n_threads = n_threads or os.cpu_count() or 1
        shp = (self.B, self.Hkv)
        self.summ = {l: np.zeros(shp + (self.nb_max, 2, self.d), dtype=self.sdt) for l in self.layers_kept}
        self.resident = {l: np.full(shp + (self.nb_max,), -1, dtype=np.int32) for l in self.layers_kept}
        self.slot_block = {l: np.full(shp + (self.kb,), -1, dtype=np.int32) for l in self.layers_kept}
        self.stamp = {l: np.full(shp + (self.kb,), -1, dtype=np.int32) for l in self.layers_kept}
        self.sel_ids = {l: np.full(shp + (self.kb,), -1, dtype=np.int32) for l in self.layers_kept}
        self.sel_scores = {l: np.zeros(shp + (self.kb,), dtype=np.float32) for l in self.layers_kept}
        self.n_sel = {l: np.zeros(shp, dtype=np.int32) for l in self.layers_kept}
        self.fetch = {l: np.zeros(shp + (self.kb, 2), dtype=np.int32) for l in self.layers_kept}
        self.n_fetch = {l: np.zeros(shp, dtype=np.int32) for l in self.layers_kept}
        self.scores = {l: np.zeros(shp + (self.nb_max,), dtype=np.float32) for l in self.layers_kept}
        self.local_cap = np.full(self.B, -1, dtype=np.int32) if local_cap is None else \
            np.array(np.broadcast_to(np.asarray(local_cap, dtype=np.int32), (self.B,)))
        self.local_of = {l: np.full(shp + (self.nb_max,), -1, dtype=np.int32) for l in self.layers_kept}
        self.local_used = {l: np.zeros(shp, dtype=np.int32) for l in self.layers_kept}
        self.route = {l: np.full(shp + (self.kb,), -1, dtype=np.int32) for l in self.layers_kept}
        self.host = None
        if host_fill is not None:
            self.req_keys = [int(k) for k in req_keys]
            self.host = {}
            for l in self.layers_kept:
                for r, k in enumerate(self.req_keys):
                    if (l, k) in self.host:
                        continue
                    a = np.zeros((self.Hkv, int(self.cap_blocks[r]), 2, self.bs, self.d), dtype=self.sdt)
                    host_fill(l, k, a)
                    self.host[(l, k)] = a

    def host_unit_ptr(self, layer: int, r: int, h: int) -> int:
        if self.host is not None:
            return self.host[(layer, self.req_keys[r])][h].ctypes.data
        unit = int(self.cap_blocks[r]) * 2 * self.bs * self.d
        return self.req_ptrs[r] + (layer * self.Hkv + h) * unit * self.elem

    def host_unit(self, layer: int, r: int, h: int) -> np.ndarray:
        """numpy view of one unit's host region (no copy): [cap_blocks][2][bs][d]."""
        if self.host is not None:
            return self.host[(layer, self.req_keys[r])][h]
        n = int(self.cap_blocks[r]) * 2 * self.bs * self.d
        buf = (ctypes.c_char * (n * self.elem)).from_address(self.host_unit_ptr(layer, r, h))
        return np.frombuffer(buf, dtype=self.sdt).reshape(int(self.cap_blocks[r]), 2, self.bs, self.d)

    def _units(self, layer, q=None, out=None, sel_override=None, requests=None):
        reqs = range(self.B) if requests is None else requests
        units = []
        keep = []
        for r in reqs:
            for h in range(self.Hkv):
                u = Unit()
                u.host_unit = self.host_unit_ptr(layer, r, h)
                u.summ = self.summ[layer][r, h].ctypes.data
                if q is not None:
                    qq = np.ascontiguousarray(q[r, h * self.g:(h + 1) * self.g])
                    keep.append(qq)
                    u.q = qq.ctypes.data
                u.n_tok = int(self.n_tok[layer, r])
                u.n_sel_override = -1
                if sel_override is not None:
                    ids, cnt = sel_override
                    so = np.ascontiguousarray(ids[r, h, :cnt[r, h]], dtype=np.int32)
                    keep.append(so)
                    u.sel_override = so.ctypes.data
                    u.n_sel_override = int(cnt[r, h])
                u.resident = self.resident[layer][r, h].ctypes.data
                u.slot_block = self.slot_block[layer][r, h].ctypes.data
                u.stamp = self.stamp[layer][r, h].ctypes.data
                u.scores = self.scores[layer][r, h].ctypes.data
                u.sel_ids = self.sel_ids[layer][r, h].ctypes.data
                u.sel_scores = self.sel_scores[layer][r, h].ctypes.data
                u.n_sel = self.n_sel[layer][r, h:h + 1].ctypes.data
                u.fetch = self.fetch[layer][r, h].ctypes.data
                u.n_fetch = self.n_fetch[layer][r, h:h + 1].ctypes.data
                if out is not None:
                    u.out = out[r, h * self.g:(h + 1) * self.g].ctypes.data
                u.local_cap = int(self.local_cap[r])
                u.local_of = self.local_of[layer][r, h].ctypes.data
                u.local_used = self.local_used[layer][r, h:h + 1].ctypes.data
                u.route = self.route[layer][r, h].ctypes.data
                units.append(u)
        return (Unit * len(units))(*units), keep

    def _run(self, units, what, cap_blocks=1, step=0):
        dims = Dims(self.dtype, self.bs, self.d, self.g, self.kb, cap_blocks, step)
        rc = lib().oracle_run_units(units, len(units), ctypes.byref(dims), what, self.n_threads)
        if rc != 0:
            raise RuntimeError("oracle_run_units failed")

    def build_summaries(self, layer: int, requests=None) -> None:
        units, _k = self._units(layer, requests=requests)
        self._run(units, DO_SUMMARY)

    def score_topk(self, layer: int, draft: np.ndarray, requests=None) -> None:
        """draft: [B][Hq][d] storage. Fills scores / sel_ids / sel_scores / n_sel."""
        units, _k = self._units(layer, q=np.ascontiguousarray(draft), requests=requests)
        self._run(units, DO_SCORE)

    def select(self, layer: int, cap_blocks: int, step: int, sel_override=None, requests=None) -> None:
        """Diff / admit / evict; sel_override = (ids[B][Hkv][kb], counts[B][Hkv]) re-syncs the
        selection to a given (validated) one."""
        units, _k = self._units(layer, sel_override=sel_override, requests=requests)
        self._run(units, DO_SELECT, cap_blocks, step)

    def stage(self, layer: int, draft: np.ndarray, cap_blocks: int, step: int) -> None:
        self.score_topk(layer, draft)
        self.select(layer, cap_blocks, step)

    def attend(self, layer: int, q: np.ndarray, requests=None, dense: bool = False) -> np.ndarray:
        """q: [B][Hq][d] storage -> float64 [B][Hq][d] (rows of requests not listed stay 0)."""
        out = np.zeros((self.B, self.Hq, self.d), dtype=np.float64)
        units, _k = self._units(layer, q=np.ascontiguousarray(q), out=out, requests=requests)
        self._run(units, DO_DENSE if dense else DO_ATTEND)
        return out

    def append(self, layer: int, k_new: np.ndarray, v_new: np.ndarray) -> None:
        """k_new, v_new: [B][Hkv][d] storage; appends at n_tok[layer, r] then advances it."""
        for r in range(self.B):
            for h in range(self.Hkv):
                hu = self.host_unit(layer, r, h)
                append(hu, self.summ[layer][r, h], int(self.n_tok[layer, r]), self.bs, self.d,
                       k_new[r, h], v_new[r, h])
            self.n_tok[layer, r] += 1
