"""ctypes binding of libokv.so: the C ABI of include/okv.h with the same names.

Argument marshalling only: tensors become device pointers, streams become cudaStream_t
handles, host arrays become numpy views. Every step of the path runs in the library's CUDA
kernels; nothing here computes. The library must have been built for sm_103a
(``python -m sparse_kv_cache_draft_gb300.build``); loading fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

F32, BF16 = 0, 1
OK, EINVAL, ENOMEM, ECUDA, EDEVICE, ETIMEOUT, ESTATE = range(7)
KERNEL_KINDS = ("summary", "score_topk", "coef", "gather", "attend", "combine", "append")

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return os.path.join(_HERE, "libokv.so")


class OkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"okv status {status}: {msg}")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("q_heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("budget_tokens", ctypes.c_int32), ("max_requests", ctypes.c_int32),
                ("max_blocks_per_request", ctypes.c_int32), ("fetch_cap", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


class _Timing(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_double * 7), ("launches", ctypes.c_int64 * 7),
                ("fetched_blocks", ctypes.c_int64), ("attended_slots", ctypes.c_int64),
                ("local_hits", ctypes.c_int64), ("local_fills", ctypes.c_int64), ("full_reads", ctypes.c_int64)]


def load_library():
    """Load libokv.so (raises ImportError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with `python -m sparse_kv_cache_draft_gb300.build` "
                              "(nvcc, sm_103a); there is no CPU fallback")
        L = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        st = ctypes.c_int
        sig = {
            "okv_create": ([ctypes.POINTER(_Config), ctypes.POINTER(vp)], st),
            "okv_destroy": ([vp], None),
            "okv_last_error": ([vp], ctypes.c_char_p),
            "okv_status_string": ([st], ctypes.c_char_p),
            "okv_host_alloc": ([i64, ctypes.POINTER(vp)], st),
            "okv_host_free": ([vp], st),
            "okv_add_request": ([vp, i32, vp, i32, i32, vp], st),
            "okv_add_request_partial": ([vp, i32, vp, i32, vp, i32, i32, vp], st),
            "okv_remove_request": ([vp, i32], st),
            "okv_append": ([vp, i32, vp, vp, vp], st),
            "okv_stage": ([vp, i32, vp, i32, f32, vp], st),
            "okv_attend": ([vp, i32, vp, vp, vp], st),
            "okv_attend_lookahead": ([vp, i32, vp, vp, vp, vp, vp], st),
            "okv_predict": ([vp, i32, vp, vp, vp, vp], st),
            "okv_step": ([vp, vp, vp, vp, vp, vp, i32, f32, vp], st),
            "okv_sync": ([vp, i64], st),
            "okv_join": ([vp, vp], st),
            "okv_read_summaries": ([vp, i32, i32, vp], st),
            "okv_read_selection": ([vp, i32, vp, vp, vp], st),
            "okv_read_slot_table": ([vp, i32, vp, vp], st),
            "okv_read_fetch_list": ([vp, i32, vp, vp], st),
            "okv_read_pool": ([vp, i32, i32, i32, vp], st),
            "okv_read_lengths": ([vp, i32, vp], st),
            "okv_read_local": ([vp, i32, vp, vp, vp], st),
            "okv_set_timing": ([vp, i32], st),
            "okv_read_timing": ([vp, ctypes.POINTER(_Timing)], st),
            "okv_launch_count": ([vp], i64),
            "okv_attend_static": ([i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp], st),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
        return L


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _np_ptr(a: np.ndarray) -> ctypes.c_void_p:
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


@dataclass
class Config:
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    block_size: int
    budget_tokens: int
    max_requests: int
    max_blocks_per_request: int
    fetch_cap: float = 0.05
    dtype: int = BF16

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def slots(self) -> int:
        return self.budget_tokens // self.block_size

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def host_bytes(self, capacity_blocks: int) -> int:
        """Bytes of one request's host KV buffer in the okv host layout."""
        return (self.layers * self.kv_heads * capacity_blocks * 2 * self.block_size * self.head_dim
                * self.elem_bytes)

    def _c(self) -> _Config:
        return _Config(self.layers, self.q_heads, self.kv_heads, self.head_dim, self.block_size,
                       self.budget_tokens, self.max_requests, self.max_blocks_per_request,
                       self.fetch_cap, self.dtype)


class HostBuffer:
    """Page-locked, device-mapped host memory from okv_host_alloc."""

    def __init__(self, nbytes: int):
        L = load_library()
        p = ctypes.c_void_p()
        st = L.okv_host_alloc(nbytes, ctypes.byref(p))
        if st != OK:
            raise OkvError(st, f"okv_host_alloc({nbytes}) failed")
        self.ptr = int(p.value)
        self.nbytes = nbytes

    def numpy(self, dtype=np.uint8, shape=None) -> np.ndarray:
        buf = (ctypes.c_char * self.nbytes).from_address(self.ptr)
        a = np.frombuffer(buf, dtype=dtype)
        return a.reshape(shape) if shape is not None else a

    def free(self) -> None:
        if self.ptr:
            load_library().okv_host_free(ctypes.c_void_p(self.ptr))
            self.ptr = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Context:
    """One okv context (okv_create). Methods mirror the C calls."""

    def __init__(self, cfg: Config):
        self.L = load_library()
        self.cfg = cfg
        h = ctypes.c_void_p()
        st = self.L.okv_create(ctypes.byref(cfg._c()), ctypes.byref(h))
        if st != OK:
            raise OkvError(st, "okv_create failed (see stderr)")
        self.h = h

    # -- helpers -------------------------------------------------------------------------------
    def _check(self, st: int, what: str) -> None:
        if st != OK:
            msg = self.L.okv_last_error(self.h).decode(errors="replace")
            raise OkvError(st, f"{what}: {msg}")

    def _tensor_ptr(self, t, shape, what: str) -> ctypes.c_void_p:
        import torch
        want = torch.float32 if self.cfg.dtype == F32 else torch.bfloat16
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{what}: expected a CUDA tensor")
        if t.dtype != want or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{what}: expected contiguous {want} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
        return ctypes.c_void_p(t.data_ptr())

    @property
    def _qshape(self):
        c = self.cfg
        return (c.max_requests, c.q_heads, c.head_dim)

    @property
    def _kvshape(self):
        c = self.cfg
        return (c.max_requests, c.kv_heads, c.head_dim)

    # -- calls ---------------------------------------------------------------------------------
    def add_request(self, req: int, host_ptr: int, capacity_blocks: int, n_tokens: int, stream=None):
        self._check(self.L.okv_add_request(self.h, req, ctypes.c_void_p(host_ptr), capacity_blocks, n_tokens,
                                           ctypes.c_void_p(_stream_handle(stream))), "okv_add_request")

    def add_request_partial(self, req: int, full_ptr: int, capacity_blocks: int, local_ptr: int,
                            local_capacity_blocks: int, n_tokens: int, stream=None):
        self._check(self.L.okv_add_request_partial(self.h, req, ctypes.c_void_p(full_ptr), capacity_blocks,
                                                   ctypes.c_void_p(local_ptr or None), local_capacity_blocks,
                                                   n_tokens, ctypes.c_void_p(_stream_handle(stream))),
                    "okv_add_request_partial")

    def remove_request(self, req: int):
        self._check(self.L.okv_remove_request(self.h, req), "okv_remove_request")

    def append(self, layer: int, k_new, v_new, stream=None):
        self._check(self.L.okv_append(self.h, layer, self._tensor_ptr(k_new, self._kvshape, "k_new"),
                                      self._tensor_ptr(v_new, self._kvshape, "v_new"),
                                      ctypes.c_void_p(_stream_handle(stream))), "okv_append")

    def stage(self, layer: int, draft, step: int, fetch_cap: float = -1.0, stream=None):
        self._check(self.L.okv_stage(self.h, layer, self._tensor_ptr(draft, self._qshape, "draft"), step,
                                     fetch_cap, ctypes.c_void_p(_stream_handle(stream))), "okv_stage")

    def attend(self, layer: int, q, out, stream=None):
        self._check(self.L.okv_attend(self.h, layer, self._tensor_ptr(q, self._qshape, "q"),
                                      self._tensor_ptr(out, self._qshape, "out"),
                                      ctypes.c_void_p(_stream_handle(stream))), "okv_attend")

    def predict(self, layer: int, query, counts, ids, stream=None):
        """Top-K of `query` into device int32 tensors counts [R][Hkv] and ids [R][Hkv][Kb]."""
        import torch
        c = self.cfg
        for name, t, shp in (("counts", counts, (c.max_requests, c.kv_heads)),
                             ("ids", ids, (c.max_requests, c.kv_heads, c.slots))):
            if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous() or tuple(t.shape) != shp:
                raise ValueError(f"{name}: expected contiguous CUDA int32 {shp}")
        self._check(self.L.okv_predict(self.h, layer, self._tensor_ptr(query, self._qshape, "query"),
                                       ctypes.c_void_p(counts.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
                                       ctypes.c_void_p(_stream_handle(stream))), "okv_predict")

    def attend_lookahead(self, layer: int, q, draft, out, draft_out, stream=None):
        self._check(self.L.okv_attend_lookahead(self.h, layer, self._tensor_ptr(q, self._qshape, "q"),
                                                self._tensor_ptr(draft, self._qshape, "draft"),
                                                self._tensor_ptr(out, self._qshape, "out"),
                                                self._tensor_ptr(draft_out, self._qshape, "draft_out"),
                                                ctypes.c_void_p(_stream_handle(stream))), "okv_attend_lookahead")

    def step(self, q, draft, out, step: int, fetch_cap: float = -1.0, k_new=None, v_new=None, stream=None):
        c = self.cfg
        qs = (c.layers,) + self._qshape
        kvs = (c.layers,) + self._kvshape
        kp = self._tensor_ptr(k_new, kvs, "k_new") if k_new is not None else ctypes.c_void_p(0)
        vp = self._tensor_ptr(v_new, kvs, "v_new") if v_new is not None else ctypes.c_void_p(0)
        self._check(self.L.okv_step(self.h, self._tensor_ptr(q, qs, "q"), self._tensor_ptr(draft, qs, "draft"),
                                    self._tensor_ptr(out, qs, "out"), kp, vp, step, fetch_cap,
                                    ctypes.c_void_p(_stream_handle(stream))), "okv_step")

    def join(self, stream=None):
        self._check(self.L.okv_join(self.h, ctypes.c_void_p(_stream_handle(stream))), "okv_join")

    def sync(self, timeout_ms: int = -1) -> int:
        st = self.L.okv_sync(self.h, timeout_ms)
        if st not in (OK, ETIMEOUT):
            self._check(st, "okv_sync")
        return st

    def read_summaries(self, layer: int, req: int) -> np.ndarray:
        c = self.cfg
        dt = np.float32 if c.dtype == F32 else np.uint16
        out = np.empty((c.kv_heads, c.max_blocks_per_request, 2, c.head_dim), dtype=dt)
        self._check(self.L.okv_read_summaries(self.h, layer, req, _np_ptr(out)), "okv_read_summaries")
        return out

    def read_selection(self, layer: int):
        c = self.cfg
        counts = np.empty((c.max_requests, c.kv_heads), np.int32)
        ids = np.empty((c.max_requests, c.kv_heads, c.slots), np.int32)
        scores = np.empty((c.max_requests, c.kv_heads, c.slots), np.float32)
        self._check(self.L.okv_read_selection(self.h, layer, _np_ptr(counts), _np_ptr(ids), _np_ptr(scores)),
                    "okv_read_selection")
        return counts, ids, scores

    def read_slot_table(self, layer: int):
        c = self.cfg
        sb = np.empty((c.max_requests, c.kv_heads, c.slots), np.int32)
        stamps = np.empty_like(sb)
        self._check(self.L.okv_read_slot_table(self.h, layer, _np_ptr(sb), _np_ptr(stamps)), "okv_read_slot_table")
        return sb, stamps

    def read_fetch_list(self, layer: int):
        c = self.cfg
        counts = np.empty((c.max_requests, c.kv_heads), np.int32)
        entries = np.empty((c.max_requests, c.kv_heads, c.slots, 2), np.int32)
        self._check(self.L.okv_read_fetch_list(self.h, layer, _np_ptr(counts), _np_ptr(entries)),
                    "okv_read_fetch_list")
        return counts, entries

    def read_pool(self, layer: int, req: int, kv_head: int) -> np.ndarray:
        c = self.cfg
        dt = np.float32 if c.dtype == F32 else np.uint16
        out = np.empty((c.slots, 2, c.block_size, c.head_dim), dtype=dt)
        self._check(self.L.okv_read_pool(self.h, layer, req, kv_head, _np_ptr(out)), "okv_read_pool")
        return out

    def read_lengths(self, layer: int) -> np.ndarray:
        out = np.empty(self.cfg.max_requests, np.int32)
        self._check(self.L.okv_read_lengths(self.h, layer, _np_ptr(out)), "okv_read_lengths")
        return out

    def read_local(self, layer: int):
        """(local_used [R][Hkv], local_of [R][Hkv][max_blocks], routes [R][Hkv][Kb])."""
        c = self.cfg
        used = np.empty((c.max_requests, c.kv_heads), np.int32)
        local_of = np.empty((c.max_requests, c.kv_heads, c.max_blocks_per_request), np.int32)
        routes = np.empty((c.max_requests, c.kv_heads, c.slots), np.int32)
        self._check(self.L.okv_read_local(self.h, layer, _np_ptr(used), _np_ptr(local_of), _np_ptr(routes)),
                    "okv_read_local")
        return used, local_of, routes

    def set_timing(self, enable: bool):
        self._check(self.L.okv_set_timing(self.h, 1 if enable else 0), "okv_set_timing")

    def read_timing(self) -> dict:
        t = _Timing()
        self._check(self.L.okv_read_timing(self.h, ctypes.byref(t)), "okv_read_timing")
        return {"ms": {k: t.ms[i] for i, k in enumerate(KERNEL_KINDS)},
                "launches": {k: int(t.launches[i]) for i, k in enumerate(KERNEL_KINDS)},
                "fetched_blocks": int(t.fetched_blocks), "attended_slots": int(t.attended_slots),
                "local_hits": int(t.local_hits), "local_fills": int(t.local_fills),
                "full_reads": int(t.full_reads)}

    def launch_count(self) -> int:
        return int(self.L.okv_launch_count(self.h))

    def close(self):
        if getattr(self, "h", None):
            self.L.okv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def attend_static(pool, slot_block, lengths, q, out, *, q_heads: int, kv_heads: int, head_dim: int,
                  block_size: int, slots: int, dtype: int, stream=None) -> None:
    """okv_attend_static: context-free sparse attention whose only workspace is the library's
    fixed device array (nothing is allocated). Tensors are CUDA, contiguous:
    pool [R][kv_heads][slots][2][block_size][head_dim] (bf16/fp32), slot_block [R][kv_heads][slots]
    int32, lengths [R] int32, q and out [R][q_heads][head_dim]."""
    import torch
    L = load_library()
    R = int(lengths.shape[0])
    want = torch.float32 if dtype == F32 else torch.bfloat16
    for name, t, shape, dt in (("pool", pool, (R, kv_heads, slots, 2, block_size, head_dim), want),
                               ("slot_block", slot_block, (R, kv_heads, slots), torch.int32),
                               ("lengths", lengths, (R,), torch.int32),
                               ("q", q, (R, q_heads, head_dim), want), ("out", out, (R, q_heads, head_dim), want)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name}: expected contiguous CUDA {dt} {shape}, got {t.dtype} {tuple(t.shape)}")
    st = L.okv_attend_static(R, q_heads, kv_heads, head_dim, block_size, slots, dtype,
                             ctypes.c_void_p(pool.data_ptr()), ctypes.c_void_p(slot_block.data_ptr()),
                             ctypes.c_void_p(lengths.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                             ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(_stream_handle(stream)))
    if st != OK:
        raise OkvError(st, "okv_attend_static failed (shape or size outside its limits, or a CUDA error)")
