"""Thin Python binding of libafd (include/afd.h) over ctypes.

Argument marshalling only: tensors become pointers and sizes (CUDA tensors,
or page-locked CPU tensors, which the library reads and writes in place over
the host link; it refuses pageable ones), the current PyTorch stream becomes
the call's stream, and the library's device memory comes back as zero-copy
tensors. Every step of the exchange runs in
the library's CUDA kernels; there is no fallback. If ``libafd.so`` has not
been built, :func:`load_library` raises.

The names follow the afdEP-comm "API contract": ``source_dispatch``,
``worker_receive``, ``worker_reply``, ``source_collect``. On one GPU the
source and worker ranks are index arguments of one :class:`Buffer`.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libafd.so")

OK, ERR_ARG, ERR_STATE, ERR_BUCKET, ERR_RECEIPT = 0, 1, 2, 3, 4
ERR_ROUTE_RANGE, ERR_ROUTE_DUP, ERR_CUDA, ERR_OOM, ERR_CAPTURING, ERR_UNSUPPORTED = 5, 6, 7, 8, 9, 10
ERR_TIMEOUT = 11
BF16, FP8_E4M3 = 0, 1
COMBINE_FUSED, COMBINE_TWO_STAGE, COMBINE_TWO_STAGE_FP8 = 0, 1, 2

EXPORTS = ("afd_create", "afd_destroy", "afd_source_dispatch", "afd_source_dispatch_cached",
           "afd_worker_receive",
           "afd_worker_reply", "afd_source_collect", "afd_source_collect_all", "afd_get_error",
           "afd_clear_error",
           "afd_reset_exchange", "afd_status_string", "afd_error_detail", "afd_arena_rows",
           "afd_recv_rows_for_bucket", "afd_version", "afd_route_layout_noalloc",
           "afd_set_wait_limit", "afd_phase_stamps", "afd_l2_flush")


class AfdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_sources", "num_workers", "num_experts", "top_k", "hidden", "capacity",
        "expert_alignment", "dtype", "num_sms", "combine_mode")]


class Recv(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_void_p), ("row_scales", ctypes.c_void_p),
                ("weights", ctypes.c_void_p), ("row_src", ctypes.c_void_p),
                ("ends", ctypes.c_void_p), ("host_counts", ctypes.c_void_p),
                ("num_rows", ctypes.c_int64), ("receipt", ctypes.c_uint64)]


class View(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("row_stride", ctypes.c_int64),
                ("num_tokens", ctypes.c_int32), ("is_view", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads libafd.so (once). Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise AfdError(ERR_UNSUPPORTED, f"{p} is missing; build it with "
                       "`python -m combine_attention_ffn_gb300.build`")
    lib = ctypes.CDLL(p)
    v, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    P = ctypes.POINTER
    sigs = {
        "afd_create": (i32, [P(Config), i32, P(v)]),
        "afd_destroy": (i32, [v]),
        "afd_source_dispatch": (i32, [v, i32, v, v, v, v, i64, i64, i32, i32, i32, v]),
        "afd_source_dispatch_cached": (i32, [v, i32, v, v, v, i64, i64, i32, i32, i32, v]),
        "afd_worker_receive": (i32, [v, i32, i32, i32, v, P(Recv)]),
        "afd_worker_reply": (i32, [v, i32, v, i64, u64, v]),
        "afd_source_collect": (i32, [v, i32, v, i32, v, P(View)]),
        "afd_source_collect_all": (i32, [v, v, i32, v, v]),
        "afd_get_error": (i32, [v, P(i32), P(i32), P(i32), P(i32)]),
        "afd_clear_error": (i32, [v, v]),
        "afd_reset_exchange": (i32, [v]),
        "afd_status_string": (ctypes.c_char_p, [i32]),
        "afd_error_detail": (ctypes.c_char_p, [v]),
        "afd_arena_rows": (i64, [v]),
        "afd_recv_rows_for_bucket": (i64, [v, i32]),
        "afd_version": (i32, []),
        "afd_route_layout_noalloc": (i32, [v, i32, i32, i32, i32, i32, v, v, v, v]),
        "afd_set_wait_limit": (i32, [v, i32]),
        "afd_phase_stamps": (i32, [v, P(u64), i64, i32]),
        "afd_l2_flush": (i32, [v, i64, v]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if path is None:
        _lib = lib
    return lib


def use_library(path: str) -> ctypes.CDLL:
    """Makes the library at `path` (e.g. the phase-timer build) the one every
    Buffer created afterwards calls."""
    global _lib
    _lib = load_library(path)
    return _lib


# afd_phase_stamps: [kind][block][point] (afd.h)
STAMP_KINDS = ("dispatch", "scatter", "combine", "combine-early")
STAMP_SHAPE = (4, 4096, 8)


class _Context:
    """Owns one afd_ctx. It is destroyed when the Buffer is closed and no
    tensor that views the context's memory is alive any more, so a view can
    never outlive the memory it points at."""

    def __init__(self, lib, handle: ctypes.c_void_p):
        self.lib = lib
        self.handle = handle

    def __del__(self):
        try:
            if self.handle is not None and self.handle.value:
                self.lib.afd_destroy(self.handle)
                self.handle = None
        except Exception:
            pass


class _DeviceArray:
    """Exposes library-owned device memory through __cuda_array_interface__;
    the tensor made from it keeps the owning context alive."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self.__cuda_array_interface__ = {"shape": tuple(int(s) for s in shape), "typestr": typestr,
                                         "data": (int(ptr or 0), False), "version": 2,
                                         "strides": None}
        self._owner = owner


def _wrap(ptr, shape, dtype: torch.dtype, owner, device) -> torch.Tensor:
    base = {torch.int32: "<i4", torch.float32: "<f4", torch.bfloat16: "<i2",
            torch.float8_e4m3fn: "|u1", torch.uint8: "|u1"}[dtype]
    t = torch.as_tensor(_DeviceArray(ptr, shape, base, owner), device=device)
    if dtype == torch.bfloat16:
        t = t.view(torch.bfloat16)
    elif dtype == torch.float8_e4m3fn:
        t = t.view(torch.float8_e4m3fn)
    return t


def _stream_handle(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device.index)
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


@dataclass
class Receive:
    """One worker's received rows (zero-copy views of the context's arena)."""
    rows: torch.Tensor                 # [num_rows, H] bf16 or float8_e4m3fn
    row_scales: Optional[torch.Tensor]  # [num_rows, H/128] f32 (FP8)
    weights: torch.Tensor              # [num_rows] f32
    row_src: torch.Tensor              # [num_rows] i32
    ends: torch.Tensor                 # [E/F] i32 on the device
    host_counts: Optional[np.ndarray]  # [E/F] aligned counts (read_host_counts)
    num_rows: int
    receipt: int


class Buffer:
    """One context: A sources and F workers exchanging through this GPU's HBM."""

    def __init__(self, num_sources: int, num_workers: int, num_experts: int, top_k: int,
                 hidden: int, capacity: int, expert_alignment: int = 1, dtype: str = "bf16",
                 num_sms: int = 0, device=None, combine_mode: int = COMBINE_FUSED):
        self._lib = load_library()
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        self.cfg = Config(num_sources, num_workers, num_experts, top_k, hidden, capacity,
                          expert_alignment, FP8_E4M3 if dtype == "fp8" else BF16, num_sms,
                          combine_mode)
        self.dtype = dtype
        self.A, self.F, self.E, self.K, self.H = num_sources, num_workers, num_experts, top_k, hidden
        self.Ef = num_experts // max(num_workers, 1)
        self.capacity, self.alpha = capacity, expert_alignment
        h = ctypes.c_void_p()
        st = self._lib.afd_create(ctypes.byref(self.cfg), self.device.index, ctypes.byref(h))
        if st != OK:
            raise AfdError(st, "afd_create: " + self._lib.afd_status_string(st).decode())
        self._ctx = _Context(self._lib, h)
        self._h = h
        self._views = {}

    # the dtype the top-k IDs must have ("API contract": buffer.topk_idx_dtype)
    topk_idx_dtype = torch.int64

    # -- helpers ------------------------------------------------------------
    def _check(self, st: int, what: str):
        if st != OK:
            detail = self._lib.afd_error_detail(self._h).decode() if self._h else ""
            raise AfdError(st, f"{what}: {self._lib.afd_status_string(st).decode()}: {detail}")

    def _view(self, ptr, shape, dtype: torch.dtype) -> torch.Tensor:
        """A tensor over context-owned memory. The arenas never move, so the
        tensors are made once per (address, shape, dtype) and reused."""
        key = (int(ptr or 0), tuple(shape), dtype)
        t = self._views.get(key)
        if t is None:
            if len(self._views) >= 256:  # exact receive shapes vary with read_host_counts
                self._views.clear()
            t = _wrap(ptr, shape, dtype, self._ctx, self.device)
            self._views[key] = t
        return t

    @property
    def handle(self) -> int:
        return int(self._h.value or 0)

    def arena_rows(self) -> int:
        return int(self._lib.afd_arena_rows(self._h))

    def recv_rows_for_bucket(self, bucket: int) -> int:
        return int(self._lib.afd_recv_rows_for_bucket(self._h, bucket))

    # -- the four calls -------------------------------------------------------
    def source_dispatch(self, source: int, x: torch.Tensor, ids: torch.Tensor,
                        weights: torch.Tensor, x_scale: Optional[torch.Tensor] = None, *,
                        bucket: int, read_host_counts: bool = False, stream=None) -> None:
        T = int(x.shape[0]) if x is not None else 0
        if T:
            want = torch.float8_e4m3fn if self.dtype == "fp8" else torch.bfloat16
            if x.dtype != want or tuple(x.shape) != (T, self.H) or not x.is_contiguous():
                raise AfdError(ERR_ARG, f"x must be contiguous {want} [T, {self.H}]")
            if ids.dtype != torch.int64 or tuple(ids.shape) != (T, self.K) or not ids.is_contiguous():
                raise AfdError(ERR_ARG, f"ids must be contiguous int64 [T, {self.K}]")
            if weights.dtype != torch.float32 or tuple(weights.shape) != (T, self.K) \
                    or not weights.is_contiguous():
                raise AfdError(ERR_ARG, f"weights must be contiguous float32 [T, {self.K}]")
        sst = ssb = 0
        if x_scale is not None:
            if x_scale.dtype != torch.float32 or tuple(x_scale.shape) != (T, self.H // 128):
                raise AfdError(ERR_ARG, f"x_scale must be float32 [T, {self.H // 128}]")
            sst, ssb = x_scale.stride()
        st = self._lib.afd_source_dispatch(self._h, source, _ptr(x) if T else None,
                                           _ptr(ids) if T else None, _ptr(weights) if T else None,
                                           _ptr(x_scale) if T else None, sst, ssb, T, bucket,
                                           int(bool(read_host_counts)),
                                           _stream_handle(stream, self.device))
        self._check(st, "source_dispatch")

    def source_dispatch_cached(self, source: int, x: torch.Tensor, weights: Optional[torch.Tensor] = None,
                               x_scale: Optional[torch.Tensor] = None, *, bucket: int,
                               read_host_counts: bool = False, stream=None) -> None:
        """Dispatch with the routing (IDs, layout, receipts) of the last exchange;
        only the rows move. `weights` replaces the routing weights of the same
        IDs, or None keeps them."""
        T = int(x.shape[0]) if x is not None else 0
        if T:
            want = torch.float8_e4m3fn if self.dtype == "fp8" else torch.bfloat16
            if x.dtype != want or tuple(x.shape) != (T, self.H) or not x.is_contiguous():
                raise AfdError(ERR_ARG, f"x must be contiguous {want} [T, {self.H}]")
            if weights is not None and (weights.dtype != torch.float32 or
                                        tuple(weights.shape) != (T, self.K) or not weights.is_contiguous()):
                raise AfdError(ERR_ARG, f"weights must be contiguous float32 [T, {self.K}]")
        sst = ssb = 0
        if x_scale is not None:
            if x_scale.dtype != torch.float32 or tuple(x_scale.shape) != (T, self.H // 128):
                raise AfdError(ERR_ARG, f"x_scale must be float32 [T, {self.H // 128}]")
            sst, ssb = x_scale.stride()
        st = self._lib.afd_source_dispatch_cached(self._h, source, _ptr(x) if T else None,
                                                  _ptr(weights) if T else None,
                                                  _ptr(x_scale) if T else None, sst, ssb, T, bucket,
                                                  int(bool(read_host_counts)),
                                                  _stream_handle(stream, self.device))
        self._check(st, "source_dispatch_cached")

    def worker_receive(self, worker: int, *, bucket: int, read_host_counts: bool = False,
                       stream=None) -> Receive:
        r = Recv()
        st = self._lib.afd_worker_receive(self._h, worker, bucket, int(bool(read_host_counts)),
                                          _stream_handle(stream, self.device), ctypes.byref(r))
        self._check(st, "worker_receive")
        n = int(r.num_rows)
        rows_dtype = torch.float8_e4m3fn if self.dtype == "fp8" else torch.bfloat16
        hc = None
        if r.host_counts:
            hc = np.ctypeslib.as_array(ctypes.cast(r.host_counts, ctypes.POINTER(ctypes.c_int32)),
                                       shape=(self.Ef,)).copy()
        return Receive(
            rows=self._view(r.rows, (n, self.H), rows_dtype),
            row_scales=self._view(r.row_scales, (n, self.H // 128), torch.float32) if r.row_scales else None,
            weights=self._view(r.weights, (n,), torch.float32),
            row_src=self._view(r.row_src, (n,), torch.int32),
            ends=self._view(r.ends, (self.Ef,), torch.int32),
            host_counts=hc, num_rows=n, receipt=int(r.receipt))

    def worker_reply(self, worker: int, rows: torch.Tensor, receipt: int, stream=None) -> None:
        if rows.dtype != torch.bfloat16 or rows.dim() != 2 or rows.shape[1] != self.H \
                or not rows.is_contiguous():
            raise AfdError(ERR_ARG, f"reply rows must be contiguous bfloat16 [rows, {self.H}]")
        st = self._lib.afd_worker_reply(self._h, worker, _ptr(rows), int(rows.shape[0]),
                                        ctypes.c_uint64(receipt), _stream_handle(stream, self.device))
        self._check(st, "worker_reply")

    def source_collect(self, source: int, *, view: bool = False, out: Optional[torch.Tensor] = None,
                       num_tokens: Optional[int] = None, stream=None) -> torch.Tensor:
        """BF16 [T, H]. With view=True and one worker, a read-only view of the
        context's inbox (valid until the next source_dispatch)."""
        v = View()
        if out is None and not (view and self.F == 1):
            if num_tokens is None:
                raise AfdError(ERR_ARG, "pass out= or num_tokens=")
            out = torch.empty((num_tokens, self.H), dtype=torch.bfloat16, device=self.device)
        st = self._lib.afd_source_collect(self._h, source, _ptr(out), int(bool(view)),
                                          _stream_handle(stream, self.device), ctypes.byref(v))
        self._check(st, "source_collect")
        if v.is_view:
            return self._view(v.data, (int(v.num_tokens), int(v.row_stride)), torch.bfloat16)[:, : self.H]
        return out

    def source_collect_all(self, *, view: bool = False, outs=None, num_tokens=None, stream=None):
        """Every source's result with one call (one combine launch).
        Returns a list of BF16 [T_s, H] tensors (views with view=True and F == 1)."""
        if outs is None:
            if view and self.F == 1:
                outs = [None] * self.A
            else:
                if num_tokens is None:
                    raise AfdError(ERR_ARG, "pass outs= or num_tokens=")
                outs = [torch.empty((t, self.H), dtype=torch.bfloat16, device=self.device)
                        for t in num_tokens]
        ptrs = (ctypes.c_void_p * self.A)(*[_ptr(o) if o is not None else None for o in outs])
        views = (View * self.A)()
        st = self._lib.afd_source_collect_all(self._h, ptrs, int(bool(view)),
                                              _stream_handle(stream, self.device), views)
        self._check(st, "source_collect_all")
        res = []
        for s in range(self.A):
            v = views[s]
            if v.is_view:
                res.append(self._view(v.data, (int(v.num_tokens), int(v.row_stride)), torch.bfloat16)[:, : self.H])
            else:
                res.append(outs[s])
        return res

    # -- errors and lifetime ---------------------------------------------------
    def get_error(self):
        c, s, t, k = (ctypes.c_int32() for _ in range(4))
        st = self._lib.afd_get_error(self._h, ctypes.byref(c), ctypes.byref(s), ctypes.byref(t),
                                     ctypes.byref(k))
        self._check(st, "get_error")
        return c.value, s.value, t.value, k.value

    def clear_error(self, stream=None) -> None:
        self._check(self._lib.afd_clear_error(self._h, _stream_handle(stream, self.device)),
                    "clear_error")

    def reset_exchange(self) -> None:
        self._check(self._lib.afd_reset_exchange(self._h), "reset_exchange")

    def phase_stamps(self, clear: bool = False) -> np.ndarray:
        """The phase-timer build's %globaltimer stamps, uint64 STAMP_SHAPE
        (afd_phase_stamps); synchronizes the device. Raises AfdError with
        ERR_UNSUPPORTED on the default build."""
        out = np.zeros(STAMP_SHAPE, dtype=np.uint64)
        st = self._lib.afd_phase_stamps(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                        out.size, int(bool(clear)))
        self._check(st, "phase_stamps")
        return out

    def set_wait_limit(self, polls: int) -> None:
        """Polls of each bulk row load before the scatter reports AFD_ERR_TIMEOUT
        (afd_set_wait_limit; 0 makes every first wait give up at once)."""
        self._check(self._lib.afd_set_wait_limit(self._h, polls), "set_wait_limit")

    def __enter__(self) -> "Buffer":
        return self

    def __exit__(self, *exc) -> None:
        self.close()

    def close(self) -> None:
        """Releases the context. Its memory is freed (after the device work
        completes) once no tensor viewing it is alive."""
        self._views = {}
        self._ctx = None
        self._h = ctypes.c_void_p()


def route_layout_noalloc(ids: torch.Tensor, num_experts: int, num_workers: int,
                         expert_alignment: int, ends: torch.Tensor, slots: torch.Tensor,
                         error: torch.Tensor, stream=None) -> None:
    """Routing layout into caller-provided outputs; the library allocates
    nothing (its scratch is a fixed device array). See
    afd_route_layout_noalloc in include/afd.h for the limits and rules."""
    lib = load_library()
    T, K = (int(ids.shape[0]), int(ids.shape[1])) if ids.dim() == 2 else (0, 1)
    for name, t, dt in (("ends", ends, torch.int32), ("slots", slots, torch.int32),
                        ("error", error, torch.int32), ("ids", ids, torch.int64)):
        if t.dtype != dt or not t.is_contiguous():
            raise AfdError(ERR_ARG, f"{name} must be contiguous {dt}")
    st = lib.afd_route_layout_noalloc(_ptr(ids) if T else None, T, K, num_experts, num_workers,
                                      expert_alignment, _ptr(ends), _ptr(slots) if T else None,
                                      _ptr(error), _stream_handle(stream, ids.device))
    if st != OK:
        raise AfdError(st, "afd_route_layout_noalloc: " + lib.afd_status_string(st).decode())
