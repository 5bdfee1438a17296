"""CPU oracle for the Attention -> FFN MoE dispatch and combine.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The library never
does, and this package shares no code with it: the arithmetic lives in
``orc.c`` (plain sequential C, built with ``-ffp-contract=off``), and this
module only marshals numpy arrays into it.

What each function follows (afdEP-comm pages):

* ``validate``  -- "API contract", Roles and tensors: IDs unique per token,
  in [0, E) or -1 to skip; anything else is an invalid route.
* ``layout``    -- "API contract", Roles and tensors: the receive prefix sum
  ``ends[]``, expert e in [align_up(ends[e-1], alpha), ends[e]), aligned host
  counts.
* ``dispatch``  -- "DeepEP V2 ElasticBuffer first principles", section 3:
  one slot per valid route in expert-major order, rows copied byte for byte
  (section 7: FP8 rows travel with their block scales).
* ``combine``   -- "API contract" (source_collect: BF16 [T,H], summed over the
  selected experts in token order, weight applied once) and design page
  section 19 (FP32 sum in slot order, one rounding to BF16).
* ``combine_two_stage`` -- design page sections 6 and 19: per-worker BF16
  partials (optionally E4M3 with one power-of-two factor shared by each block of 128 values),
  summed in FP32 in the order of each worker's last route, rounded once.

Parity pins for each of these live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orc.c")
_HDR = os.path.join(_HERE, "orc.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liborc.so")

ROUTE_OK, ROUTE_RANGE, ROUTE_DUP = 0, 1, 2
BF16, FP8 = 0, 1
EXPERT_IDENTITY, EXPERT_SCALE = 0, 1

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``orc.c`` into a shared object (gcc, no GPU needed)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = (not os.path.exists(out)
             or os.path.getmtime(out) < max(os.path.getmtime(src), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, "-I", _HERE, src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)
    return out


class _Problem(ctypes.Structure):
    _fields_ = [("A", ctypes.c_int32), ("F", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("H", ctypes.c_int32), ("alpha", ctypes.c_int32),
                ("bucket", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("T", ctypes.POINTER(ctypes.c_int32))]


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes handle on one compiled copy of ``orc.c``."""

    def __init__(self, lib_path: Optional[str] = None):
        self.lib = ctypes.CDLL(lib_path or build())
        P = ctypes.POINTER(_Problem)
        v, i64 = ctypes.c_void_p, ctypes.c_int64
        sig = {
            "orc_bf16_to_float_n": [v, v, i64],
            "orc_float_to_bf16_n": [v, v, i64],
            "orc_e4m3_to_float_n": [v, v, i64],
            "orc_validate": [P, v, v, v, v],
            "orc_layout": [P, v, v, v, v, v, v],
            "orc_dispatch": [P, v, v, v, v, v, v, i64, v, v, v, v, v],
            "orc_expert": [P, ctypes.c_int32, v, v, i64, v, v, v],
            "orc_combine": [P, v, v, v, i64, v, v],
            "orc_float_to_e4m3_n": [v, v, i64],
            "orc_group_exponent_n": [v, v, i64],
            "orc_combine_two_stage": [P, v, v, v, i64, v, ctypes.c_int32, v],
        }
        for name, args in sig.items():
            fn = getattr(self.lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int32 if name == "orc_validate" else None

    # -- number formats -------------------------------------------------
    def bf16_to_float(self, b: np.ndarray) -> np.ndarray:
        b = np.ascontiguousarray(b, dtype=np.uint16)
        out = np.empty(b.shape, np.float32)
        self.lib.orc_bf16_to_float_n(_ptr(b), _ptr(out), b.size)
        return out

    def float_to_bf16(self, f: np.ndarray) -> np.ndarray:
        f = np.ascontiguousarray(f, dtype=np.float32)
        out = np.empty(f.shape, np.uint16)
        self.lib.orc_float_to_bf16_n(_ptr(f), _ptr(out), f.size)
        return out

    def float_to_e4m3(self, f: np.ndarray) -> np.ndarray:
        f = np.ascontiguousarray(f, dtype=np.float32)
        out = np.empty(f.shape, np.uint8)
        self.lib.orc_float_to_e4m3_n(_ptr(f), _ptr(out), f.size)
        return out

    def group_exponent(self, amax: np.ndarray) -> np.ndarray:
        amax = np.ascontiguousarray(amax, dtype=np.float32)
        out = np.empty(amax.shape, np.int32)
        self.lib.orc_group_exponent_n(_ptr(amax), _ptr(out), amax.size)
        return out

    def e4m3_to_float(self, q: np.ndarray) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.uint8)
        out = np.empty(q.shape, np.float32)
        self.lib.orc_e4m3_to_float_n(_ptr(q), _ptr(out), q.size)
        return out


@dataclass
class Problem:
    """One exchange's shape. Arrays are padded to ``bucket`` tokens per source."""
    A: int
    F: int
    E: int
    K: int
    H: int
    alpha: int
    bucket: int
    dtype: int
    T: Sequence[int]

    @property
    def Ef(self) -> int:
        return self.E // self.F

    @property
    def row_bytes(self) -> int:
        return self.H if self.dtype == FP8 else 2 * self.H

    def _c(self):
        self._T = np.ascontiguousarray(np.asarray(self.T, dtype=np.int32))
        return _Problem(self.A, self.F, self.E, self.K, self.H, self.alpha, self.bucket,
                        self.dtype, self._T.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))


_default: Optional[Oracle] = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def validate(p: Problem, ids: np.ndarray, orc: Optional[Oracle] = None):
    """First invalid route as (code, s, t, k); code 0 when all routes are valid."""
    orc = orc or get()
    ids = np.ascontiguousarray(ids, np.int64)
    es, et, ek = (np.zeros(1, np.int32) for _ in range(3))
    pc = p._c()
    code = orc.lib.orc_validate(ctypes.byref(pc), _ptr(ids), _ptr(es), _ptr(et), _ptr(ek))
    return int(code), int(es[0]), int(et[0]), int(ek[0])


def layout(p: Problem, ids: np.ndarray, orc: Optional[Oracle] = None) -> dict:
    """Per-expert counts, aligned starts, ends[], host counts ([F, E/F]) and exact rows."""
    orc = orc or get()
    ids = np.ascontiguousarray(ids, np.int64)
    count, start, ends, hc = (np.zeros((p.F, p.Ef), np.int32) for _ in range(4))
    r_exact = np.zeros(p.F, np.int64)
    pc = p._c()
    orc.lib.orc_layout(ctypes.byref(pc), _ptr(ids), _ptr(count), _ptr(start), _ptr(ends),
                       _ptr(hc), _ptr(r_exact))
    return dict(count=count, start=start, ends=ends, host_counts=hc, r_exact=r_exact)


def dispatch(p: Problem, ids, w, x, x_scales, lay: dict, r_stride: int,
             orc: Optional[Oracle] = None) -> dict:
    """Slot map, receipts and expert-major rows (see ``orc_dispatch``)."""
    orc = orc or get()
    ids = np.ascontiguousarray(ids, np.int64)
    w = np.ascontiguousarray(w, np.float32)
    xb = np.ascontiguousarray(x).view(np.uint8)
    nb = p.H // 128
    slot = np.zeros((p.A, p.bucket, p.K), np.int32)
    row_src = np.full((p.F, r_stride), -2, np.int32)
    row_w = np.full((p.F, r_stride), np.nan, np.float32)
    rows = np.zeros((p.F, r_stride, p.row_bytes), np.uint8)
    row_scales = np.zeros((p.F, r_stride, nb), np.float32) if p.dtype == FP8 else None
    xs = np.ascontiguousarray(x_scales, np.float32) if p.dtype == FP8 else None
    pc = p._c()
    orc.lib.orc_dispatch(ctypes.byref(pc), _ptr(ids), _ptr(w), _ptr(xb), _ptr(xs),
                         _ptr(np.ascontiguousarray(lay["start"])),
                         _ptr(np.ascontiguousarray(lay["r_exact"])), r_stride, _ptr(slot),
                         _ptr(row_src), _ptr(row_w), _ptr(rows), _ptr(row_scales))
    return dict(slot=slot, row_src=row_src, row_w=row_w, rows=rows, row_scales=row_scales)


def expert(p: Problem, mode: int, lay: dict, r_stride: int, rows: np.ndarray,
           row_scales: Optional[np.ndarray], orc: Optional[Oracle] = None) -> np.ndarray:
    """Stand-in FFN expert: BF16 replies [F, r_stride, H] (zeros outside live rows)."""
    orc = orc or get()
    reply = np.zeros((p.F, r_stride, p.H), np.uint16)
    pc = p._c()
    orc.lib.orc_expert(ctypes.byref(pc), mode, _ptr(np.ascontiguousarray(lay["start"])),
                       _ptr(np.ascontiguousarray(lay["ends"])), r_stride,
                       _ptr(np.ascontiguousarray(rows)),
                       _ptr(None if row_scales is None else np.ascontiguousarray(row_scales)),
                       _ptr(reply))
    return reply


def combine(p: Problem, ids, w, slot, r_stride: int, reply: np.ndarray,
            orc: Optional[Oracle] = None) -> np.ndarray:
    """BF16 bits [A, bucket, H]; rows t >= T[s] stay zero."""
    orc = orc or get()
    out = np.zeros((p.A, p.bucket, p.H), np.uint16)
    pc = p._c()
    orc.lib.orc_combine(ctypes.byref(pc), _ptr(np.ascontiguousarray(ids, np.int64)),
                        _ptr(np.ascontiguousarray(w, np.float32)),
                        _ptr(np.ascontiguousarray(slot)), r_stride,
                        _ptr(np.ascontiguousarray(reply)), _ptr(out))
    return out


COMBINE_FUSED, COMBINE_TWO_STAGE, COMBINE_TWO_STAGE_FP8 = 0, 1, 2


def combine_two_stage(p: Problem, ids, w, slot, r_stride: int, reply: np.ndarray, fp8: bool,
                      orc: Optional[Oracle] = None) -> np.ndarray:
    """Two-stage combine (per-worker BF16 partials, optionally FP8) -> BF16 bits."""
    orc = orc or get()
    out = np.zeros((p.A, p.bucket, p.H), np.uint16)
    pc = p._c()
    orc.lib.orc_combine_two_stage(ctypes.byref(pc), _ptr(np.ascontiguousarray(ids, np.int64)),
                                  _ptr(np.ascontiguousarray(w, np.float32)),
                                  _ptr(np.ascontiguousarray(slot)), r_stride,
                                  _ptr(np.ascontiguousarray(reply)), int(bool(fp8)), _ptr(out))
    return out


def round_trip(p: Problem, ids, w, x, x_scales=None, expert_mode: int = EXPERT_IDENTITY,
               orc: Optional[Oracle] = None, combine_mode: int = COMBINE_FUSED) -> dict:
    """validate -> layout -> dispatch -> expert -> combine, all on the CPU."""
    orc = orc or get()
    err = validate(p, ids, orc)
    lay = layout(p, ids, orc)
    r_stride = max(1, int(lay["r_exact"].max()))
    d = dispatch(p, ids, w, x, x_scales, lay, r_stride, orc)
    reply = expert(p, expert_mode, lay, r_stride, d["rows"], d["row_scales"], orc)
    if combine_mode == COMBINE_FUSED:
        out = combine(p, ids, w, d["slot"], r_stride, reply, orc)
    else:
        out = combine_two_stage(p, ids, w, d["slot"], r_stride, reply,
                                combine_mode == COMBINE_TWO_STAGE_FP8, orc)
    return dict(err=err, r_stride=r_stride, reply=reply, out=out, **lay, **d)
