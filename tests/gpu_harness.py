"""Runs one exchange through the library and checks it against the oracle.

Used by the GPU parity tests. The stand-in expert here (PyTorch ops on the
GPU) is harness, not library: it turns received rows into BF16 replies the
same way the oracle's stand-in does (reply = bf16(value * c_e), c_e =
2^((e mod 4) - 1)), independently of the oracle's code.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
from combine_attention_ffn_gb300 import afd
from combine_attention_ffn_gb300 import workloads as W

IDENTITY, SCALE = oracle.EXPERT_IDENTITY, oracle.EXPERT_SCALE


def make_buffer(wl: W.Workload, num_sms: int = 0, combine_mode: int = 0) -> afd.Buffer:
    return afd.Buffer(wl.A, wl.F, wl.E, wl.K, wl.H, wl.capacity, wl.alpha, wl.dtype, num_sms,
                      combine_mode=combine_mode)


@dataclass
class DeviceInputs:
    x: List[torch.Tensor]
    ids: List[torch.Tensor]
    w: List[torch.Tensor]
    scales: List[Optional[torch.Tensor]]


def to_device(inp: W.Inputs, transposed_scales: bool = False, device="cuda") -> DeviceInputs:
    wl = inp.wl
    xs, ids, ws, scs = [], [], [], []
    for s, T in enumerate(wl.T):
        if wl.dtype == "fp8":
            x = torch.from_numpy(inp.x[s, :T].copy()).to(device).view(torch.float8_e4m3fn)
            sc = torch.from_numpy(inp.x_scales[s, :T].copy()).to(device)
            if transposed_scales:
                # a strided [T, H/128] view of a [H/128, T] tensor
                sc = sc.t().contiguous().t()
            scs.append(sc)
        else:
            x = torch.from_numpy(inp.x[s, :T].view(np.int16).copy()).to(device).view(torch.bfloat16)
            scs.append(None)
        xs.append(x.contiguous())
        ids.append(torch.from_numpy(inp.ids[s, :T].copy()).to(device))
        ws.append(torch.from_numpy(inp.w[s, :T].copy()).to(device))
    return DeviceInputs(xs, ids, ws, scs)


def refresh_device(dev: DeviceInputs, inp: W.Inputs) -> None:
    """Copies new input values into the captured tensors in place."""
    wl = inp.wl
    for s, T in enumerate(wl.T):
        if T == 0:
            continue
        if wl.dtype == "fp8":
            dev.x[s].view(torch.uint8).copy_(torch.from_numpy(inp.x[s, :T].copy()))
            dev.scales[s].copy_(torch.from_numpy(inp.x_scales[s, :T].copy()))
        else:
            dev.x[s].view(torch.int16).copy_(torch.from_numpy(inp.x[s, :T].view(np.int16).copy()))
        dev.ids[s].copy_(torch.from_numpy(inp.ids[s, :T].copy()))
        dev.w[s].copy_(torch.from_numpy(inp.w[s, :T].copy()))


def expert_reply(wl: W.Workload, worker: int, recv: afd.Receive, mode: int) -> torch.Tensor:
    """Stand-in expert on the GPU (harness only, no host synchronization so
    that it can sit inside a captured graph)."""
    if mode == IDENTITY and wl.dtype == "bf16":
        return recv.rows
    dev = recv.rows.device
    ends = recv.ends.to(torch.int64)
    prev = torch.cat([torch.zeros(1, dtype=torch.int64, device=dev), ends[:-1]])
    starts = (prev + wl.alpha - 1) // wl.alpha * wl.alpha
    r = torch.arange(recv.num_rows, device=dev, dtype=torch.int64)
    l = (torch.searchsorted(starts, r, right=True) - 1).clamp(min=0)
    live = r < ends[l]
    e = worker * wl.Ef + l
    c = torch.pow(2.0, (e % 4 - 1).to(torch.float32)) if mode == SCALE else torch.ones_like(r, dtype=torch.float32)
    factor = torch.where(live, c, torch.zeros_like(c))[:, None]
    if wl.dtype == "fp8":
        sc = recv.row_scales.repeat_interleave(128, dim=1)
        v = recv.rows.float() * sc
        v = torch.where(live[:, None], v, torch.zeros_like(v))
        return (v * factor).to(torch.bfloat16).contiguous()
    return (recv.rows.float() * factor).to(torch.bfloat16).contiguous()


def alloc_outs(wl: W.Workload, device="cuda") -> List[torch.Tensor]:
    return [torch.empty((T, wl.H), dtype=torch.bfloat16, device=device) for T in wl.T]


def run_exchange(buf: afd.Buffer, wl: W.Workload, dev: DeviceInputs, mode: int = SCALE,
                 rhc: bool = False, view: bool = False, outs=None, keep_recv: bool = True,
                 bucket: Optional[int] = None, source_order=None, worker_order=None):
    bucket = wl.bucket if bucket is None else bucket
    for s in (source_order or range(wl.A)):
        buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], dev.scales[s], bucket=bucket,
                            read_host_counts=rhc)
    recvs = {}
    for f in (worker_order or range(wl.F)):
        r = buf.worker_receive(f, bucket=bucket, read_host_counts=rhc)
        recvs[f] = r
    replies = {}
    for f in (worker_order or range(wl.F)):
        replies[f] = expert_reply(wl, f, recvs[f], mode)
        buf.worker_reply(f, replies[f], recvs[f].receipt)
    outs = outs if outs is not None else alloc_outs(wl)
    results = []
    for s in range(wl.A):
        results.append(buf.source_collect(s, view=view, out=None if view and wl.F == 1 else outs[s]))
    return recvs, replies, results


def snapshot(recvs) -> dict:
    """Copies each worker's receive to host numpy (before the next exchange)."""
    snap = {}
    for f, r in recvs.items():
        snap[f] = dict(
            ends=r.ends.cpu().numpy().copy(),
            row_src=r.row_src.cpu().numpy().copy(),
            weights=r.weights.cpu().numpy().copy(),
            rows=r.rows.view(torch.uint8).cpu().numpy().copy(),
            row_scales=None if r.row_scales is None else r.row_scales.cpu().numpy().copy(),
            host_counts=None if r.host_counts is None else r.host_counts.copy(),
            num_rows=r.num_rows)
    return snap


def expected(inp: W.Inputs, mode: int, combine_mode: int = 0) -> dict:
    wl = inp.wl
    p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket,
                       oracle.FP8 if wl.dtype == "fp8" else oracle.BF16, list(wl.T))
    r = oracle.round_trip(p, inp.ids, inp.w, inp.x, inp.x_scales, expert_mode=mode,
                          combine_mode=combine_mode)
    return r


def out_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_layout(wl: W.Workload, snap: dict, exp: dict, rhc: bool, buf: afd.Buffer) -> None:
    row_bytes = wl.row_bytes
    for f in range(wl.F):
        g = snap[f]
        assert np.array_equal(g["ends"], exp["ends"][f]), f"ends, worker {f}"
        R = int(exp["r_exact"][f])
        if rhc:
            assert g["num_rows"] == R
            assert np.array_equal(g["host_counts"], exp["host_counts"][f])
        else:
            assert g["num_rows"] == buf.recv_rows_for_bucket(wl.bucket)
            assert g["num_rows"] >= R
        assert np.array_equal(g["row_src"][:R], exp["row_src"][f, :R]), f"row_src, worker {f}"
        assert np.array_equal(g["weights"][:R].view(np.uint32),
                              exp["row_w"][f, :R].view(np.uint32)), f"row weights, worker {f}"
        live = exp["row_src"][f, :R] >= 0
        got_rows = g["rows"].reshape(g["num_rows"], row_bytes)[:R]
        assert np.array_equal(got_rows[live], exp["rows"][f, :R][live]), f"row bytes, worker {f}"
        if wl.dtype == "fp8":
            gs = g["row_scales"][:R]
            assert np.array_equal(gs[live].view(np.uint32),
                                  exp["row_scales"][f, :R][live].view(np.uint32))


def ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in BF16 units in the last place between two bit arrays."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))


def check_outputs(wl: W.Workload, results, exp: dict) -> None:
    for s in range(wl.A):
        T = wl.T[s]
        got = out_bits(results[s]) if T else np.zeros((0, wl.H), np.uint16)
        want = exp["out"][s, :T]
        assert got.shape == want.shape
        if not np.array_equal(got, want):
            d = ulp_diff(got, want)
            raise AssertionError(f"source {s}: {(d > 0).sum()} of {d.size} elements differ, "
                                 f"max {d.max()} ulp")
