"""The allocation-free routing layout (afd_route_layout_noalloc) against the
ordinary dispatch path.

Callers that cannot call cudaMalloc (inside another framework's memory pool or
allocator hook, or with device memory fully reserved up front) use this entry
point; its scratch is a fixed device array in the library. Its ends[] must
equal what afd_worker_receive reports for the same routing, and every route's
row must be the one whose receipt (row_src) names that route. Checked on two
calls in a row, since the calls share the scratch array. This file is
collected last so that a run stopping at the first failure has run every other
test first.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_attention_ffn_gb300 import afd
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _reference(wl, ids_dev):
    """ends and row_src from the ordinary dispatch of one source's routing."""
    buf = afd.Buffer(1, wl.F, wl.E, wl.K, wl.H, wl.capacity, wl.alpha)
    try:
        T = wl.T[0]
        x = torch.zeros((T, wl.H), dtype=torch.bfloat16, device="cuda")
        w = torch.ones((T, wl.K), dtype=torch.float32, device="cuda")
        buf.source_dispatch(0, x, ids_dev, w, bucket=T, read_host_counts=True)
        ends, row_src = [], []
        for f in range(wl.F):
            r = buf.worker_receive(f, bucket=T, read_host_counts=True)
            ends.append(r.ends.cpu().numpy().copy())
            row_src.append(r.row_src.cpu().numpy().copy())
            buf.worker_reply(f, torch.zeros((r.num_rows, wl.H), dtype=torch.bfloat16, device="cuda"),
                             r.receipt)
        torch.cuda.synchronize()
        buf.reset_exchange()
        return np.concatenate(ends), row_src
    finally:
        buf.close()


def _call_c_abi(ids_dev, E, F, alpha):
    """Calls the entry point through the C ABI with raw device pointers."""
    lib = afd.load_library()
    T, K = ids_dev.shape
    ends = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    slots = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    err = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    st = lib.afd_route_layout_noalloc(
        ctypes.c_void_p(ids_dev.data_ptr()), T, K, E, F, alpha, ctypes.c_void_p(ends.data_ptr()),
        ctypes.c_void_p(slots.data_ptr()), ctypes.c_void_p(err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == afd.OK
    torch.cuda.synchronize()
    return ends.cpu().numpy(), slots.cpu().numpy(), err.cpu().numpy()


def _check(wl, ids_np, ends, slots, err, ref_ends, ref_row_src):
    assert err.tolist() == [0, -1, -1]
    assert np.array_equal(ends, ref_ends)
    Ef = wl.E // wl.F
    T, K = ids_np.shape
    for t in range(T):
        for k in range(K):
            e = int(ids_np[t, k])
            if e < 0:
                assert slots[t, k] == -1
                continue
            f = e // Ef
            assert ref_row_src[f][slots[t, k]] == t * K + k


@pytest.mark.parametrize("name,T", [("2A2F", 2048), ("skew-1A3F", 512)])
def test_noalloc_layout_matches_dispatch_twice(name, T):
    base = W.named(name, T=T)
    first = W.Workload(**{**base.__dict__, "A": 1, "T": (T,), "bucket": T, "capacity": T})
    second = W.Workload(**{**first.__dict__, "seed": first.seed + 99})
    for wl in (first, second):   # two calls in a row share the scratch array
        ids_np = W.make_inputs(wl).ids[0, :T].copy()
        ids_dev = torch.from_numpy(ids_np).cuda()
        ref_ends, ref_row_src = _reference(wl, ids_dev)
        ends, slots, err = _call_c_abi(ids_dev, wl.E, wl.F, wl.alpha)
        _check(wl, ids_np, ends, slots, err, ref_ends, ref_row_src)


def test_noalloc_reports_invalid_route_and_rejects_oversize():
    wl = W.Workload("small", A=1, F=2, E=16, K=4, H=256, alpha=4, capacity=64, bucket=64, T=(64,))
    ids_np = W.make_inputs(wl).ids[0].copy()
    ids_np[9, 2] = 16
    ids_np[3, 3] = ids_np[3, 1]
    ids_dev = torch.from_numpy(ids_np).cuda()
    _, _, err = _call_c_abi(ids_dev, wl.E, wl.F, wl.alpha)
    assert err.tolist() == [afd.ERR_ROUTE_DUP, 3, 3]
    lib = afd.load_library()
    st = lib.afd_route_layout_noalloc(ctypes.c_void_p(ids_dev.data_ptr()), 8193, 1, 16, 2, 4,
                                      ctypes.c_void_p(1), ctypes.c_void_p(1), ctypes.c_void_p(1),
                                      None)
    assert st == afd.ERR_UNSUPPORTED


def test_noalloc_refuses_pageable_host_buffers():
    """Buffers the GPU cannot reach (pageable host memory) are refused on the
    host, before anything is enqueued."""
    lib = afd.load_library()
    ids_dev = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    ids_dev[:, 1] = 1
    ends_host = np.zeros(8, dtype=np.int32)            # pageable
    slots = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    err = torch.zeros((3,), dtype=torch.int32, device="cuda")
    st = lib.afd_route_layout_noalloc(
        ctypes.c_void_p(ids_dev.data_ptr()), 4, 2, 8, 2, 1, ctypes.c_void_p(ends_host.ctypes.data),
        ctypes.c_void_p(slots.data_ptr()), ctypes.c_void_p(err.data_ptr()), None)
    assert st == afd.ERR_ARG
    ids_host = ids_dev.cpu().numpy()                   # pageable
    ends = torch.zeros((8,), dtype=torch.int32, device="cuda")
    st = lib.afd_route_layout_noalloc(
        ctypes.c_void_p(ids_host.ctypes.data), 4, 2, 8, 2, 1, ctypes.c_void_p(ends.data_ptr()),
        ctypes.c_void_p(slots.data_ptr()), ctypes.c_void_p(err.data_ptr()), None)
    assert st == afd.ERR_ARG
