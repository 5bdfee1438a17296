"""The allocation-free routing layout (afd_route_layout_noalloc) against the
CPU oracle.

Callers that cannot call cudaMalloc (code inside another framework's memory
pool or allocator hook, or a process whose device memory is fully reserved up
front) use this entry point; its scratch is a fixed device array in the
library. For one source's routing its ends[], every route's row and its first
invalid route must equal what the oracle computes for a single source
(A = 1, bucket = T): the oracle's layout gives ends[], its dispatch the row of
every route, its validation the first invalid route. Calls share the scratch
array, so several calls run in a row in one process. This file is collected
last so that a run stopping at the first failure has run every other test
first.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_attention_ffn_gb300 import afd
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

_ORACLE_CODE = {oracle.ROUTE_OK: afd.OK, oracle.ROUTE_RANGE: afd.ERR_ROUTE_RANGE,
                oracle.ROUTE_DUP: afd.ERR_ROUTE_DUP}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _ids(name, T, seed_offset=0, **over):
    """One source's IDs [T, K] drawn like the named workload (bucket = T)."""
    base = W.named(name, T=min(T, 2048))
    wl = W.Workload(**{**base.__dict__, "A": 1, "T": (T,), "bucket": max(T, 1),
                       "capacity": max(T, 1), "seed": base.seed + seed_offset, **over})
    return wl, W.make_inputs(wl).ids[0, :T].copy()


def _oracle(ids_np, E, F, alpha):
    """(error triple, ends [E], slots [T, K]) from the oracle for one source."""
    T, K = ids_np.shape
    bucket = max(T, 1)
    ids3 = np.full((1, bucket, K), -1, np.int64)
    ids3[0, :T] = ids_np
    p = oracle.Problem(1, F, E, K, 256, alpha, bucket, oracle.BF16, [T])
    code, _, t, k = oracle.validate(p, ids3)
    lay = oracle.layout(p, ids3)
    r_stride = max(1, int(lay["r_exact"].max()))
    x = np.zeros((1, bucket, 256), np.uint16)
    w = np.zeros((1, bucket, K), np.float32)
    d = oracle.dispatch(p, ids3, w, x, None, lay, r_stride)
    return [_ORACLE_CODE[code], t, k], lay["ends"].reshape(-1), d["slot"][0, :T]


def _call_c_abi(ids, E, F, alpha, where="cuda"):
    """Calls the entry point through the C ABI with raw pointers. `ids` is a
    tensor (device or pinned host); the outputs go to `where` ("cuda", or
    "pinned" for page-locked host memory the kernels write over the link)."""
    lib = afd.load_library()
    T, K = ids.shape
    kw = dict(device="cuda") if where == "cuda" else dict(pin_memory=True)
    ends = torch.full((E,), -7, dtype=torch.int32, **kw)
    slots = torch.full((max(T, 1), K), -7, dtype=torch.int32, **kw)
    err = torch.full((3,), -7, dtype=torch.int32, **kw)
    st = lib.afd_route_layout_noalloc(
        ctypes.c_void_p(ids.data_ptr() if T else None), T, K, E, F, alpha,
        ctypes.c_void_p(ends.data_ptr()), ctypes.c_void_p(slots.data_ptr() if T else None),
        ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == afd.OK, afd.load_library().afd_status_string(st)
    torch.cuda.synchronize()
    return ends.cpu().numpy(), slots[:T].cpu().numpy(), err.cpu().numpy()


def _check(ids_np, E, F, alpha, where="cuda", ids_where="cuda"):
    want_err, want_ends, want_slots = _oracle(ids_np, E, F, alpha)
    t_ids = torch.from_numpy(ids_np)
    t_ids = t_ids.cuda() if ids_where == "cuda" else t_ids.pin_memory()
    ends, slots, err = _call_c_abi(t_ids, E, F, alpha, where)
    assert err.tolist() == want_err
    assert np.array_equal(ends, want_ends)
    assert np.array_equal(slots, want_slots)
    return err


@pytest.mark.parametrize("T", [1, 255, 257, 2047, 8192])
def test_noalloc_layout_matches_oracle_twice(T):
    """Uniform 2A2F-shaped routing (E=128, K=8, two workers, alignment 128),
    token counts on both sides of the 256-token counting chunk and the
    largest accepted (8,192 tokens = 65,536 routes); two different routings in
    a row, since the calls share the scratch array."""
    for seed_offset in (0, 99):
        wl, ids_np = _ids("2A2F", T, seed_offset)
        _check(ids_np, wl.E, wl.F, wl.alpha)


def test_noalloc_skewed_routing_with_skips():
    """Zipf-like routing with 10% of the slots -1, three workers of 32
    experts (the 1A:3F shape)."""
    wl, ids_np = _ids("skew-1A3F", 1000)
    assert (ids_np == -1).any()
    _check(ids_np, wl.E, wl.F, wl.alpha)


def test_noalloc_most_experts():
    """E = 1,024, the largest accepted, where the counting kernel's per-warp
    masks and bases fill its 48 KB of shared memory."""
    wl, ids_np = _ids("2A2F", 2047, E=1024, F=4, alpha=16)
    _check(ids_np, 1024, 4, 16)


def test_noalloc_first_invalid_route_in_token_then_k_order():
    """Range and duplicate errors: the one that comes first in (token, k)
    order is reported, whatever its kind; invalid routes get no row."""
    wl, ids_np = _ids("2A2F", 300)
    a = ids_np.copy()
    a[5, 1] = wl.E + 3                # range error at (5, 1) ...
    a[9, 3] = a[9, 0]                 # ... before a duplicate at (9, 3)
    a[270, 6] = -9                    # and a range error in the second chunk
    err = _check(a, wl.E, wl.F, wl.alpha)
    assert err.tolist() == [afd.ERR_ROUTE_RANGE, 5, 1]
    b = ids_np.copy()
    b[7, 2] = b[7, 0]                 # duplicate at (7, 2) ...
    b[7, 5] = -9                      # ... before a range error later in the same token
    b[260, 1] = (1 << 33) + 2         # an int64 ID outside int32 (2 if truncated)
    err = _check(b, wl.E, wl.F, wl.alpha)
    assert err.tolist() == [afd.ERR_ROUTE_DUP, 7, 2]
    c = ids_np.copy()
    c[260, 1] = (1 << 33) + 2
    err = _check(c, wl.E, wl.F, wl.alpha)
    assert err.tolist() == [afd.ERR_ROUTE_RANGE, 260, 1]


def test_noalloc_outputs_and_ids_in_pinned_host_memory():
    """Page-locked host buffers are reached through their mapped device
    addresses: the outputs written there, and the IDs read from there, give
    the oracle's result."""
    wl, ids_np = _ids("2A2F", 600)
    _check(ids_np, wl.E, wl.F, wl.alpha, where="pinned")
    _check(ids_np, wl.E, wl.F, wl.alpha, ids_where="pinned")


def test_noalloc_empty_routing():
    """No tokens: every expert's end is 0 and no error is reported."""
    ids = torch.zeros((0, 8), dtype=torch.int64, device="cuda")
    ends, _, err = _call_c_abi(ids, 128, 2, 128)
    assert err.tolist() == [0, -1, -1]
    assert not ends.any()


def test_noalloc_rejects_oversize_before_enqueueing():
    lib = afd.load_library()
    bogus = ctypes.c_void_p(16)
    for T, K, E, F, alpha in ((8193, 1, 16, 2, 4), (4096, 17, 32, 2, 1), (64, 8, 1025, 1, 1),
                              (8192, 8, 1024, 1, 1 << 21)):
        st = lib.afd_route_layout_noalloc(bogus, T, K, E, F, alpha, bogus, bogus, bogus, None)
        assert st == afd.ERR_UNSUPPORTED, (T, K, E, F, alpha)


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
