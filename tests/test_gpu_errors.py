"""Error paths. Invalid routes are found on the GPU and reported through the
sticky route error (never a trap); call-order and shape mistakes are caught
on the host before anything is enqueued."""
import numpy as np
import pytest
import torch

import gpu_harness as GH
import oracle
from combine_attention_ffn_gb300 import afd
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _oracle_first_error(inp):
    wl = inp.wl
    p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, oracle.BF16, list(wl.T))
    code, s, t, k = oracle.validate(p, inp.ids)
    return {0: 0, oracle.ROUTE_RANGE: afd.ERR_ROUTE_RANGE, oracle.ROUTE_DUP: afd.ERR_ROUTE_DUP}[code], s, t, k


@pytest.mark.parametrize("T", [300, 100, 8])
@pytest.mark.parametrize("plant", ["range_high", "range_low", "wide", "dup", "two_errors",
                                   "dup_and_range_later"])
def test_invalid_routes_reported_like_the_oracle(plant, T):
    wl = W.named("2A2F", T=T)
    inp = W.make_inputs(wl)
    at = lambda t: t * T // 300  # the same relative positions at every size
    if plant == "range_high":
        inp.ids[1, at(123), 4] = 128
    elif plant == "range_low":
        inp.ids[0, at(299), 7] = -5
    elif plant == "wide":
        inp.ids[1, 0, 0] = (1 << 33) + 3   # 3 if truncated to 32 bits
    elif plant == "dup":
        inp.ids[0, at(77), 6] = inp.ids[0, at(77), 2]
    elif plant == "two_errors":
        inp.ids[1, at(5), 1] = 999
        inp.ids[0, at(260), 3] = inp.ids[0, at(260), 0]
    elif plant == "dup_and_range_later":
        inp.ids[0, at(10), 5] = inp.ids[0, at(10), 4]
        inp.ids[0, at(10), 6] = 4000
    want = _oracle_first_error(inp)
    assert want[0] != 0
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        GH.run_exchange(buf, wl, dev)
        assert buf.get_error() == want
        # sticky across an exchange with valid routes
        good = W.make_inputs(W.named("2A2F", T=T))
        GH.run_exchange(buf, wl, GH.to_device(good))
        assert buf.get_error() == want
        buf.clear_error()
        torch.cuda.synchronize()
        assert buf.get_error() == (0, -1, -1, -1)
        # and the context still computes correct exchanges
        exp = GH.expected(good, GH.SCALE)
        recvs, _, results = GH.run_exchange(buf, wl, GH.to_device(good))
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
    finally:
        buf.close()


def test_read_host_counts_reports_route_error():
    wl = W.named("2A2F", T=64)
    inp = W.make_inputs(wl)
    inp.ids[1, 3, 3] = 130
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        for s in range(wl.A):
            buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], bucket=wl.bucket, read_host_counts=True)
        with pytest.raises(afd.AfdError) as ei:
            buf.worker_receive(0, bucket=wl.bucket, read_host_counts=True)
        assert ei.value.status == afd.ERR_ROUTE_RANGE
        buf.reset_exchange()
        buf.clear_error()
        good = W.make_inputs(wl)
        recvs, _, results = GH.run_exchange(buf, wl, GH.to_device(good), rhc=True)
        exp = GH.expected(good, GH.SCALE)
        GH.check_outputs(wl, results, exp)
    finally:
        buf.close()


def _status(fn):
    try:
        fn()
    except afd.AfdError as e:
        return e.status
    return afd.OK


def test_host_side_errors_enqueue_nothing():
    wl = W.named("tiny")
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        d = GH.to_device(inp)
        B = wl.bucket
        # bucket and token checks
        assert _status(lambda: buf.source_dispatch(0, d.x[0], d.ids[0], d.w[0], bucket=B + 1)) == afd.ERR_BUCKET
        assert _status(lambda: buf.source_dispatch(0, d.x[0], d.ids[0], d.w[0], bucket=B - 1)) == afd.ERR_BUCKET
        assert _status(lambda: buf.source_dispatch(9, d.x[0], d.ids[0], d.w[0], bucket=B)) == afd.ERR_ARG
        # receive / reply / collect before dispatch
        assert _status(lambda: buf.worker_receive(0, bucket=B)) == afd.ERR_STATE
        assert _status(lambda: buf.source_collect(0, num_tokens=16)) == afd.ERR_STATE
        buf.source_dispatch(0, d.x[0], d.ids[0], d.w[0], bucket=B)
        # double dispatch, and a role disagreeing on the bucket / policy
        assert _status(lambda: buf.source_dispatch(0, d.x[0], d.ids[0], d.w[0], bucket=B)) == afd.ERR_STATE
        assert _status(lambda: buf.source_dispatch(1, d.x[1][:8], d.ids[1][:8], d.w[1][:8], bucket=8)) \
            == afd.ERR_BUCKET
        assert _status(lambda: buf.source_dispatch(1, d.x[1], d.ids[1], d.w[1], bucket=B,
                                                   read_host_counts=True)) == afd.ERR_BUCKET
        buf.source_dispatch(1, d.x[1], d.ids[1], d.w[1], bucket=B)
        assert _status(lambda: buf.worker_receive(0, bucket=8)) == afd.ERR_BUCKET
        r0 = buf.worker_receive(0, bucket=B)
        assert _status(lambda: buf.worker_receive(0, bucket=B)) == afd.ERR_STATE
        # reply before receive, wrong receipt, wrong shape
        rows1 = torch.zeros((r0.num_rows, wl.H), dtype=torch.bfloat16, device="cuda")
        assert _status(lambda: buf.worker_reply(1, rows1, r0.receipt)) == afd.ERR_STATE
        r1 = buf.worker_receive(1, bucket=B)
        assert _status(lambda: buf.worker_reply(1, rows1, r0.receipt)) == afd.ERR_RECEIPT
        short = torch.zeros((r1.num_rows - 1, wl.H), dtype=torch.bfloat16, device="cuda")
        assert _status(lambda: buf.worker_reply(1, short, r1.receipt)) == afd.ERR_RECEIPT
        assert _status(lambda: buf.source_collect(0, num_tokens=16)) == afd.ERR_STATE
        # the reply rows must stay alive until the combine has read them
        rep0 = GH.expert_reply(wl, 0, r0, GH.SCALE)
        rep1 = GH.expert_reply(wl, 1, r1, GH.SCALE)
        buf.worker_reply(0, rep0, r0.receipt)
        assert _status(lambda: buf.worker_reply(0, rows1, r0.receipt)) == afd.ERR_STATE
        buf.worker_reply(1, rep1, r1.receipt)
        out0 = buf.source_collect(0, num_tokens=16)
        assert _status(lambda: buf.source_collect(0, num_tokens=16)) == afd.ERR_STATE
        # a stale receipt from the finished exchange is rejected next time
        out1 = buf.source_collect(1, num_tokens=16)
        exp = GH.expected(inp, GH.SCALE)
        GH.check_outputs(wl, [out0, out1], exp)
        recvs, _, results = GH.run_exchange(buf, wl, d, mode=GH.SCALE)
        GH.check_outputs(wl, results, exp)
        buf.source_dispatch(0, d.x[0], d.ids[0], d.w[0], bucket=B)
        buf.source_dispatch(1, d.x[1], d.ids[1], d.w[1], bucket=B)
        r0b = buf.worker_receive(0, bucket=B)
        rep0b = GH.expert_reply(wl, 0, r0b, GH.SCALE)
        assert _status(lambda: buf.worker_reply(0, rep0b, r0.receipt)) == afd.ERR_RECEIPT
        torch.cuda.synchronize()
        buf.reset_exchange()
    finally:
        buf.close()


def test_read_host_counts_during_capture_is_refused():
    wl = W.named("tiny")
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        d = GH.to_device(inp)
        GH.run_exchange(buf, wl, d)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        st = None
        with torch.cuda.graph(g):
            st = _status(lambda: buf.source_dispatch(0, d.x[0], d.ids[0], d.w[0], bucket=wl.bucket,
                                                     read_host_counts=True))
        assert st == afd.ERR_CAPTURING
        del g
    finally:
        buf.close()


@pytest.mark.parametrize("name,T", [("2A2F", 512), ("fp8-2A2F", 300)])
def test_scatter_wait_that_gives_up_is_reported_and_recoverable(name, T):
    """The bulk-copy scatter waits a bounded number of polls for each source
    row's load. With the limit at 0 every warp's first wait gives up at once:
    the scatter reports AFD_ERR_TIMEOUT at the first token in (source, token)
    order, waits for the load still in flight, and writes every receipt
    anyway, so the receive side is the oracle's layout and the combine reads
    only rows inside the arenas. The context then runs a correct exchange."""
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    assert sum(wl.T) * wl.K > 2048 and sum(wl.T) > 32  # the layout + bulk-scatter path
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        buf.set_wait_limit(0)
        recvs, _, _ = GH.run_exchange(buf, wl, dev)
        snap = GH.snapshot(recvs)
        torch.cuda.synchronize()
        assert buf.get_error() == (afd.ERR_TIMEOUT, 0, 0, 0)
        for f in range(wl.F):
            R = int(exp["r_exact"][f])
            assert np.array_equal(snap[f]["ends"], exp["ends"][f])
            assert np.array_equal(snap[f]["row_src"][:R], exp["row_src"][f, :R])
            assert np.array_equal(snap[f]["weights"][:R].view(np.uint32),
                                  exp["row_w"][f, :R].view(np.uint32))
        with pytest.raises(afd.AfdError):
            buf.set_wait_limit(-1)
        buf.set_wait_limit(1 << 22)
        buf.clear_error()
        recvs, _, results = GH.run_exchange(buf, wl, dev)
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
        assert buf.get_error() == (0, -1, -1, -1)
    finally:
        buf.close()


def test_l2_flush_runs_and_keeps_the_exchange_exact():
    """The benchmark flush (evict-last writes and reads of a scratch buffer,
    then a discard of the read half) runs between exchanges without touching
    anything but its scratch: the exchange after it still matches the
    oracle."""
    from combine_attention_ffn_gb300 import afd

    lib = afd.load_library()
    scratch = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    wl = W.named("2A2F", T=300)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        for _ in range(2):
            st = lib.afd_l2_flush(scratch.data_ptr(), scratch.numel(), torch.cuda.current_stream().cuda_stream)
            assert st == afd.OK
            recvs, _, results = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, outs=outs)
            torch.cuda.synchronize()
            GH.check_outputs(wl, results, exp)
    finally:
        buf.close()
