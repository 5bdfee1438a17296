"""Page-locked host buffers passed straight to the calls: the kernels read
the inputs and write the results over the host link, and the exchange must be
bit-identical to the oracle, as with device buffers. Pageable host memory is
refused on the host before anything is enqueued, and the exchange can then
go on with valid buffers."""
import numpy as np
import pytest
import torch

import gpu_harness as GH
from combine_attention_ffn_gb300 import afd
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _pinned(inp):
    host = GH.to_device(inp, device="cpu")
    pin = lambda t: None if t is None else t.pin_memory()
    return GH.DeviceInputs([pin(t) for t in host.x], [pin(t) for t in host.ids],
                           [pin(t) for t in host.w], [pin(t) for t in host.scales])


@pytest.mark.parametrize("name,T,host_reply", [("2A2F", 1, False), ("2A2F", 128, True), ("2A2F", 2048, False),
                                               ("skew-3A1F", 32, True), ("fp8-2A2F", 64, False),
                                               ("skew-1A3F", 300, True)])
def test_pinned_host_inputs_outputs_replies(name, T, host_reply):
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = _pinned(inp)
        for s in range(wl.A):
            buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], dev.scales[s], bucket=wl.bucket)
        recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
        replies = {}
        for f in range(wl.F):
            rep = GH.expert_reply(wl, f, recvs[f], GH.SCALE)
            if host_reply:
                torch.cuda.synchronize()
                rep = rep.cpu().pin_memory()
            replies[f] = rep
            buf.worker_reply(f, rep, recvs[f].receipt)
        outs = [torch.empty((t, wl.H), dtype=torch.bfloat16).pin_memory() for t in wl.T]
        res = buf.source_collect_all(outs=outs) if T % 2 else \
            [buf.source_collect(s, out=outs[s]) for s in range(wl.A)]
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, res, exp)
        assert all(r.device.type == "cpu" for r in res)
    finally:
        buf.close()


def test_pageable_input_refused_then_exchange_proceeds():
    wl = W.named("2A2F", T=64)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        pageable = GH.to_device(inp, device="cpu")
        assert not pageable.x[0].is_pinned()
        for field in ("x", "ids", "w"):
            args = [dev.x[0], dev.ids[0], dev.w[0]]
            args[("x", "ids", "w").index(field)] = getattr(pageable, field)[0]
            with pytest.raises(afd.AfdError) as e:
                buf.source_dispatch(0, *args, bucket=wl.bucket)
            assert e.value.status == afd.ERR_ARG
            assert "pageable" in str(e.value)
        recvs, _, res = GH.run_exchange(buf, wl, dev, mode=GH.SCALE)
        torch.cuda.synchronize()
        GH.check_outputs(wl, res, exp)
    finally:
        buf.close()


def test_pageable_reply_and_out_refused():
    wl = W.named("2A2F", T=64)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        for s in range(wl.A):
            buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], bucket=wl.bucket)
        recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
        replies = {f: GH.expert_reply(wl, f, recvs[f], GH.SCALE) for f in range(wl.F)}
        torch.cuda.synchronize()
        with pytest.raises(afd.AfdError) as e:
            buf.worker_reply(0, replies[0].cpu(), recvs[0].receipt)
        assert e.value.status == afd.ERR_ARG
        for f in range(wl.F):
            buf.worker_reply(f, replies[f], recvs[f].receipt)
        bad = [torch.empty((t, wl.H), dtype=torch.bfloat16) for t in wl.T]
        with pytest.raises(afd.AfdError) as e:
            buf.source_collect(0, out=bad[0])
        assert e.value.status == afd.ERR_ARG
        with pytest.raises(afd.AfdError) as e:
            buf.source_collect_all(outs=bad)
        assert e.value.status == afd.ERR_ARG
        res = buf.source_collect_all(outs=GH.alloc_outs(wl))
        torch.cuda.synchronize()
        GH.check_outputs(wl, res, exp)
    finally:
        buf.close()


def test_pinned_host_buffers_in_a_captured_graph():
    """The pinned buffers' addresses are fixed, so the exchange can be
    captured once and replayed on new values written into them."""
    wl = W.named("2A2F", T=256)
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        dev = _pinned(inp)
        outs = [torch.empty((t, wl.H), dtype=torch.bfloat16).pin_memory() for t in wl.T]

        def step():
            GH.run_exchange(buf, wl, dev, mode=GH.IDENTITY, outs=outs)

        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for seed in (11, 12):
            new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": seed}))
            GH.refresh_device(dev, new)
            g.replay()
            torch.cuda.synchronize()
            GH.check_outputs(wl, outs, GH.expected(new, GH.IDENTITY))
        del g
    finally:
        buf.close()


def test_cached_dispatch_from_pinned_host_inputs():
    """A cached dispatch (the last routing reused) reading new activations and
    weights straight from pinned host memory matches a full dispatch of the
    same IDs from device memory."""
    wl = W.named("2A2F", T=300)
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
        other = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 5}))
        w = other.w.copy()
        w[inp.ids < 0] = inp.w[inp.ids < 0]
        new = W.Inputs(wl, inp.ids.copy(), w, other.x.copy(), None)
        exp = GH.expected(new, GH.SCALE)
        host = _pinned(new)
        for s in range(wl.A):
            buf.source_dispatch_cached(s, host.x[s], host.w[s], bucket=wl.bucket)
        recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
        replies = {f: GH.expert_reply(wl, f, recvs[f], GH.SCALE) for f in range(wl.F)}  # kept alive
        for f in range(wl.F):
            buf.worker_reply(f, replies[f], recvs[f].receipt)
        res = buf.source_collect_all(outs=GH.alloc_outs(wl))
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, res, exp)
    finally:
        buf.close()
