"""Cached dispatch (reuse of the last exchange's routing): the result must be
bit-identical to a full dispatch of the same IDs with the new activations
(and, when given, the new weights)."""
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


def _fresh_values(inp, seed, new_weights):
    """Same IDs, new activations (and maybe new weights)."""
    wl = inp.wl
    other = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": seed}))
    w = other.w.copy() if new_weights else inp.w.copy()
    w[inp.ids < 0] = inp.w[inp.ids < 0]
    return W.Inputs(wl, inp.ids.copy(), w, other.x.copy(), None if other.x_scales is None else other.x_scales.copy())


def _cached_exchange(buf, wl, dev, new_w, mode, rhc=False, outs=None):
    for s in range(wl.A):
        buf.source_dispatch_cached(s, dev.x[s], dev.w[s] if new_w else None, dev.scales[s],
                                   bucket=wl.bucket, read_host_counts=rhc)
    recvs = {f: buf.worker_receive(f, bucket=wl.bucket, read_host_counts=rhc) for f in range(wl.F)}
    replies = {f: GH.expert_reply(wl, f, recvs[f], mode) for f in range(wl.F)}
    for f in range(wl.F):
        buf.worker_reply(f, replies[f], recvs[f].receipt)
    outs = outs if outs is not None else GH.alloc_outs(wl)
    res = [buf.source_collect(s, out=outs[s]) for s in range(wl.A)]
    return recvs, replies, res


@pytest.mark.parametrize("name,T,new_w", [("2A2F", 1, True), ("2A2F", 128, False), ("2A2F", 2048, True),
                                          ("skew-3A1F", 32, True), ("fp8-2A2F", 128, True),
                                          ("skew-1A3F", 512, False)])
def test_cached_dispatch_matches_full_dispatch(name, T, new_w):
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
        for rep in range(2):
            new = _fresh_values(inp, wl.seed + 7 + rep, new_w)
            exp = GH.expected(new, GH.SCALE)
            dev = GH.to_device(new)
            recvs, _, res = _cached_exchange(buf, wl, dev, new_w, GH.SCALE, rhc=(rep == 1))
            torch.cuda.synchronize()
            GH.check_layout(wl, GH.snapshot(recvs), exp, rep == 1, buf)
            GH.check_outputs(wl, res, exp)
            if not new_w:
                inp = new
    finally:
        buf.close()


def test_cached_dispatch_rules():
    wl = W.named("2A2F", T=64)
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)

        def status(fn):
            try:
                fn()
            except afd.AfdError as e:
                return e.status
            return afd.OK

        # nothing to reuse yet
        assert status(lambda: buf.source_dispatch_cached(0, dev.x[0], bucket=wl.bucket)) == afd.ERR_STATE
        GH.run_exchange(buf, wl, dev)
        # a different token count or bucket
        assert status(lambda: buf.source_dispatch_cached(0, dev.x[0][:10], bucket=wl.bucket)) == afd.ERR_STATE
        assert status(lambda: buf.source_dispatch_cached(0, dev.x[0], bucket=1024)) == afd.ERR_STATE
        # no mixing of the two dispatch calls in one exchange
        buf.source_dispatch_cached(0, dev.x[0], bucket=wl.bucket)
        assert status(lambda: buf.source_dispatch(1, dev.x[1], dev.ids[1], dev.w[1], bucket=wl.bucket)) \
            == afd.ERR_STATE
        buf.source_dispatch_cached(1, dev.x[1], bucket=wl.bucket)
        torch.cuda.synchronize()
        buf.reset_exchange()
        buf.source_dispatch(0, dev.x[0], dev.ids[0], dev.w[0], bucket=wl.bucket)
        assert status(lambda: buf.source_dispatch_cached(1, dev.x[1], bucket=wl.bucket)) == afd.ERR_STATE
        buf.reset_exchange()
    finally:
        buf.close()


def test_cached_exchange_in_a_graph():
    wl = W.named("2A2F", T=8)
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        GH.run_exchange(buf, wl, dev, mode=GH.IDENTITY, outs=outs)
        _cached_exchange(buf, wl, dev, True, GH.IDENTITY, outs=outs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            recvs, _, res = _cached_exchange(buf, wl, dev, True, GH.IDENTITY, outs=outs)
        for rep in range(3):
            new = _fresh_values(inp, wl.seed + 100 + rep, True)
            GH.refresh_device(dev, new)
            g.replay()
            torch.cuda.synchronize()
            GH.check_outputs(wl, res, GH.expected(new, GH.IDENTITY))
        del g
    finally:
        buf.close()
