"""A combine launched right after the previous combine of the same exchange
on the same stream starts without the dependency wait (its launch implies
that the scatter and the expert have completed) and waits at its end
instead.

These tests aim at what could go wrong with that: reply rows read before
they are final, or through lines an earlier kernel left in an SM's L1. The
identity expert makes the combine read the arena rows the scatter has just
rewritten; between exchanges a reduction reads every arena row through
ordinary, L1-allocating loads, so that old contents of those rows sit in L1
caches when the next exchange runs. Every exchange has new inputs and must
match the oracle bit for bit, issued call by call and replayed from a graph.
The last source's combine must also complete only after the others: a
result read right after it (same stream) is complete for every source."""
import numpy as np
import pytest
import torch

import gpu_harness as GH
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


def _touch_through_l1(recvs):
    """An ordinary PyTorch reduction over every received row (plain global
    loads, which allocate in L1)."""
    acc = torch.zeros((), dtype=torch.float64, device="cuda")
    for r in recvs.values():
        acc += r.rows.view(torch.int16).to(torch.float64).sum()
    return acc


@pytest.mark.parametrize("name,T", [("2A2F", 2048), ("2A2F", 64), ("2A2F-H4096", 700),
                                    ("fp8-2A2F", 300),
                                    # a large launch then a small early one (L2-only loads, no
                                    # fence), and a small launch then a large early one (fence)
                                    ("2A2F", (2048, 100)), ("2A2F", (100, 2048))])
def test_early_combine_sees_every_new_reply(name, T):
    wl = W.named(name, T=T) if isinstance(T, int) else W.named(name).with_tokens(T)
    mode = GH.IDENTITY if wl.dtype == "bf16" else GH.SCALE
    buf = GH.make_buffer(wl)
    try:
        inp = W.make_inputs(wl)
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        # call by call
        for rep in range(4):
            new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 101 * (rep + 1)}))
            GH.refresh_device(dev, new)
            recvs, _, results = GH.run_exchange(buf, wl, dev, mode=mode, outs=outs)
            GH.check_outputs(wl, results, GH.expected(new, mode))
            _touch_through_l1(recvs)
        # captured once, replayed with new inputs
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        holder = {}
        with torch.cuda.graph(g):
            holder["recvs"], _, holder["results"] = GH.run_exchange(buf, wl, dev, mode=mode, outs=outs)
        for rep in range(4):
            new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 211 * (rep + 1)}))
            GH.refresh_device(dev, new)
            g.replay()
            # read on the same stream, right after the replay: the last
            # combine completes only after every earlier one
            got = [o.view(torch.int16).to("cpu", non_blocking=False) for o in holder["results"]]
            exp = GH.expected(new, mode)
            for s, o in enumerate(got):
                assert np.array_equal(o.numpy().view(np.uint16), exp["out"][s, :wl.T[s]]), f"source {s}"
            _touch_through_l1(holder["recvs"])
        del g
    finally:
        buf.close()


@pytest.mark.parametrize("order", [(0, 1, 2), (2, 0, 1)])
def test_three_sources_collected_one_by_one(order):
    """Three sources, two workers: each later collect starts its combine
    early; with ragged mid-size batches every per-source launch takes a third
    of the SMs. Any collect order, call by call and from a graph."""
    wl = W.Workload("3A2F-ragged", A=3, F=2, E=64, K=6, H=2048, alpha=16, capacity=512, bucket=512,
                    T=(300, 512, 417), seed=717)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)

        def exchange():
            for s in range(wl.A):
                buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], bucket=wl.bucket)
            recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
            replies = {f: GH.expert_reply(wl, f, recvs[f], GH.SCALE) for f in range(wl.F)}
            for f in range(wl.F):
                buf.worker_reply(f, replies[f], recvs[f].receipt)
            for s in order:
                buf.source_collect(s, out=outs[s])

        exchange()
        torch.cuda.synchronize()
        GH.check_outputs(wl, outs, exp)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            exchange()
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        GH.check_outputs(wl, outs, exp)
        del g
    finally:
        buf.close()
