"""The phase-timer build (-DAFD_PHASE_TIMERS=1): its exchanges still match the
oracle bit for bit, and its %globaltimer stamps respect the order the kernels'
dependency waits impose (a kernel passes its wait only after the kernel before
it has ended)."""
import numpy as np
import pytest
import torch

import gpu_harness as GH
from combine_attention_ffn_gb300 import afd, build
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SLACK_NS = 1000  # the global timer's ticks and its reading on different SMs


@pytest.fixture(scope="module")
def timer_lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    prev = afd.load_library()
    afd.use_library(build.build_timers())
    yield
    afd._lib = prev


def _kernel(st, kind, points):
    """Stamps [blocks, points] of the blocks that recorded this kind."""
    v = st[kind][:, list(points)].astype(np.int64)
    return v[(v > 0).all(axis=1)]


@pytest.mark.parametrize("name,T", [("2A2F", 2048), ("2A2F", 512), ("2A2F", 8)])
def test_timer_build_matches_oracle_and_orders_phases(timer_lib, name, T):
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        GH.run_exchange(buf, wl, dev, mode=GH.SCALE, outs=outs)
        torch.cuda.synchronize()
        buf.phase_stamps(clear=True)
        recvs, _, results = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, outs=outs)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
        st = buf.phase_stamps()
    finally:
        buf.close()
    large = wl.A * T * wl.K > 2048
    first = _kernel(st, 0, (0, 1, 2, 3, 4, 5, 6, 7) if large else (0, 1, 7))
    assert len(first) > 0
    assert (np.diff(first, axis=1) >= 0).all()  # points in program order
    end_of_dispatch = first[:, -1].max()
    if large:
        sc = _kernel(st, 1, (0, 1, 2, 3, 4, 5))
        assert len(sc) > 0 and (np.diff(sc, axis=1) >= 0).all()
        assert sc[:, 1].min() + SLACK_NS >= end_of_dispatch  # its wait passes after the layout ends
        end_of_dispatch = sc[:, -1].max()
    comb = _kernel(st, 2, (0, 1, 2, 3))
    assert len(comb) > 0 and (np.diff(comb, axis=1) >= 0).all()
    assert comb[:, 1].min() + SLACK_NS >= end_of_dispatch  # the first combine waits for the dispatch
    early = _kernel(st, 3, (0, 1, 2, 3))
    assert len(early) > 0
    assert early[:, 3].min() + SLACK_NS >= comb[:, 3].max()  # the early combine ends after the first


def test_timeline_tool_runs(timer_lib):
    from combine_attention_ffn_gb300 import timeline

    lines = timeline.run("2A2F", 512, 2, False, "fused")
    assert any(line.startswith("dispatch") for line in lines)
    assert any(line.startswith("combine-early") for line in lines)
