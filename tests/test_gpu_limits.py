"""The largest role counts the library accepts (64 sources, 64 workers),
against the oracle. With 64 sources that each collect on their own, the
second to the last combine all start early, each on a 64th of the SMs."""
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


RAGGED_64 = tuple((s * 37) % 101 for s in range(64))  # 0 .. 100 tokens, source 0 empty


def _check(wl, view=False, graph=False):
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        recvs, _, results = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, view=view, outs=outs)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
        if graph:
            g = torch.cuda.CUDAGraph()
            holder = {}
            with torch.cuda.graph(g):
                holder["r"] = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, view=view, outs=outs)[2]
            new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 5}))
            GH.refresh_device(dev, new)
            g.replay()
            torch.cuda.synchronize()
            GH.check_outputs(wl, holder["r"], GH.expected(new, GH.SCALE))
            del g
        assert buf.get_error()[0] == 0
    finally:
        buf.close()


def test_sixty_four_sources_collected_one_by_one():
    wl = W.Workload("64A2F", A=64, F=2, E=16, K=4, H=256, alpha=8, capacity=128, bucket=128,
                    T=RAGGED_64, seed=801)
    _check(wl, graph=True)


def test_sixty_four_workers():
    wl = W.Workload("2A64F", A=2, F=64, E=128, K=8, H=512, alpha=1, capacity=320, bucket=320,
                    T=(300, 257), seed=802)
    _check(wl, graph=True)


@pytest.mark.parametrize("view", [False, True])
def test_sixty_four_sources_one_worker(view):
    wl = W.Workload("64A1F", A=64, F=1, E=32, K=4, H=256, alpha=4, capacity=128, bucket=128,
                    T=RAGGED_64, routing="zipf", drop=0.1, seed=803)
    _check(wl, view=view)
