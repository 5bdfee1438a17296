"""The exchange under compute load (afdEP-comm design page, section 14: a
fixed batch of 2,048^3 BF16 GEMMs on a side stream while the exchanges run).

The GEMMs are queued on their own stream ahead of the exchange, so the
exchange's kernels share the SMs with running GEMMs; every exchange, issued
call by call and replayed from a CUDA graph with new inputs, must still match
the oracle bit for bit, with every SM available and with the exchange's
kernels capped at 24 SMs. The GEMMs' own result is checked too (the exchange
must not disturb a concurrent kernel's memory)."""
import pytest
import torch

import gpu_harness as GH
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_GEMM = 120   # about 2 ms of GEMMs, longer than the exchanges they overlap


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


class SideLoad:
    """A batch of BF16 2048^3 GEMMs on a side stream, started after the
    current stream's work so far."""

    def __init__(self):
        g = torch.Generator(device="cuda").manual_seed(7)
        self.a = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16, generator=g) / 32
        self.b = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16, generator=g) / 32
        self.c = torch.empty(2048, 2048, device="cuda", dtype=torch.bfloat16)
        self.want = torch.matmul(self.a, self.b)
        self.stream = torch.cuda.Stream()

    def start(self):
        self.c.zero_()
        ev = torch.cuda.Event()
        ev.record()
        self.stream.wait_event(ev)
        with torch.cuda.stream(self.stream):
            for _ in range(N_GEMM):
                torch.matmul(self.a, self.b, out=self.c)

    def check(self):
        torch.cuda.current_stream().wait_stream(self.stream)
        torch.cuda.synchronize()
        # the same product as computed alone (any disturbance would be far larger)
        torch.testing.assert_close(self.c.float(), self.want.float(), rtol=1e-2, atol=1e-2)


@pytest.mark.parametrize("T", [512, 2048])
@pytest.mark.parametrize("num_sms", [0, 24])
def test_exchange_under_side_stream_gemms(T, num_sms):
    wl = W.named("2A2F", T=T)
    inp = W.make_inputs(wl)
    load = SideLoad()
    buf = GH.make_buffer(wl, num_sms=num_sms)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        # call by call, twice, while the GEMMs run
        exp = GH.expected(inp, GH.SCALE)
        load.start()
        for _ in range(2):
            recvs, _, results = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, outs=outs)
            snap = GH.snapshot(recvs)
            GH.check_layout(wl, snap, exp, False, buf)
            GH.check_outputs(wl, results, exp)
        load.check()
        # captured once, replayed with new inputs while the GEMMs run
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        holder = {}
        with torch.cuda.graph(g):
            holder["recvs"], _, holder["results"] = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, outs=outs)
        for rep in range(3):
            new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 31 * (rep + 1)}))
            GH.refresh_device(dev, new)
            load.start()
            g.replay()
            torch.cuda.synchronize()
            exp = GH.expected(new, GH.SCALE)
            GH.check_layout(wl, GH.snapshot(holder["recvs"]), exp, False, buf)
            GH.check_outputs(wl, holder["results"], exp)
            load.check()
        del g
        assert buf.get_error() == (0, -1, -1, -1)
    finally:
        buf.close()
