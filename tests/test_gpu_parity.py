"""GPU parity: the library's kernels against the CPU oracle, element by element.

Layout (ends[], host counts, receive shape), receipts (row_src, row weights)
and row bytes must match bit for bit. The combine uses the same fixed-order
FP32 fused multiply-add chain and one round-to-nearest-even as the oracle, so
it must match bit for bit as well (the looser bound of 1 BF16 ulp is not
needed and not used).
"""
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


def _roundtrip_check(wl, mode=GH.SCALE, rhc=False, view=False, transposed=False, num_sms=0,
                     buf=None):
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, mode)
    own = buf is None
    buf = buf or GH.make_buffer(wl, num_sms)
    try:
        dev = GH.to_device(inp, transposed_scales=transposed)
        recvs, _, results = GH.run_exchange(buf, wl, dev, mode=mode, rhc=rhc, view=view)
        torch.cuda.synchronize()
        snap = GH.snapshot(recvs)
        GH.check_layout(wl, snap, exp, rhc, buf)
        GH.check_outputs(wl, results, exp)
        assert buf.get_error()[0] == 0
        return [GH.out_bits(r) for r in results]
    finally:
        if own:
            buf.close()


CASES = (
    [("tiny", None)]
    + [("2A2F", T) for T in (1, 8, 32, 128, 512, 607, 608, 2048)]  # 608 = 4 tokens per SM: per-token combine
    + [("2A2F-H4096", T) for T in (1, 128, 2048)]
    + [("skew-3A1F", T) for T in (1, 32, 512, 2048)]
    + [("skew-1A3F", T) for T in (1, 32, 512, 2048)]
    + [("fp8-2A2F", T) for T in (1, 128, 2048)]
    + [("fp8-2A1F", T) for T in (1, 128, 2048)]
)


@pytest.mark.parametrize("name,T", CASES)
def test_parity_workloads(name, T):
    wl = W.named(name, T=T)
    _roundtrip_check(wl, mode=GH.SCALE)


@pytest.mark.parametrize("name,T", [("tiny", None), ("2A2F", 512), ("skew-3A1F", 128),
                                    ("2A2F-H4096", 2048)])
def test_parity_identity_expert(name, T):
    _roundtrip_check(W.named(name, T=T), mode=GH.IDENTITY)


@pytest.mark.parametrize("name,T", [("tiny", None), ("2A2F", 128), ("skew-1A3F", 512),
                                    ("fp8-2A2F", 128)])
def test_parity_read_host_counts(name, T):
    _roundtrip_check(W.named(name, T=T), rhc=True)


@pytest.mark.parametrize("name,T", [("skew-3A1F", 512), ("fp8-2A1F", 128), ("skew-3A1F", 1)])
def test_single_worker_view_and_copy(name, T):
    wl = W.named(name, T=T)
    res_view = _roundtrip_check(wl, view=True)
    res_copy = _roundtrip_check(wl, view=False)
    for a, b in zip(res_view, res_copy):
        assert np.array_equal(a, b)


def test_view_flag_with_several_workers_returns_ordinary_result():
    wl = W.named("2A2F", T=32)
    _roundtrip_check(wl, view=True)


def test_fp8_transposed_scale_view():
    _roundtrip_check(W.named("fp8-2A2F", T=128), transposed=True)


@pytest.mark.parametrize("T,sms", [(512, 3), (64, 1), (2048, 7)])
def test_sm_cap_gives_identical_results(T, sms):
    _roundtrip_check(W.named("2A2F", T=T), num_sms=sms)


LARGE_LAYOUTS = [
    # several 256-token slices per layout CTA
    W.Workload("many-slices", A=4, F=2, E=128, K=8, H=256, alpha=128, capacity=4096, bucket=4096,
               T=(4096, 4000, 3000, 4096), seed=611),
    # top-k 32: the layout's route codes do not fit shared memory
    W.Workload("wide-topk", A=2, F=4, E=64, K=32, H=256, alpha=8, capacity=2100, bucket=2100,
               T=(2100, 2033), seed=612),
    # ragged sources, one of them empty, three workers, alpha 1
    W.Workload("ragged-5A3F", A=5, F=3, E=96, K=6, H=512, alpha=1, capacity=2048, bucket=2048,
               T=(0, 2048, 1, 1500, 777), routing="zipf", drop=0.1, seed=613),
]


@pytest.mark.parametrize("wl", LARGE_LAYOUTS, ids=lambda w: w.name)
def test_parity_large_layouts(wl):
    _roundtrip_check(wl, mode=GH.SCALE)
    _roundtrip_check(wl, mode=GH.SCALE, rhc=True, num_sms=5)


def test_crafted_fused_ascending_chain_on_gpu():
    """The element whose BF16 result depends on using a fused, ascending
    FP32 chain (worked out in test_oracle_combine): must come out 0x3F81."""
    wl = W.Workload("crafted", A=1, F=1, E=2, K=2, H=256, alpha=1, capacity=1, bucket=1, T=(1,))
    buf = GH.make_buffer(wl)
    try:
        x = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
        ids = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
        w = torch.tensor([[1.0 + 2.0 ** -8, 16647161 * 2.0 ** -24]], dtype=torch.float32, device="cuda")
        buf.source_dispatch(0, x, ids, w, bucket=1)
        r = buf.worker_receive(0, bucket=1)
        ends = r.ends.cpu().tolist()
        assert ends == [1, 2]
        reply = torch.zeros((r.num_rows, 256), dtype=torch.int16, device="cuda")
        reply[0] = 0x3F80
        reply[1] = 0x3381
        buf.worker_reply(0, reply.view(torch.bfloat16), r.receipt)
        out = buf.source_collect(0, num_tokens=1)
        assert torch.all(out.view(torch.int16) == 0x3F81)
    finally:
        buf.close()


def test_exhaustive_tiny_patterns():
    """E=4, K=2, A=2, F=2: every ID pattern (with -1) for two live tokens,
    alpha in {1, 2}, on one reused context."""
    import itertools

    E, K = 4, 2
    pats = [p for p in itertools.product(range(-1, E), repeat=K)
            if len({v for v in p if v >= 0}) == len([v for v in p if v >= 0])]
    rng = np.random.default_rng(0)
    for alpha in (1, 2):
        wl0 = W.Workload("exh", A=2, F=2, E=E, K=K, H=256, alpha=alpha, capacity=2, bucket=2, T=(1, 1))
        buf = GH.make_buffer(wl0)
        try:
            for T in ((1, 1), (0, 2)):
                wl = wl0.with_tokens(T)
                for combo in itertools.product(pats, repeat=2):
                    ids = np.full((2, 2, K), -1, np.int64)
                    it = iter(combo)
                    for s in range(2):
                        for t in range(T[s]):
                            ids[s, t] = next(it)
                    w = rng.random((2, 2, K)).astype(np.float32)
                    xf = rng.standard_normal((2, 2, 256)).astype(np.float32)
                    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                    inp = W.Inputs(wl, ids, w, x)
                    exp = GH.expected(inp, GH.SCALE)
                    dev = GH.to_device(inp)
                    recvs, _, results = GH.run_exchange(buf, wl, dev, mode=GH.SCALE)
                    snap = GH.snapshot(recvs)
                    GH.check_layout(wl, snap, exp, False, buf)
                    GH.check_outputs(wl, results, exp)
        finally:
            buf.close()


def test_edge_cases():
    base = W.named("2A2F", T=64)
    cases = [
        base.with_tokens((0, 64)),                                # a source with no tokens
        base.with_tokens((0, 0)),                                 # nothing at all
        base.with_tokens((2048, 3)),                              # T = capacity next to a small one
        W.Workload("k1", A=2, F=2, E=8, K=1, H=256, alpha=1, capacity=64, bucket=64, T=(64, 17)),
        W.Workload("k=Ef", A=2, F=2, E=8, K=4, H=256, alpha=4, capacity=64, bucket=64, T=(33, 64)),
        W.Workload("k=E", A=1, F=4, E=8, K=8, H=512, alpha=3, capacity=40, bucket=40, T=(40,)),
        W.Workload("bucket>T", A=2, F=2, E=16, K=4, H=768, alpha=128, capacity=300, bucket=300,
                   T=(257, 1)),
        W.Workload("k32", A=2, F=4, E=64, K=32, H=256, alpha=2, capacity=96, bucket=96, T=(96, 50)),
        W.Workload("a=5", A=5, F=2, E=32, K=6, H=1024, alpha=16, capacity=200, bucket=160,
                   T=(160, 0, 77, 1, 159)),
        # the one-warp dispatch takes up to 32 tokens, the one-kernel dispatch up
        # to 2048 routes; both sides of each switch
        W.Workload("tiny-max", A=1, F=2, E=64, K=8, H=512, alpha=8, capacity=40, bucket=40, T=(32,)),
        W.Workload("tiny-max+1", A=1, F=2, E=64, K=8, H=512, alpha=8, capacity=40, bucket=40, T=(33,)),
        W.Workload("tiny-3src", A=3, F=3, E=96, K=32, H=256, alpha=128, capacity=16, bucket=16, T=(11, 0, 9)),
        W.Workload("small-max", A=1, F=2, E=8, K=1, H=256, alpha=1, capacity=4097, bucket=4097,
                   T=(2048,)),
        W.Workload("small-max+1", A=1, F=2, E=8, K=1, H=256, alpha=1, capacity=4097, bucket=4097,
                   T=(2049,)),
        W.Workload("cluster-16x256", A=1, F=2, E=8, K=1, H=256, alpha=1, capacity=4097, bucket=4097,
                   T=(4096,)),
        W.Workload("large-min", A=1, F=2, E=8, K=1, H=256, alpha=1, capacity=4097, bucket=4097,
                   T=(4097,)),
        W.Workload("E1024-small", A=2, F=4, E=1024, K=4, H=256, alpha=8, capacity=600, bucket=600,
                   T=(128, 100)),
        W.Workload("E1024-mid", A=2, F=4, E=1024, K=4, H=256, alpha=8, capacity=600, bucket=600,
                   T=(512, 500)),
        W.Workload("E1024-large", A=2, F=4, E=1024, K=4, H=256, alpha=8, capacity=600, bucket=600,
                   T=(600, 600)),
    ]
    for wl in cases:
        _roundtrip_check(wl, mode=GH.SCALE)


def test_all_skipped_tokens_and_empty_worker():
    wl = W.named("2A2F", T=200)
    inp = W.make_inputs(wl)
    inp.ids[0, :50] = -1                 # all-skipped tokens -> +0 rows
    inp.ids[inp.ids >= 64] = -1          # worker 1 receives nothing
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        recvs, _, results = GH.run_exchange(buf, wl, dev, rhc=True)
        snap = GH.snapshot(recvs)
        GH.check_layout(wl, snap, exp, True, buf)
        GH.check_outputs(wl, results, exp)
        assert snap[1]["num_rows"] == 0
        assert torch.all(results[0][:50].view(torch.int16) == 0)
    finally:
        buf.close()


def test_consecutive_exchanges_with_changing_tokens_and_buckets():
    wl = W.named("2A2F", T=512)
    buf = GH.make_buffer(wl)
    try:
        for i, (T, bucket) in enumerate([((512, 512), 2048), ((7, 300), 300), ((2048, 2048), 2048),
                                         ((1, 0), 1), ((130, 129), 1024)]):
            w2 = wl.with_tokens(T, bucket=bucket)
            w2 = W.Workload(**{**w2.__dict__, "seed": 1000 + i})
            _roundtrip_check(w2, rhc=(i % 2 == 1), buf=buf)
    finally:
        buf.close()


def test_roles_on_separate_streams():
    wl = W.named("2A2F", T=256)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    try:
        dev = GH.to_device(inp)
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            for s in range(wl.A):
                buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], bucket=wl.bucket)
        with torch.cuda.stream(s2):
            recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
            replies = {f: GH.expert_reply(wl, f, recvs[f], GH.SCALE) for f in range(wl.F)}
            for f in range(wl.F):
                buf.worker_reply(f, replies[f], recvs[f].receipt)
        with torch.cuda.stream(s3):
            outs = GH.alloc_outs(wl)
            res = [buf.source_collect(s, out=outs[s]) for s in range(wl.A)]
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, res, exp)
    finally:
        buf.close()


def test_calls_on_another_stream_wait_for_the_callers_work():
    """A call on a new stream waits for everything enqueued before the previous
    call on the old stream, including the caller's own kernels: a slow producer
    of x before source 0's dispatch on one stream, the last dispatch on
    another; a slow expert before the replies on one stream, the collects on
    another. Each slow kernel spins a fixed number of cycles first."""
    wl = W.named("2A2F", T=512)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        dev = GH.to_device(inp)
        x0 = torch.zeros_like(dev.x[0])
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            torch.cuda._sleep(2_000_000)  # about a millisecond
            x0.copy_(dev.x[0])            # the producer of source 0's rows
            buf.source_dispatch(0, x0, dev.ids[0], dev.w[0], bucket=wl.bucket)
        with torch.cuda.stream(s2):
            buf.source_dispatch(1, dev.x[1], dev.ids[1], dev.w[1], bucket=wl.bucket)
            recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
            torch.cuda._sleep(2_000_000)
            replies = {f: GH.expert_reply(wl, f, recvs[f], GH.SCALE) for f in range(wl.F)}
            for f in range(wl.F):
                buf.worker_reply(f, replies[f], recvs[f].receipt)
        with torch.cuda.stream(s1):
            outs = GH.alloc_outs(wl)
            res = [buf.source_collect(s, out=outs[s]) for s in range(wl.A)]
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, res, exp)
    finally:
        buf.close()


@pytest.mark.parametrize("name,T", [("2A2F", 128), ("fp8-2A1F", 64), ("skew-1A3F", 512),
                                    # the benchmark's launch configuration
                                    ("2A2F", 2048), ("2A2F-H4096", 2048)])
def test_graph_replay_with_changed_routing(name, T):
    """Capture one complete exchange, then change IDs, weights and payloads in
    place and replay; every replay must match the oracle on its new inputs."""
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        outs = GH.alloc_outs(wl)
        # warm up eagerly, then capture
        GH.run_exchange(buf, wl, dev, mode=GH.SCALE, outs=outs)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        holder = {}
        with torch.cuda.graph(g):
            recvs, replies, results = GH.run_exchange(buf, wl, dev, mode=GH.IDENTITY if wl.dtype == "bf16"
                                                      else GH.SCALE, outs=outs, view=False)
            holder["recvs"], holder["results"] = recvs, results
        mode = GH.IDENTITY if wl.dtype == "bf16" else GH.SCALE
        for rep in range(3):
            new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 17 * (rep + 1)}))
            GH.refresh_device(dev, new)
            g.replay()
            torch.cuda.synchronize()
            exp = GH.expected(new, mode)
            GH.check_layout(wl, GH.snapshot(holder["recvs"]), exp, False, buf)
            GH.check_outputs(wl, holder["results"], exp)
        del g
    finally:
        buf.close()


@pytest.mark.parametrize("name,T", [("2A2F", 2048), ("2A2F", 8), ("skew-1A3F", 512), ("skew-3A1F", 64),
                                    ("fp8-2A2F", 128)])
@pytest.mark.parametrize("view", [False, True])
def test_collect_all_matches_per_source_collect(name, T, view):
    """One collect call for every source (one combine launch when F > 1)."""
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        dev = GH.to_device(inp)
        for s in range(wl.A):
            buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], dev.scales[s], bucket=wl.bucket)
        recvs = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
        reps = {f: GH.expert_reply(wl, f, recvs[f], GH.SCALE) for f in range(wl.F)}
        for f in range(wl.F):
            buf.worker_reply(f, reps[f], recvs[f].receipt)
        res = buf.source_collect_all(view=view, num_tokens=list(wl.T))
        torch.cuda.synchronize()
        GH.check_outputs(wl, res, exp)
        # the exchange is complete: the next one starts normally
        GH.run_exchange(buf, wl, dev)
    finally:
        buf.close()
