"""Seeded random exchanges: shapes, routing skew, drops, alignment, worker
counts, dtypes, combine modes, SM caps and host-count modes drawn at random,
one exchange each (plus a cached dispatch and a second exchange on the same
context), every result compared with the oracle bit for bit. The draws cover
the one-warp, one-kernel and cluster dispatch paths and both combine kernels;
the wide draws add many sources and workers, top-k up to 32, rows past the
bulk-copy limit, shuffled call orders, one collect for all sources and graph
replays on new inputs."""
import random

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


def _draw(seed: int):
    rng = random.Random(seed)
    F = rng.choice([1, 2, 3, 4])
    Ef = rng.choice([2, 4, 8, 16, 32, 64])
    E = F * Ef
    K = rng.randint(1, min(E, 16))
    A = rng.randint(1, 4)
    H = rng.choice([256, 512, 768, 1024])
    alpha = rng.choice([1, 2, 4, 16, 128])
    size = rng.choice(["tiny", "small", "large"])
    cap = {"tiny": 16, "small": 256, "large": 2048}[size]
    T = tuple(rng.choice([0, 1, rng.randint(1, cap), cap]) for _ in range(A))
    bucket = max(max(T), 1) if rng.random() < 0.3 else cap
    dtype = "fp8" if rng.random() < 0.25 else "bf16"
    mode = rng.choice([0, 0, 1, 2]) if K <= 8 else 0
    routing = "zipf" if rng.random() < 0.4 else "uniform"
    drop = rng.choice([0.0, 0.0, 0.1, 0.5])
    wl = W.Workload(f"fuzz{seed}", A=A, F=F, E=E, K=K, H=H, alpha=alpha, capacity=cap, bucket=bucket,
                    T=T, dtype=dtype, routing=routing, drop=drop, seed=1000 + seed)
    return wl, mode, rng.choice([0, 0, 5, 37]), rng.random() < 0.3


@pytest.mark.parametrize("seed", range(48))
def test_random_exchange_matches_oracle(seed):
    wl, mode, sms, rhc = _draw(seed)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE, combine_mode=mode)
    buf = GH.make_buffer(wl, num_sms=sms, combine_mode=mode)
    try:
        dev = GH.to_device(inp, transposed_scales=(seed % 2 == 1))
        recvs, replies, res = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, rhc=rhc,
                                              view=(wl.F == 1 and seed % 3 == 0))
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, rhc, buf)
        GH.check_outputs(wl, res, exp)
        assert buf.get_error()[0] == 0
        # the same IDs with new activations through a cached dispatch
        other = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 1}))
        new = W.Inputs(wl, inp.ids.copy(), inp.w.copy(), other.x.copy(),
                       None if other.x_scales is None else other.x_scales.copy())
        exp2 = GH.expected(new, GH.SCALE, combine_mode=mode)
        dev2 = GH.to_device(new)
        for s in range(wl.A):
            buf.source_dispatch_cached(s, dev2.x[s], None, dev2.scales[s], bucket=wl.bucket)
        recvs2 = {f: buf.worker_receive(f, bucket=wl.bucket) for f in range(wl.F)}
        replies2 = {f: GH.expert_reply(wl, f, recvs2[f], GH.SCALE) for f in range(wl.F)}
        for f in range(wl.F):
            buf.worker_reply(f, replies2[f], recvs2[f].receipt)
        res2 = buf.source_collect_all(outs=GH.alloc_outs(wl))
        torch.cuda.synchronize()
        GH.check_outputs(wl, res2, exp2)
    finally:
        buf.close()


def _draw_large(seed: int):
    rng = random.Random(7000 + seed)
    F = rng.choice([1, 2, 3, 4])
    E = F * rng.choice([16, 32, 64])
    K = rng.choice([4, 6, 8])
    A = rng.randint(1, 3)
    H = rng.choice([2048, 4096])
    T = tuple(rng.choice([rng.randint(600, 2048), 2048]) for _ in range(A))
    dtype = "fp8" if rng.random() < 0.3 else "bf16"
    mode = rng.choice([0, 0, 1, 2])
    wl = W.Workload(f"fuzz-large{seed}", A=A, F=F, E=E, K=K, H=H, alpha=rng.choice([1, 64, 128]),
                    capacity=2048, bucket=2048, T=T, dtype=dtype,
                    routing=rng.choice(["uniform", "zipf"]), drop=rng.choice([0.0, 0.1]), seed=2000 + seed)
    return wl, mode


@pytest.mark.parametrize("seed", range(6))
def test_random_large_exchange_matches_oracle(seed):
    """Production-sized random exchanges (H 2048 or 4096, 600-2048 tokens per
    source): the cluster layout, the scatter and the per-token combine."""
    wl, mode = _draw_large(seed)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE, combine_mode=mode)
    buf = GH.make_buffer(wl, combine_mode=mode)
    try:
        recvs, replies, res = GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, res, exp)
    finally:
        buf.close()


def _draw_wide(seed: int):
    """Wider draws: up to 64 sources and workers, 1,024 experts, top-32, rows
    past the bulk-copy limit (H 8448: 16.5 KB), alignment that is not a power
    of two, every slot dropped, sources dispatched and workers served in a
    shuffled order."""
    rng = random.Random(90000 + seed)
    F = rng.choice([1, 1, 2, 2, 3, 4, 5, 8, 16, 64])
    E = min(F * rng.choice([1, 2, 3, 4, 8, 16, 32, 64, 128]), 1024)
    E -= E % F
    K = rng.randint(1, min(E, rng.choice([8, 8, 16, 32])))
    A = rng.choice([1, 1, 2, 2, 3, 4, 8, rng.randint(1, 64)])
    dtype = "fp8" if rng.random() < 0.25 else "bf16"
    H = rng.choice([256, 512, 1280, 2048, 2304, 4096, 7168, 8192, 8448])
    cap = rng.choice([1, 16, 33, 256, 700, 2048])
    while A * cap * K * H > 2048 * 8 * 4096 * 2 and cap > 1:  # bounds the oracle's work
        cap //= 2
    T = tuple(rng.choice([0, 1, rng.randint(1, cap), cap]) for _ in range(A))
    bucket = max(max(T), 1) if rng.random() < 0.3 else cap
    alpha = rng.choice([1, 2, 3, 7, 16, 64, 128, 256])
    mode = rng.choice([0, 0, 1, 2]) if K <= 8 else 0
    routing = "zipf" if rng.random() < 0.4 else "uniform"
    drop = rng.choice([0.0, 0.0, 0.1, 0.5, 1.0])
    wl = W.Workload(f"wide{seed}", A=A, F=F, E=E, K=K, H=H, alpha=alpha, capacity=cap, bucket=bucket, T=T,
                    dtype=dtype, routing=routing, drop=drop, seed=50000 + seed)
    sms = rng.choice([0, 0, 0, 1, 5, 37, 151])
    rhc = rng.random() < 0.2
    sources, workers = list(range(A)), list(range(F))
    rng.shuffle(sources)
    rng.shuffle(workers)
    return wl, mode, sms, rhc, sources, workers, rng.random() < 0.3, rng.random() < 0.5


@pytest.mark.parametrize("seed", range(64))
def test_random_wide_exchange_matches_oracle(seed):
    wl, mode, sms, rhc, sources, workers, collect_all, transposed = _draw_wide(seed)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE, combine_mode=mode)
    buf = GH.make_buffer(wl, num_sms=sms, combine_mode=mode)
    try:
        dev = GH.to_device(inp, transposed_scales=transposed)
        if collect_all:
            for s in sources:
                buf.source_dispatch(s, dev.x[s], dev.ids[s], dev.w[s], dev.scales[s], bucket=wl.bucket,
                                    read_host_counts=rhc)
            recvs = {f: buf.worker_receive(f, bucket=wl.bucket, read_host_counts=rhc) for f in workers}
            replies = {}  # the reply rows stay alive until the combine has read them
            for f in workers:
                replies[f] = GH.expert_reply(wl, f, recvs[f], GH.SCALE)
                buf.worker_reply(f, replies[f], recvs[f].receipt)
            res = buf.source_collect_all(outs=GH.alloc_outs(wl))
        else:
            recvs, _, res = GH.run_exchange(buf, wl, dev, mode=GH.SCALE, rhc=rhc,
                                            view=(wl.F == 1 and seed % 3 == 0), source_order=sources,
                                            worker_order=workers)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, rhc, buf)
        GH.check_outputs(wl, res, exp)
        assert buf.get_error()[0] == 0
        if seed % 3 == 1:  # the same exchange captured in a graph, replayed on new inputs
            outs = GH.alloc_outs(wl)
            g = torch.cuda.CUDAGraph()
            held = {}
            with torch.cuda.graph(g):
                held["recvs"], held["replies"], held["res"] = GH.run_exchange(
                    buf, wl, dev, mode=GH.SCALE, outs=outs, source_order=sources, worker_order=workers)
            for rep in range(2):
                new = W.make_inputs(W.Workload(**{**wl.__dict__, "seed": wl.seed + 17 * (rep + 1)}))
                GH.refresh_device(dev, new)
                g.replay()
                torch.cuda.synchronize()
                exp2 = GH.expected(new, GH.SCALE, combine_mode=mode)
                GH.check_layout(wl, GH.snapshot(held["recvs"]), exp2, False, buf)
                GH.check_outputs(wl, held["res"], exp2)
            del g
    finally:
        buf.close()
