"""Seeded random exchanges: shapes, routing skew, drops, alignment, worker
counts, dtypes, combine modes, SM caps and host-count modes drawn at random,
one exchange each (plus a cached dispatch and a second exchange on the same
context), every result compared with the oracle bit for bit. The draws cover
the one-warp, one-kernel and cluster dispatch paths and both combine kernels."""
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
