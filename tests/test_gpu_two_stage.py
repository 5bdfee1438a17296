"""The two-stage combine modes (per-worker BF16 partials, optionally FP8
partials with one power-of-two factor shared by each block of 128 values) against the oracle, bit
for bit."""
import numpy as np
import pytest
import torch

import gpu_harness as GH
import oracle
import test_oracle_two_stage as TS
from combine_attention_ffn_gb300 import afd
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


MODES = [afd.COMBINE_TWO_STAGE, afd.COMBINE_TWO_STAGE_FP8]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,T", [("tiny", None), ("2A2F", 1), ("2A2F", 128), ("2A2F", 2048),
                                    ("2A2F-H4096", 128), ("skew-1A3F", 512), ("skew-3A1F", 64),
                                    ("fp8-2A2F", 128),
                                    # per-token kernels (at least 8 tokens per SM)
                                    ("2A2F-H4096", 2048), ("skew-1A3F", 2048), ("skew-3A1F", 2048),
                                    ("fp8-2A2F", 2048)])
def test_two_stage_matches_oracle(mode, name, T):
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE, combine_mode=mode)
    buf = GH.make_buffer(wl, combine_mode=mode)
    try:
        recvs, _, results = GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
    finally:
        buf.close()


def test_two_stage_single_worker_equals_fused():
    wl = W.named("skew-3A1F", T=256)
    inp = W.make_inputs(wl)
    outs = {}
    for mode in (afd.COMBINE_FUSED, afd.COMBINE_TWO_STAGE):
        buf = GH.make_buffer(wl, combine_mode=mode)
        try:
            _, _, res = GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
            outs[mode] = [GH.out_bits(r) for r in res]
        finally:
            buf.close()
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)


def test_two_stage_crafted_order_on_gpu():
    """The hand-built token whose BF16 result depends on summing the workers'
    partials in the order of their last routes: 0x3F81 (fused gives 0x3F80)."""
    ids, w, vals = TS.crafted_order_case()
    H = 256
    for mode, want in ((afd.COMBINE_TWO_STAGE, 0x3F81), (afd.COMBINE_FUSED, 0x3F80)):
        buf = afd.Buffer(1, 4, 8, 5, H, 1, 1, "bf16", combine_mode=mode)
        try:
            x = torch.zeros((1, H), dtype=torch.bfloat16, device="cuda")
            buf.source_dispatch(0, x, torch.from_numpy(ids[0]).cuda(), torch.from_numpy(w[0]).cuda(), bucket=1)
            recvs = [buf.worker_receive(f, bucket=1) for f in range(4)]
            replies = []
            row_src = [r.row_src.cpu().numpy() for r in recvs]
            for f in range(4):
                rep = torch.zeros((recvs[f].num_rows, H), dtype=torch.int16)
                for row, src in enumerate(row_src[f]):
                    if src >= 0:
                        rep[row] = int(np.float32(vals[src % 5]).view(np.uint32) >> 16)
                replies.append(rep.cuda().view(torch.bfloat16))
                buf.worker_reply(f, replies[f], recvs[f].receipt)
            out = buf.source_collect(0, num_tokens=1)
            assert torch.all(out.view(torch.int16) == want), mode
        finally:
            buf.close()


def test_two_stage_rejects_large_top_k():
    with pytest.raises(afd.AfdError) as ei:
        afd.Buffer(2, 2, 64, 9, 256, 16, 1, "bf16", combine_mode=afd.COMBINE_TWO_STAGE)
    assert ei.value.status == afd.ERR_UNSUPPORTED


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("F,T", [(8, 300), (16, 1024), (64, 700)])
def test_two_stage_many_workers(mode, F, T):
    """Many workers: a token's eight routes fall on up to eight workers, in
    any interleaving, so the per-token regrouping into summation order has up
    to eight runs; 300 tokens per source take the segmented kernel, 1,024 and
    700 the per-token one."""
    wl = W.Workload(f"2A{F}F", A=2, F=F, E=128, K=8, H=512, alpha=4, capacity=T, bucket=T,
                    T=(T, T // 2 + 1), routing="uniform" if F == 8 else "zipf", drop=0.1, seed=900 + F)
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE, combine_mode=mode)
    buf = GH.make_buffer(wl, combine_mode=mode)
    try:
        recvs, _, results = GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
    finally:
        buf.close()


@pytest.mark.parametrize("v,want", sorted(TS.TOP_BINADE_CASES.items()))
def test_two_stage_fp8_top_binade_on_gpu(v, want):
    """A worker partial in BF16's top binade: from a group amax of 248 * 2^120
    the decoded partial is infinite (design page, section 19, "Accuracy"), so
    the sum is too; the oracle's pin gives the same bits."""
    H = 256
    buf = afd.Buffer(1, 2, 4, 2, H, 1, 1, "bf16", combine_mode=afd.COMBINE_TWO_STAGE_FP8)
    try:
        x = torch.zeros((1, H), dtype=torch.bfloat16, device="cuda")
        ids = torch.tensor([[0, 2]], dtype=torch.int64, device="cuda")
        w = torch.ones((1, 2), dtype=torch.float32, device="cuda")
        buf.source_dispatch(0, x, ids, w, bucket=1)
        recvs = [buf.worker_receive(f, bucket=1) for f in range(2)]
        replies = []
        for f in range(2):
            rep = torch.zeros((recvs[f].num_rows, H), dtype=torch.int32)
            for row, src in enumerate(recvs[f].row_src.cpu().tolist()):
                if src >= 0:
                    rep[row] = TS.TOP_BINADE_OTHER if src % 2 == 0 else v
            replies.append(rep.to(torch.int16).cuda().view(torch.bfloat16))
            buf.worker_reply(f, replies[f], recvs[f].receipt)
        out = buf.source_collect(0, num_tokens=1)
        torch.cuda.synchronize()
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.all(got == want), (hex(v), hex(int(got[0, 0])))
    finally:
        buf.close()
