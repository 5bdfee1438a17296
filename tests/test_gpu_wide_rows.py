"""Wide rows: BF16 rows of 14 and 16 KB (16 KB is the widest the bulk-copy
scatter takes) and FP8 rows of 8 KB go through the bulk scatter with large
shared-memory buffers; BF16 rows of 32 KB go through the register scatter
(16-byte vector copies) and, for a cached dispatch, the register cached
scatter. Ragged multi-source batches (one source empty) exercise the
scatter's source order (last source first). Every result is compared with
the oracle bit for bit."""
import pytest
import torch

import gpu_harness as GH
import test_gpu_cached as TC
from combine_attention_ffn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from combine_attention_ffn_gb300 import build

    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no GPU")


WIDE = [
    W.Workload("3A2F-H8192", A=3, F=2, E=64, K=4, H=8192, alpha=16, capacity=1024, bucket=1024,
               T=(300, 0, 513), routing="zipf", drop=0.1, seed=1201),
    W.Workload("2A2F-H7168", A=2, F=2, E=64, K=8, H=7168, alpha=8, capacity=512, bucket=512,
               T=(512, 77), seed=1202),
    W.Workload("fp8-3A2F-H8192", A=3, F=2, E=64, K=4, H=8192, alpha=16, capacity=1024, bucket=1024,
               T=(257, 640, 0), dtype="fp8", seed=1203),
    W.Workload("3A2F-H16384", A=3, F=2, E=32, K=4, H=16384, alpha=4, capacity=256, bucket=256,
               T=(256, 131, 0), seed=1204),
]


@pytest.mark.parametrize("wl", WIDE, ids=lambda w: w.name)
def test_wide_rows_match_oracle(wl):
    inp = W.make_inputs(wl)
    exp = GH.expected(inp, GH.SCALE)
    buf = GH.make_buffer(wl)
    try:
        recvs, _, results = GH.run_exchange(buf, wl, GH.to_device(inp), mode=GH.SCALE)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp, False, buf)
        GH.check_outputs(wl, results, exp)
        # the cached dispatch of the same routing, new activations and weights
        new = TC._fresh_values(inp, wl.seed + 11, True)
        exp2 = GH.expected(new, GH.SCALE)
        recvs, _, res = TC._cached_exchange(buf, wl, GH.to_device(new), True, GH.SCALE)
        torch.cuda.synchronize()
        GH.check_layout(wl, GH.snapshot(recvs), exp2, False, buf)
        GH.check_outputs(wl, res, exp2)
    finally:
        buf.close()
