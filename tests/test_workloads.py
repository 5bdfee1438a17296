"""The seeded input generator produces what its recipe states (CPU only)."""
import numpy as np
import pytest
import torch

from combine_attention_ffn_gb300 import workloads as W


@pytest.mark.parametrize("name", ["tiny", "2A2F", "2A2F-H4096", "skew-3A1F", "skew-1A3F", "fp8-2A2F", "fp8-2A1F"])
def test_shapes_padding_and_determinism(name):
    wl = W.named(name, T=None if name == "tiny" else 64)
    a, b = W.make_inputs(wl), W.make_inputs(wl)
    for x, y in ((a.ids, b.ids), (a.w, b.w), (a.x, b.x)):
        assert np.array_equal(x, y)
    assert a.ids.shape == (wl.A, wl.bucket, wl.K) and a.w.shape == (wl.A, wl.bucket, wl.K)
    assert a.x.shape == (wl.A, wl.bucket, wl.H)
    for s, T in enumerate(wl.T):
        assert np.all(a.ids[s, T:] == -1) and np.all(a.w[s, T:] == 0)
        live = a.ids[s, :T]
        assert np.all((live >= -1) & (live < wl.E))
        for row in live:  # distinct experts per token
            v = row[row >= 0]
            assert len(set(v.tolist())) == len(v)
        # softmax over all K slots, taken before any slot is dropped
        assert np.allclose(a.w[s, :T].astype(np.float64).sum(-1), 1.0, atol=1e-6)


def test_uniform_routing_has_no_drops_and_is_roughly_uniform():
    wl = W.named("2A2F", T=2048)
    ids = W.make_inputs(wl).ids
    assert np.all(ids >= 0)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    expect = ids.size / wl.E
    assert counts.min() > 0.8 * expect and counts.max() < 1.2 * expect


def test_skew_routing_popularity_and_drops():
    wl = W.named("skew-3A1F", T=2048)
    ids = W.make_inputs(wl).ids
    drop = (ids == -1).mean()
    assert 0.08 < drop < 0.12                                  # 10% of slots set to -1
    counts = np.bincount(ids[ids >= 0], minlength=wl.E)
    assert counts[0] == counts.max()                           # expert 0 is the most popular
    assert counts[:8].sum() > counts[-64:].sum()               # heavy head
    assert np.all(np.diff(counts[:4]) <= 0)                    # popularity falls with the rank


def test_a_different_seed_gives_different_routing():
    wl = W.named("2A2F", T=64)
    other = W.Workload(**{**wl.__dict__, "seed": wl.seed + 1})
    assert not np.array_equal(W.make_inputs(wl).ids, W.make_inputs(other).ids)


def test_fp8_scales_are_absmax_over_448():
    wl = W.named("fp8-2A2F", T=32)
    inp = W.make_inputs(wl)
    q = torch.from_numpy(inp.x[0, :32].copy()).view(torch.float8_e4m3fn).float().numpy()
    deq = q.reshape(32, wl.H // 128, 128) * inp.x_scales[0, :32, :, None]
    amax_q = np.abs(q.reshape(32, wl.H // 128, 128)).max(-1)
    assert np.all(amax_q <= 448) and np.all(amax_q >= 400)      # the block maximum maps near 448
    assert np.all(inp.x_scales[0, :32] > 0) and np.isfinite(deq).all()


def test_bf16_activations_are_standard_normal():
    x = W.make_inputs(W.named("2A2F", T=512)).x[:, :512]
    xf = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert abs(xf.mean()) < 0.01 and abs(xf.std() - 1.0) < 0.01
