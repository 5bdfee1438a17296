"""Pins for the oracle's combine and the harness expert.

Closed forms (identity expert: K=1 gives back x; K=8 with weights 1/8 gives
back x exactly), the weight-applied-once check, the +0 row of a token without
routes, and an exact-rational brute force of the FP32 fused-multiply-add chain
and its single BF16 rounding on small inputs (tests/exact.py, independent of
the oracle's C code).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact
import oracle
from combine_attention_ffn_gb300 import workloads as W


def _bf16_float(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float().numpy()


def _rand_bf16(rng, shape, scale=1.0):
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _uniform_ids(rng, A, B, K, E):
    return np.stack([np.stack([rng.permutation(E)[:K] for _ in range(B)]) for _ in range(A)]).astype(np.int64)


def test_k1_unit_weight_identity_is_permutation_round_trip():
    rng = np.random.default_rng(0)
    A, B, K, E, F, H = 2, 24, 1, 16, 4, 256
    ids = _uniform_ids(rng, A, B, K, E)
    w = np.ones((A, B, K), np.float32)
    x = _rand_bf16(rng, (A, B, H))
    p = oracle.Problem(A, F, E, K, H, 8, B, oracle.BF16, [B, B - 5])
    r = oracle.round_trip(p, ids, w, x)
    assert np.array_equal(r["out"][0], x[0])
    assert np.array_equal(r["out"][1, : B - 5], x[1, : B - 5])


def test_k8_eighth_weights_identity_is_exact():
    # every partial sum j * x / 8 of a BF16 x is exact in FP32, so the single
    # rounding at the end gives x back bit for bit
    rng = np.random.default_rng(1)
    A, B, K, E, F, H = 2, 16, 8, 64, 2, 256
    ids = _uniform_ids(rng, A, B, K, E)
    w = np.full((A, B, K), 0.125, np.float32)
    x = _rand_bf16(rng, (A, B, H), scale=3.0)
    p = oracle.Problem(A, F, E, K, H, 4, B, oracle.BF16, [B, B])
    r = oracle.round_trip(p, ids, w, x)
    assert np.array_equal(r["out"], x)


def test_weight_applied_exactly_once():
    # identity expert, weights 0.25 and 0.5: x * sum(w) = 0.75 x, distinct from
    # x * sum(w^2) = 0.3125 x and from K * x = 2 x
    rng = np.random.default_rng(2)
    A, B, K, E, F, H = 1, 8, 2, 8, 2, 128
    ids = _uniform_ids(rng, A, B, K, E)
    w = np.tile(np.array([0.25, 0.5], np.float32), (A, B, 1))
    x = _rand_bf16(rng, (A, B, H))
    p = oracle.Problem(A, F, E, K, H, 1, B, oracle.BF16, [B])
    out = _bf16_float(oracle.round_trip(p, ids, w, x)["out"])
    xf = _bf16_float(x)
    want = torch.from_numpy(xf * np.float32(0.75)).to(torch.bfloat16).float().numpy()
    assert np.array_equal(out, want)
    assert not np.array_equal(out, xf * np.float32(0.3125))


def test_token_without_routes_is_positive_zero():
    rng = np.random.default_rng(3)
    A, B, K, E, F, H = 2, 6, 3, 12, 3, 256
    ids = _uniform_ids(rng, A, B, K, E)
    ids[0, 2] = -1
    ids[1, 5] = -1
    w = rng.random((A, B, K)).astype(np.float32)
    x = _rand_bf16(rng, (A, B, H))
    p = oracle.Problem(A, F, E, K, H, 2, B, oracle.BF16, [B, B])
    out = oracle.round_trip(p, ids, w, x)["out"]
    assert np.all(out[0, 2] == 0) and np.all(out[1, 5] == 0)
    assert np.any(out[0, 1] != 0)


def _exact_combine(ids, w, x_bits, T, F, E, expert_c):
    """Exact-rational restatement: acc_0 = 0, acc_{j+1} = round_f32(w_k r_k +
    acc_j) for the valid routes in ascending k, out = round_bf16(acc)."""
    A, B, K = ids.shape
    H = x_bits.shape[-1]
    out = np.zeros((A, B, H), np.uint16)
    xf = _bf16_float(x_bits)
    for s in range(A):
        for t in range(T[s]):
            for h in range(H):
                acc = Fraction(0)
                for k in range(K):
                    e = int(ids[s, t, k])
                    if e < 0:
                        continue
                    r = exact.round_bf16(Fraction(float(xf[s, t, h])) * expert_c(e))
                    acc = exact.round_f32(Fraction(float(w[s, t, k])) * r + acc)
                out[s, t, h] = exact.bf16_bits(exact.round_bf16(acc))
    return out


@pytest.mark.parametrize("expert_mode", [oracle.EXPERT_IDENTITY, oracle.EXPERT_SCALE])
def test_combine_brute_force_exact_rational(expert_mode):
    rng = np.random.default_rng(4 + expert_mode)
    A, B, K, E, F, H = 2, 3, 5, 12, 3, 128
    ids = _uniform_ids(rng, A, B, K, E)
    ids[rng.random(ids.shape) < 0.25] = -1
    # weights with full 24-bit significands so products round
    w = (rng.random((A, B, K)) * 1.7).astype(np.float32)
    x = _rand_bf16(rng, (A, B, H), scale=5.0)
    T = [3, 2]
    p = oracle.Problem(A, F, E, K, H, 4, B, oracle.BF16, T)
    r = oracle.round_trip(p, ids, w, x, expert_mode=expert_mode)

    def c(e):
        return Fraction(2) ** ((e % 4) - 1) if expert_mode == oracle.EXPERT_SCALE else Fraction(1)

    want = _exact_combine(ids, w, x, T, F, E, c)
    for s in range(A):
        assert np.array_equal(r["out"][s, : T[s]], want[s, : T[s]])


def test_combine_crafted_fused_ascending_chain():
    """A hand-built element on which the result depends on both the fusion and
    the order of the FP32 chain.

    route 0: w = 1 + 2^-8, reply 1.0         -> acc = 1 + 2^-8 (a BF16 tie)
    route 1: w = 16647161 * 2^-24, reply (1 + 2^-7) * 2^-24
             w * reply = 2^-24 * (1 + 121 * 2^-31): just above 2^-24.
    Fused, ascending: 1 + 2^-8 + 2^-24 + tiny rounds up in FP32 to
    1 + 2^-8 + 2^-23, which is above the BF16 tie -> 0x3F81.
    A separately rounded product drops the tiny part, the FP32 sum lands on a
    tie and goes to even (1 + 2^-8), and BF16 then ties to even -> 0x3F80.
    Descending order gives 0x3F80 as well."""
    w = np.array([[[1.0 + 2.0 ** -8, 16647161 * 2.0 ** -24]]], np.float32)
    assert float(w[0, 0, 1]) == 16647161 * 2.0 ** -24
    ids = np.array([[[0, 1]]], np.int64)
    slot = np.array([[[0, 1]]], np.int32)
    H = 128
    reply = np.zeros((1, 2, H), np.uint16)
    reply[0, 0, :] = 0x3F80          # 1.0
    reply[0, 1, :] = 0x3381          # (1 + 2^-7) * 2^-24
    p = oracle.Problem(1, 1, 2, 2, H, 1, 1, oracle.BF16, [1])
    out = oracle.combine(p, ids, w, slot, 2, reply)
    assert np.all(out[0, 0] == 0x3F81)

    r = [Fraction(1), exact.f32_bits_to_fraction(0x33810000)]
    wf = [Fraction(float(v)) for v in w[0, 0]]
    fused = Fraction(0)
    for k in (0, 1):
        fused = exact.round_f32(wf[k] * r[k] + fused)
    assert exact.bf16_bits(exact.round_bf16(fused)) == 0x3F81
    unfused = Fraction(0)
    for k in (0, 1):
        unfused = exact.round_f32(exact.round_f32(wf[k] * r[k]) + unfused)
    assert exact.bf16_bits(exact.round_bf16(unfused)) == 0x3F80
    desc = Fraction(0)
    for k in (1, 0):
        desc = exact.round_f32(wf[k] * r[k] + desc)
    assert exact.bf16_bits(exact.round_bf16(desc)) == 0x3F80


def test_expert_scale_matches_torch():
    wl = W.named("2A2F", T=8)
    inp = W.make_inputs(wl)
    p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, oracle.BF16, wl.T)
    r = oracle.round_trip(p, inp.ids, inp.w, inp.x, expert_mode=oracle.EXPERT_SCALE)
    Ef = wl.E // wl.F
    for f in range(wl.F):
        for l in range(Ef):
            e = f * Ef + l
            lo, hi = r["start"][f, l], r["ends"][f, l]
            rows = torch.from_numpy(r["rows"][f, lo:hi].view(np.int16)).view(torch.bfloat16)
            want = (rows.float() * 2.0 ** ((e % 4) - 1)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(r["reply"][f, lo:hi].view(np.int16), want)


def test_expert_fp8_matches_torch():
    wl = W.named("fp8-2A2F", T=8)
    inp = W.make_inputs(wl)
    p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, oracle.FP8, wl.T)
    r = oracle.round_trip(p, inp.ids, inp.w, inp.x, inp.x_scales, expert_mode=oracle.EXPERT_SCALE)
    Ef = wl.E // wl.F
    for f in range(wl.F):
        for l in range(Ef):
            e = f * Ef + l
            lo, hi = r["start"][f, l], r["ends"][f, l]
            q = torch.from_numpy(r["rows"][f, lo:hi]).view(torch.float8_e4m3fn).float()
            sc = torch.from_numpy(r["row_scales"][f, lo:hi]).repeat_interleave(128, dim=1)
            want = ((q * sc) * 2.0 ** ((e % 4) - 1)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(r["reply"][f, lo:hi].view(np.int16), want)


@pytest.mark.parametrize("name,T", [("2A2F", 64), ("skew-3A1F", 32), ("skew-1A3F", 32)])
def test_softmax_identity_within_one_ulp_of_x_sum_w(name, T):
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, oracle.BF16, wl.T)
    r = oracle.round_trip(p, inp.ids, inp.w, inp.x, expert_mode=oracle.EXPERT_IDENTITY)
    xf = _bf16_float(inp.x).astype(np.float64)
    sw = np.where(inp.ids >= 0, inp.w, 0).astype(np.float64).sum(-1)
    ref = xf * sw[..., None]
    out = _bf16_float(r["out"]).astype(np.float64)
    for s in range(wl.A):
        o, rf = out[s, : wl.T[s]], ref[s, : wl.T[s]]
        ulp = np.maximum(np.abs(rf), 2.0 ** -126) * 2.0 ** -7
        assert np.all(np.abs(o - rf) <= ulp * 1.01)
