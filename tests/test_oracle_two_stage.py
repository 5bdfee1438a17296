"""Pins for the oracle's two-stage combine and its FP8 partials (afdEP-comm
design page, sections 6 and 19): the E4M3 encoder, the per-group power-of-two
exponent, the error bound the page states, equality with the fused combine for
one worker, an exact-rational brute force, and a hand-built case in which the
page's summation order (each worker's last route, ascending) matters."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact
import oracle
from combine_attention_ffn_gb300 import workloads as W


# ------------------------------------------------------------- E4M3 encoding
def _e4m3_values():
    """Finite non-negative E4M3 values by code, from the format definition."""
    vals = {}
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals[code] = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return vals


E4M3 = _e4m3_values()


def e4m3_encode_exact(x: float) -> int:
    """Nearest E4M3 value, ties to the even code; saturating at 448."""
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a >= 448:
        return sign | 0x7E
    q = Fraction(a)
    best = min(E4M3, key=lambda c: (abs(E4M3[c] - q), c & 1))
    return sign | best


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 30,
                        rng.standard_normal(50000).astype(np.float32) * 0.01,
                        np.array([0.0, -0.0, 448.0, -448.0, 2 ** -9, 2 ** -10, 3 * 2 ** -10, 2 ** -6], np.float32)])
    x = x[np.abs(x) <= 448]
    got = orc.float_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_encode_ties_and_saturation(orc):
    cases = {2 ** -10: 0x00, 3 * 2 ** -10: 0x02, 448.0: 0x7E, 460.0: 0x7E, 464.0: 0x7E, 1e9: 0x7E,
             float("inf"): 0x7E, float("-inf"): 0xFE, -1.0: 0xB8, 240.0: 0x77, 248.0: 0x78,
             1.0 + 2 ** -4: 0x38, 1.0 + 3 * 2 ** -4: 0x3A}
    x = np.array(list(cases), np.float32)
    got = orc.float_to_e4m3(x).tolist()
    assert got == list(cases.values())
    assert orc.float_to_e4m3(np.array([float("nan")], np.float32))[0] & 0x7F == 0x7F


def test_e4m3_encode_matches_exact_restatement(orc):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(3000) * 60).astype(np.float32)
    got = orc.float_to_e4m3(x)
    for v, g in zip(x.tolist(), got.tolist()):
        assert g == e4m3_encode_exact(v), v


# ------------------------------------------------------- group exponent
def group_exponent_exact(amax: float) -> int:
    """Smallest integer e >= -117 with amax <= 448 * 2^e (exact); the page
    states that an infinite group gets 2^120."""
    if math.isinf(amax):
        return 120
    e = -117
    while Fraction(amax) > 448 * Fraction(2) ** e:
        e += 1
    return e


def test_group_exponent_hand_cases(orc):
    f32 = np.float32
    nxt = np.nextafter(f32(448), f32(1e9))
    cases = [(448.0, 0), (float(nxt), 1), (224.0, -1), (224.0001, 0), (0.0, -117), (1e-40, -117),
             (float("inf"), 120), (248.0 * 2.0 ** 120, 120), (1.0, -8), (1.75, -8), (1.7500001, -7)]
    got = orc.group_exponent(np.array([c[0] for c in cases], np.float32)).tolist()
    assert got == [c[1] for c in cases]


def test_group_exponent_matches_exact_definition(orc):
    rng = np.random.default_rng(3)
    amax = np.abs(rng.standard_normal(4000) * np.exp2(rng.integers(-60, 60, 4000))).astype(np.float32)
    got = orc.group_exponent(amax)
    for a, g in zip(amax.tolist(), got.tolist()):
        assert g == group_exponent_exact(a), a


def test_fp8_partial_error_bound(orc):
    """design page section 19: an element's error stays within 2^-4 times the
    largest magnitude of its 128-element group."""
    rng = np.random.default_rng(4)
    groups = (rng.standard_normal((500, 128)) * np.exp2(rng.integers(-20, 20, (500, 1)))).astype(np.float32)
    groups = torch.from_numpy(groups).to(torch.bfloat16).float().numpy()
    amax = np.abs(groups).max(axis=1)
    e = orc.group_exponent(amax)
    q = orc.float_to_e4m3((groups * np.exp2(-e[:, None].astype(np.float64))).astype(np.float32))
    deq = orc.e4m3_to_float(q).astype(np.float64) * np.exp2(e[:, None].astype(np.float64))
    assert np.all(np.abs(deq - groups) <= amax[:, None] * 2.0 ** -4)


# ------------------------------------------------------- two-stage combine
def _prob(wl):
    return oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, oracle.BF16, wl.T)


@pytest.mark.parametrize("name,T", [("skew-3A1F", 32), ("tiny", None)])
def test_two_stage_bf16_equals_fused_for_one_worker(name, T):
    wl = W.named(name, T=T)
    wl = W.Workload(**{**wl.__dict__, "F": 1})
    inp = W.make_inputs(wl)
    p = _prob(wl)
    fused = oracle.round_trip(p, inp.ids, inp.w, inp.x, expert_mode=oracle.EXPERT_SCALE)
    two = oracle.round_trip(p, inp.ids, inp.w, inp.x, expert_mode=oracle.EXPERT_SCALE,
                            combine_mode=oracle.COMBINE_TWO_STAGE)
    assert np.array_equal(fused["out"], two["out"])


def _bf16f(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).float().numpy()


def _two_stage_exact(ids, w, slot, reply, Ef, T, fp8):
    """Exact-rational restatement of the two-stage combine."""
    A, B, K = ids.shape
    H = reply.shape[-1]
    out = np.zeros((A, B, H), np.uint16)
    rf = _bf16f(reply)
    for s in range(A):
        for t in range(T[s]):
            valid = [k for k in range(K) if slot[s, t, k] >= 0]
            worker = {k: int(ids[s, t, k]) // Ef for k in valid}
            order = [k for k in valid if all(worker[j] != worker[k] for j in valid if j > k)]
            acc = [Fraction(0)] * H
            for k in order:
                f = worker[k]
                part = []
                for h in range(H):
                    a = Fraction(0)
                    for j in valid:
                        if j <= k and worker[j] == f:
                            a = exact.round_f32(Fraction(float(w[s, t, j])) * Fraction(float(rf[f, slot[s, t, j], h])) + a)
                    part.append(exact.round_bf16(a))
                if fp8:
                    for g in range(H // 128):
                        amax = max(abs(x) for x in part[g * 128:(g + 1) * 128])
                        e = group_exponent_exact(float(amax))
                        for h in range(g * 128, (g + 1) * 128):
                            code = e4m3_encode_exact(float(part[h] / Fraction(2) ** e))
                            v = E4M3[code & 0x7F] * (-1 if code & 0x80 else 1)
                            part[h] = v * Fraction(2) ** e
                acc = [exact.round_f32(a + b) for a, b in zip(acc, part)]
            for h in range(H):
                out[s, t, h] = exact.bf16_bits(exact.round_bf16(acc[h]))
    return out


@pytest.mark.parametrize("fp8", [False, True])
def test_two_stage_brute_force_exact_rational(fp8):
    rng = np.random.default_rng(5 + fp8)
    A, B, K, E, F, H = 2, 3, 6, 12, 3, 128
    ids = np.stack([np.stack([rng.permutation(E)[:K] for _ in range(B)]) for _ in range(A)]).astype(np.int64)
    ids[rng.random(ids.shape) < 0.2] = -1
    w = (rng.random((A, B, K)) * 1.5).astype(np.float32)
    xf = (rng.standard_normal((A, B, H)) * 4).astype(np.float32)
    x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    T = [3, 2]
    p = oracle.Problem(A, F, E, K, H, 2, B, oracle.BF16, T)
    r = oracle.round_trip(p, ids, w, x, expert_mode=oracle.EXPERT_SCALE,
                          combine_mode=oracle.COMBINE_TWO_STAGE_FP8 if fp8 else oracle.COMBINE_TWO_STAGE)
    want = _two_stage_exact(ids, w, r["slot"], r["reply"], E // F, T, fp8)
    for s in range(A):
        assert np.array_equal(r["out"][s, :T[s]], want[s, :T[s]])


def crafted_order_case():
    """Four workers of two experts each; one token's routes k = 0..4 go to
    workers 0, 2, 3, 1, 0 with partials 1, 2^-24, 2^-24, 2^-8 (the last route
    has weight 0). Summed in the order of each worker's last route (2, 3, 1,
    0) the FP32 result is 1 + 2^-8 + 2^-23 -> BF16 0x3F81; in ascending worker
    order it is 1 + 2^-8 -> 0x3F80; the fused chain gives 0x3F80 too."""
    ids = np.array([[[0, 4, 6, 2, 1]]], np.int64)
    w = np.array([[[1.0, 1.0, 1.0, 1.0, 0.0]]], np.float32)
    vals = [1.0, 2.0 ** -24, 2.0 ** -24, 2.0 ** -8, 1.0]
    return ids, w, vals


def test_two_stage_crafted_order():
    ids, w, vals = crafted_order_case()
    H = 128
    p = oracle.Problem(1, 4, 8, 5, H, 1, 1, oracle.BF16, [1])
    x = np.zeros((1, 1, H), np.uint16)
    lay = oracle.layout(p, ids)
    r_stride = int(lay["r_exact"].max())
    d = oracle.dispatch(p, ids, w, x, None, lay, r_stride)
    reply = np.zeros((4, r_stride, H), np.uint16)
    for k in range(5):
        f = int(ids[0, 0, k]) // 2
        reply[f, d["slot"][0, 0, k], :] = np.float32(vals[k]).view(np.uint32) >> 16
    two = oracle.combine_two_stage(p, ids, w, d["slot"], r_stride, reply, fp8=False)
    fused = oracle.combine(p, ids, w, d["slot"], r_stride, reply)
    assert np.all(two[0, 0] == 0x3F81)
    assert np.all(fused[0, 0] == 0x3F80)


# Worker 0's partial is -1.5 * 2^127 (BF16 0xFF40, exact in E4M3 with scale
# 2^119); worker 1's partial is v. The design page (section 19, "Accuracy")
# says a group amax of 248 * 2^120 or more decodes to infinity (the top BF16
# binade is not representable): with scale 2^120, 248 is the tie between the
# E4M3 values 240 and 256 and goes to the even code, 256, and 256 * 2^120 is
# beyond the FP32 range. Below it the partial decodes to 240 * 2^120.
#   v >= 248 * 2^120: -1.5 * 2^127 + inf = inf                  -> 0x7F80
#   v in (232, 248) * 2^120: -1.5 * 2^127 + 1.875 * 2^127 = 1.5 * 2^125 -> 0x7E40
# Decoding exactly and rounding only the sum (2^128 - 1.5 * 2^127 = 2^126,
# 0x7E80) is the reading this rules out.
TOP_BINADE_CASES = {0x7F78: 0x7F80, 0x7F7F: 0x7F80, 0x7F76: 0x7E40, 0x7F70: 0x7E40}
TOP_BINADE_OTHER = 0xFF40


def top_binade_outputs(orc=None):
    """{v: (FP8-partials output word, BF16-partials output word)} for the
    top-binade token above, as the oracle computes them."""
    H = 128
    ids = np.array([[[0, 2]]], np.int64)  # experts 0 and 2: workers 0 and 1
    w = np.ones((1, 1, 2), np.float32)
    p = oracle.Problem(1, 2, 4, 2, H, 1, 1, oracle.BF16, [1])
    lay = oracle.layout(p, ids, orc)
    r_stride = int(lay["r_exact"].max())
    d = oracle.dispatch(p, ids, w, np.zeros((1, 1, H), np.uint16), None, lay, r_stride, orc)
    res = {}
    for v in TOP_BINADE_CASES:
        reply = np.zeros((2, r_stride, H), np.uint16)
        reply[0, d["slot"][0, 0, 0], :] = TOP_BINADE_OTHER
        reply[1, d["slot"][0, 0, 1], :] = v
        words = []
        for fp8 in (True, False):
            out = oracle.combine_two_stage(p, ids, w, d["slot"], r_stride, reply, fp8, orc)
            assert np.all(out[0, 0] == out[0, 0, 0])
            words.append(int(out[0, 0, 0]))
        res[v] = tuple(words)
    return res


def test_two_stage_fp8_top_binade_decodes_to_infinity():
    got = top_binade_outputs()
    for v, want in TOP_BINADE_CASES.items():
        assert got[v][0] == want, (hex(v), hex(got[v][0]))
        # with BF16 partials nothing overflows: (v - 1.5 * 2^127) rounded to BF16
        vf = float(np.uint32(v << 16).view(np.float32))
        assert got[v][1] == exact.bf16_bits(exact.round_bf16(Fraction(vf) - Fraction(3, 2) * Fraction(2) ** 127))
