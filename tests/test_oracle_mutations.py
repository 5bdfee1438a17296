"""The pins must catch plausible mistakes in the oracle.

Each case copies ``oracle/orc.c`` to a temporary directory, plants one
mistake (a dropped term, a wrong sign, index or order, a transposed operand),
compiles it with the oracle's own flags, and runs a battery of the pins from
test_oracle_*.py against it. Every planted mistake must fail at least one pin,
and the unmodified source must pass them all. Nothing here touches a GPU.
"""
import json
import os
import shutil
import subprocess
import sys
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact
import oracle
import test_oracle_combine as TC
import test_oracle_layout as TL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SRC = os.path.join(os.path.dirname(oracle.__file__), "orc.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "orc.h")

MUTATIONS = {
    "unfused_multiply_add": ("acc = fmaf(w[ri], r, acc);", "acc = w[ri] * r + acc;"),
    "descending_k_in_combine": (
        "        for (int k = 0; k < p->K; ++k) {\n          int64_t ri = route_index(p, s, t, k);\n          if (slot[ri] < 0) continue;",
        "        for (int k = p->K - 1; k >= 0; --k) {\n          int64_t ri = route_index(p, s, t, k);\n          if (slot[ri] < 0) continue;"),
    "negative_zero_start": ("float acc = 0.0f;", "float acc = -0.0f;"),
    "start_not_aligned": ("start[i] = (int32_t)align_up(prev_end, p->alpha);", "start[i] = (int32_t)prev_end;"),
    "host_counts_raw": ("host_counts[i] = (int32_t)align_up(count[i], p->alpha);", "host_counts[i] = count[i];"),
    "r_exact_unaligned": ("r_exact[f] = align_up(prev_end, p->alpha);", "r_exact[f] = prev_end;"),
    "bf16_ties_away": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (dropped >= 0x8000u)"),
    "bf16_truncate": ("    kept += 1u;\n  return (uint16_t)kept;", "    kept += 0u;\n  return (uint16_t)kept;"),
    "e4m3_bias_8": ("v = ldexpf((float)(8 + m), e - 7 - 3);", "v = ldexpf((float)(8 + m), e - 8 - 3);"),
    "e4m3_subnormal_scale": ("v = ldexpf((float)m, -9);", "v = ldexpf((float)m, -10);"),
    "dup_self_compare": ("for (int j = 0; j < k; ++j)", "for (int j = 0; j <= k; ++j)"),
    "range_off_by_one": ("if (id < -1 || id >= p->E) return -ORC_ROUTE_RANGE;",
                         "if (id < -1 || id > p->E) return -ORC_ROUTE_RANGE;"),
    "row_src_transposed": ("row_src[f * r_stride + row] = (int32_t)ri;",
                           "row_src[f * r_stride + row] = (int32_t)(((int64_t)t * p->A + s) * p->K + k);"),
    "row_w_wrong_k": ("row_w[f * r_stride + row] = w[ri];",
                      "row_w[f * r_stride + row] = w[route_index(p, s, t, (k + 1) % p->K)];"),
    "tokens_descending": ("    for (int t = 0; t < p->bucket; ++t)\n      for (int k = 0; k < p->K; ++k) {\n        int64_t ri = route_index(p, s, t, k);\n        if (t >= p->T[s]",
                          "    for (int t = p->bucket - 1; t >= 0; --t)\n      for (int k = 0; k < p->K; ++k) {\n        int64_t ri = route_index(p, s, t, k);\n        if (t >= p->T[s]"),
    "row_copied_from_wrong_token": ("x + ((int64_t)s * p->bucket + t) * row_bytes",
                                    "x + ((int64_t)s * p->bucket + (t + 1) % p->T[s]) * row_bytes"),
    "expert_constant_shifted": ("ldexpf(1.0f, (e % 4) - 1)", "ldexpf(1.0f, (e % 4))"),
    "fp8_scale_dropped": ("v = v * row_scales[(f * r_stride + r) * nb + h / 128];", "v = v * 1.0f;"),
    "padding_row_src_zero": ("row_src[f * r_stride + r] = -1;", "row_src[f * r_stride + r] = 0;"),
    "group_exponent_unclamped": ("for (int e = -117; e <= 128; ++e)", "for (int e = -126; e <= 128; ++e)"),
    "group_exponent_off_by_one": ("if (amax <= ldexpf(448.0f, e)) return e;", "if (amax < ldexpf(448.0f, e)) return e;"),
    "e4m3_normal_ties_away": ("    if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) == 1.0)) n += 1.0;\n    if (n == 16.0) {",
                              "    if (r >= 0.5) n += 1.0;\n    if (n == 16.0) {"),
    "e4m3_saturates_to_nan_code": ("if (a >= 448.0) return sign | 0x7e;", "if (a >= 448.0) return sign | 0x7f;"),
    "partial_not_rounded": ("part[h] = orc_bf16_to_float(orc_float_to_bf16(a));", "part[h] = a;"),
    "worker_order_first_route": ("for (int j = k + 1; j < p->K; ++j) {\n          int64_t rj = route_index(p, s, t, j);\n          if (slot[rj] >= 0 && (int)(ids[rj] / Ef) == f) last = 0;",
                                 "for (int j = 0; j < k; ++j) {\n          int64_t rj = route_index(p, s, t, j);\n          if (slot[rj] >= 0 && (int)(ids[rj] / Ef) == f) last = 0;"),
    "fp8_decode_clamped": ("part[h] = ldexpf(orc_e4m3_to_float(q), e);",
                           "part[h] = fminf(fmaxf(ldexpf(orc_e4m3_to_float(q), e), -3.4028235e38f), 3.4028235e38f);"),
    "fp8_dequant_wrong_scale": ("part[h] = ldexpf(orc_e4m3_to_float(q), e);", "part[h] = ldexpf(orc_e4m3_to_float(q), e + 1);"),
    "dispatch_worker_modulo": ("int f = (int)(e / Ef);", "int f = (int)(e % p->F);"),
    "combine_worker_modulo": ("int f = (int)(ids[ri] / Ef);\n          float r",
                              "int f = (int)(ids[ri] % p->F);\n          float r"),
    "ends_without_count": ("ends[i] = start[i] + count[i];", "ends[i] = start[i];"),
    "padding_weight_one": ("row_w[f * r_stride + r] = 0.0f;", "row_w[f * r_stride + r] = 1.0f;"),
    "combine_weight_squared": ("acc = fmaf(w[ri], r, acc);", "acc = fmaf(w[ri] * w[ri], r, acc);"),
    "fp8_scale_from_first_block": ("x_scales[((int64_t)s * p->bucket + t) * nb + b];",
                                   "x_scales[((int64_t)s * p->bucket + t) * nb];"),
    "expert_skips_last_row": ("for (int64_t r = start[e]; r < ends[e]; ++r) {",
                              "for (int64_t r = start[e]; r < ends[e] - 1; ++r) {"),
}


def _pins(orc, report=None) -> list:
    """Runs the battery; returns the names of the pins that failed. `report`,
    when given, is called with each failed pin's name as soon as it fails."""
    failed = []

    def run(name, fn):
        try:
            fn()
        except Exception:  # a wrong value, or results too broken to index
            failed.append(name)
            if report:
                report(name)

    def golden_layout():
        with open(os.path.join(GOLDEN, "ends_convention.json")) as fh:
            g = json.load(fh)
        q = g["problem"]
        p = oracle.Problem(q["A"], q["F"], q["E"], q["K"], q["H"], q["alpha"], q["bucket"],
                           oracle.BF16, q["T"])
        ids = np.array(g["ids"], np.int64)
        lay = oracle.layout(p, ids, orc)  # the layout alone first: no arrays sized by it yet
        for key in ("count", "start", "ends", "host_counts", "r_exact"):
            assert np.array_equal(np.asarray(lay[key]), np.array(g[key])), key
        r = oracle.round_trip(p, ids, np.ones(ids.shape, np.float32),
                              np.zeros((1, q["bucket"], q["H"]), np.uint16), orc=orc)
        for key in ("count", "start", "ends", "host_counts", "r_exact", "slot"):
            assert np.array_equal(np.asarray(r[key]), np.array(g[key])), key
        for f, want in enumerate(g["row_src"]):
            assert r["row_src"][f, : len(want)].tolist() == want

    def random_layout_and_dispatch():
        rng = np.random.default_rng(21)
        for trial in range(25):
            F = int(rng.integers(1, 4)); Ef = int(rng.integers(1, 5)); E = F * Ef
            K = int(rng.integers(1, min(E, 4) + 1)); A = 2; B = 4
            a = int(rng.choice([1, 2, 4]))
            T = [int(rng.integers(1, B + 1)) for _ in range(A)]
            ids = np.stack([np.stack([rng.permutation(E)[:K] for _ in range(B)]) for _ in range(A)])
            ids = ids.astype(np.int64)
            ids[rng.random(ids.shape) < 0.2] = -1
            w = rng.random((A, B, K)).astype(np.float32)
            x = rng.integers(0, 1 << 15, size=(A, B, 128)).astype(np.uint16)
            p = oracle.Problem(A, F, E, K, 128, a, B, oracle.BF16, T)
            r = oracle.round_trip(p, ids, w, x, orc=orc)
            TL._check_ends_convention(p, ids, r)
            TL._check_dispatch(p, ids, w, x, None, r)

    def fp8_dispatch_and_expert():
        from combine_attention_ffn_gb300 import workloads as W
        wl = W.named("fp8-2A2F", T=4)
        inp = W.make_inputs(wl)
        p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, oracle.FP8, wl.T)
        r = oracle.round_trip(p, inp.ids, inp.w, inp.x, inp.x_scales,
                              expert_mode=oracle.EXPERT_SCALE, orc=orc)
        TL._check_dispatch(p, inp.ids, inp.w, inp.x, inp.x_scales, r)
        Ef = wl.E // wl.F
        for f in range(wl.F):
            for l in range(Ef):
                e = f * Ef + l
                lo, hi = r["start"][f, l], r["ends"][f, l]
                q = torch.from_numpy(r["rows"][f, lo:hi]).view(torch.float8_e4m3fn).float()
                sc = torch.from_numpy(r["row_scales"][f, lo:hi]).repeat_interleave(128, dim=1)
                want = ((q * sc) * 2.0 ** ((e % 4) - 1)).to(torch.bfloat16).view(torch.int16).numpy()
                assert np.array_equal(r["reply"][f, lo:hi].view(np.int16), want)

    def validate_rules():
        rng = np.random.default_rng(3)
        for _ in range(60):
            ids = rng.integers(-3, 8, size=(2, 5, 3)).astype(np.int64)
            T = [int(rng.integers(0, 6)) for _ in range(2)]
            p = oracle.Problem(2, 2, 6, 3, 256, 1, 5, oracle.BF16, T)
            assert oracle.validate(p, ids, orc) == TL._first_error_numpy(ids, T, 6)

    def combine_exact():
        rng = np.random.default_rng(4)
        A, B, K, E, F, H = 2, 2, 5, 12, 3, 128
        ids = TC._uniform_ids(rng, A, B, K, E)
        ids[rng.random(ids.shape) < 0.25] = -1
        ids[1, 1] = -1
        w = (rng.random((A, B, K)) * 1.7).astype(np.float32)
        x = TC._rand_bf16(rng, (A, B, H), scale=5.0)
        p = oracle.Problem(A, F, E, K, H, 4, B, oracle.BF16, [2, 2])
        r = oracle.round_trip(p, ids, w, x, expert_mode=oracle.EXPERT_SCALE, orc=orc)
        want = TC._exact_combine(ids, w, x, [2, 2], F, E, lambda e: Fraction(2) ** ((e % 4) - 1))
        assert np.array_equal(r["out"], want)

    def combine_crafted():
        w = np.array([[[1.0 + 2.0 ** -8, 16647161 * 2.0 ** -24]]], np.float32)
        reply = np.zeros((1, 2, 128), np.uint16)
        reply[0, 0, :] = 0x3F80
        reply[0, 1, :] = 0x3381
        p = oracle.Problem(1, 1, 2, 2, 128, 1, 1, oracle.BF16, [1])
        out = oracle.combine(p, np.array([[[0, 1]]], np.int64), w,
                             np.array([[[0, 1]]], np.int32), 2, reply, orc=orc)
        assert np.all(out[0, 0] == 0x3F81)

    def bf16_vs_torch():
        rng = np.random.default_rng(7)
        bits = rng.integers(0, 1 << 32, size=1 << 16, dtype=np.uint64).astype(np.uint32)
        ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], np.float32)
        f = np.concatenate([ties, bits.view(np.float32)])
        f = f[np.isfinite(f)]
        got = orc.float_to_bf16(f)
        ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, ref)

    def e4m3_vs_torch():
        codes = np.arange(256, dtype=np.uint8)
        got = orc.e4m3_to_float(codes)
        ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
        ok = ~np.isnan(ref)
        assert np.array_equal(np.isnan(got), ~ok)
        assert np.array_equal(got[ok], ref[ok])

    def two_stage():
        import test_oracle_two_stage as TS
        ids, w, vals = TS.crafted_order_case()
        H = 128
        p = oracle.Problem(1, 4, 8, 5, H, 1, 1, oracle.BF16, [1])
        lay = oracle.layout(p, ids, orc)
        r_stride = int(lay["r_exact"].max())
        d = oracle.dispatch(p, ids, w, np.zeros((1, 1, H), np.uint16), None, lay, r_stride, orc)
        reply = np.zeros((4, r_stride, H), np.uint16)
        for k in range(5):
            reply[int(ids[0, 0, k]) // 2, d["slot"][0, 0, k], :] = np.float32(vals[k]).view(np.uint32) >> 16
        assert np.all(oracle.combine_two_stage(p, ids, w, d["slot"], r_stride, reply, False, orc)[0, 0] == 0x3F81)
        rng = np.random.default_rng(5)
        A, B, K, E, F = 1, 2, 6, 12, 3
        ids = np.stack([np.stack([rng.permutation(E)[:K] for _ in range(B)]) for _ in range(A)]).astype(np.int64)
        w = (rng.random((A, B, K)) * 1.5).astype(np.float32)
        xf = (rng.standard_normal((A, B, H)) * 4).astype(np.float32)
        x = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        p = oracle.Problem(A, F, E, K, H, 2, B, oracle.BF16, [2])
        for fp8 in (False, True):
            r = oracle.round_trip(p, ids, w, x, expert_mode=oracle.EXPERT_SCALE, orc=orc,
                                  combine_mode=oracle.COMBINE_TWO_STAGE_FP8 if fp8 else oracle.COMBINE_TWO_STAGE)
            want = TS._two_stage_exact(ids, w, r["slot"], r["reply"], E // F, [2], fp8)
            assert np.array_equal(r["out"], want)

    def two_stage_top_binade():
        import test_oracle_two_stage as TS
        got = TS.top_binade_outputs(orc)
        for v, want in TS.TOP_BINADE_CASES.items():
            assert got[v][0] == want

    def fp8_formats():
        import test_oracle_two_stage as TS
        f32 = np.float32
        nxt = float(np.nextafter(f32(448), f32(1e9)))
        amax = np.array([448.0, nxt, 0.0, float("inf"), 1.75], np.float32)
        assert orc.group_exponent(amax).tolist() == [0, 1, -117, 120, -8]
        x = np.array([2 ** -10, 3 * 2 ** -10, 460.0, 1e9, 1.0 + 3 * 2 ** -4, 1.0 + 2 ** -4], np.float32)
        assert orc.float_to_e4m3(x).tolist() == [0x00, 0x02, 0x7E, 0x7E, 0x3A, 0x38]

    for name, fn in [("golden_layout", golden_layout), ("random_layout_dispatch", random_layout_and_dispatch),
                     ("two_stage", two_stage), ("two_stage_top_binade", two_stage_top_binade),
                     ("fp8_formats", fp8_formats),
                     ("fp8", fp8_dispatch_and_expert), ("validate", validate_rules),
                     ("combine_exact", combine_exact), ("combine_crafted", combine_crafted),
                     ("bf16", bf16_vs_torch), ("e4m3", e4m3_vs_torch)]:
        run(name, fn)
    return failed


def _build_variant(tmp_path, name, old, new) -> str:
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: pattern must occur once"
    d = tmp_path / name
    d.mkdir()
    shutil.copy(HDR, d / "orc.h")
    (d / "orc.c").write_text(src.replace(old, new))
    lib = d / "liborc.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", str(d), str(d / "orc.c"), "-o", str(lib), "-lm"],
                   check=True)
    return str(lib)


def _pins_in_child(lib: str):
    """Runs the battery on a mutant library in a child process, so that a
    mutant that writes out of bounds cannot take the test run down with it.
    Returns the pins that failed before the end or a crash, and "(crashed)"
    when the child did not finish."""
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]; import oracle, test_oracle_mutations as M; "
            "M._pins(oracle.Oracle(%r), report=lambda n: print('FAILED ' + n, flush=True)); "
            "print('DONE', flush=True)" % (here, os.path.dirname(here), lib))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    lines = r.stdout.splitlines()
    failed = [l[7:] for l in lines if l.startswith("FAILED ")]
    if r.returncode != 0 or "DONE" not in lines:
        failed.append("(crashed)")
    return failed


def test_unmodified_oracle_passes_battery(orc):
    assert _pins(orc) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    failed = _pins_in_child(_build_variant(tmp_path, name, old, new))
    assert [f for f in failed if f != "(crashed)"], f"mistake '{name}' passed every pin ({failed})"
