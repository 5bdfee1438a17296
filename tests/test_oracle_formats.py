"""Pins for the oracle's number formats (BF16 and OCP E4M3).

The oracle writes its codecs from the format definitions; these tests check
them against a library routine (PyTorch's own conversions), against exact
rational rounding (tests/exact.py) and against hand-worked points.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32_from_bits(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def test_bf16_widen_all_codes_match_torch(orc):
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16_to_float(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _special_floats():
    vals = [0.0, -0.0, 1.0, -1.0, float("inf"), float("-inf"), float("nan"),
            1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20,
            3.3895313892515355e38,  # largest BF16 value
            3.4e38, 1e-40, -1e-40, 2.0 ** -133, 2.0 ** -126, 2.0 ** -149]
    bits = np.array([struct.unpack("<I", struct.pack("<f", v))[0] for v in vals], np.uint32)
    # every rounding case around a kept pattern: dropped bits 0x7fff, 0x8000, 0x8001
    base = np.array([0x3F800000, 0x3F810000, 0x7F7F0000, 0x00010000, 0x80450000], np.uint32)
    around = (base[:, None] + np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)).ravel()
    return np.concatenate([bits, around])


def test_bf16_round_matches_torch(orc):
    rng = np.random.default_rng(7)
    rand_bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([_special_floats(), rand_bits])
    f = _f32_from_bits(bits)
    got = orc.float_to_bf16(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got_nan = (got & 0x7F80) == 0x7F80
    got_nan &= (got & 0x007F) != 0
    ref_nan = np.isnan(f)
    assert np.array_equal(got_nan, ref_nan)
    assert np.array_equal(got[~ref_nan], ref[~ref_nan])


def test_bf16_round_matches_exact_rational(orc):
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 32, size=4000, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, _special_floats()])
    f = _f32_from_bits(bits)
    got = orc.float_to_bf16(f)
    for v, g in zip(f.tolist(), got.tolist()):
        if math.isnan(v):
            continue
        if math.isinf(v):
            assert g == (0x7F80 if v > 0 else 0xFF80)
            continue
        r = exact.round_bf16(Fraction(v))
        want = exact.bf16_bits(r)
        if r == 0 and math.copysign(1.0, v) < 0:
            want = 0x8000
        assert g == want, (v, hex(g), hex(want))


def test_bf16_hand_ties(orc):
    # ties go to the even BF16 pattern
    f = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], np.float32)
    assert orc.float_to_bf16(f).tolist() == [0x3F80, 0x3F82, 0xBF80]


def test_e4m3_all_codes_match_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_golden_points(orc):
    with open(os.path.join(GOLDEN, "e4m3_points.json")) as fh:
        g = json.load(fh)
    for code, val in g["points"]:
        got = float(orc.e4m3_to_float(np.array([int(code, 16)], np.uint8))[0])
        if val == "nan":
            assert math.isnan(got), code
        else:
            want = float(val)
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got)
