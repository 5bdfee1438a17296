"""Pins for the oracle's route validation, layout (ends[], host counts) and
placement (slot map, receipts, rows).

Each check is written independently of the oracle's C code: a hand-worked
golden case, library primitives (numpy bincount / stable argsort), closed-form
invariants of the ends[] convention, and exhaustive enumeration on tiny
problems.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from combine_attention_ffn_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(wl, dtype=None):
    dt = oracle.FP8 if (dtype or wl.dtype) == "fp8" else oracle.BF16
    return oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket, dt, wl.T)


# ----------------------------------------------------------------- validate
def _first_error_numpy(ids, T, E):
    """Independent statement of the ID rules: scan (s,t,k) in order; -1 skips;
    outside [-1, E) is a range error; an in-range ID equal to an earlier ID of
    the same token is a duplicate."""
    A, B, K = ids.shape
    for s in range(A):
        for t in range(T[s]):
            row = ids[s, t]
            for k in range(K):
                v = int(row[k])
                if v == -1:
                    continue
                if v < -1 or v >= E:
                    return (1, s, t, k)
                if v in [int(u) for u in row[:k]]:
                    return (2, s, t, k)
    return (0, -1, -1, -1)


def test_validate_hand_cases():
    p = oracle.Problem(2, 2, 8, 3, 256, 1, 4, oracle.BF16, [4, 2])
    base = np.full((2, 4, 3), -1, np.int64)
    assert oracle.validate(p, base) == (0, -1, -1, -1)
    ids = base.copy(); ids[1, 1, 2] = 8
    assert oracle.validate(p, ids) == (1, 1, 1, 2)
    ids = base.copy(); ids[0, 3, 1] = -2
    assert oracle.validate(p, ids) == (1, 0, 3, 1)
    ids = base.copy(); ids[0, 2] = [5, 1, 5]
    assert oracle.validate(p, ids) == (2, 0, 2, 2)
    ids = base.copy(); ids[0, 2] = [9, 9, 3]          # out-of-range repeats are range errors
    assert oracle.validate(p, ids) == (1, 0, 2, 0)
    ids = base.copy(); ids[1, 3, 0] = 99              # beyond T[1] = 2: never read
    assert oracle.validate(p, ids) == (0, -1, -1, -1)
    ids = base.copy(); ids[0, 1] = [2, 2, -1]; ids[0, 0, 2] = 100   # first in (s,t,k) order wins
    assert oracle.validate(p, ids) == (1, 0, 0, 2)
    ids = base.copy(); ids[0, 0] = [-1, -1, -1]; ids[0, 1] = [1 << 40, 0, 0]  # wide value
    assert oracle.validate(p, ids) == (1, 0, 1, 0)


def test_validate_random_against_independent_rules():
    rng = np.random.default_rng(3)
    for trial in range(300):
        A, E, K, B = 2, 6, 3, 5
        T = [int(rng.integers(0, B + 1)) for _ in range(A)]
        ids = rng.integers(-3, E + 2, size=(A, B, K)).astype(np.int64)
        p = oracle.Problem(A, 2, E, K, 256, 1, B, oracle.BF16, T)
        assert oracle.validate(p, ids) == _first_error_numpy(ids, T, E), trial


# ----------------------------------------------------------------- layout
def test_layout_golden_hand_worked():
    with open(os.path.join(GOLDEN, "ends_convention.json")) as fh:
        g = json.load(fh)
    q = g["problem"]
    p = oracle.Problem(q["A"], q["F"], q["E"], q["K"], q["H"], q["alpha"], q["bucket"],
                       oracle.BF16, q["T"])
    ids = np.array(g["ids"], np.int64)
    w = np.ones(ids.shape, np.float32)
    x = np.zeros((q["A"], q["bucket"], q["H"]), np.uint16)
    r = oracle.round_trip(p, ids, w, x)
    for key in ("count", "start", "ends", "host_counts", "r_exact", "slot"):
        assert np.array_equal(np.asarray(r[key]), np.array(g[key])), key
    for f, want in enumerate(g["row_src"]):
        assert r["row_src"][f, : len(want)].tolist() == want


def _check_ends_convention(p, ids, lay):
    """Closed-form properties of the ends[] convention."""
    Ef, a = p.E // p.F, p.alpha
    valid = []
    for s in range(p.A):
        for t in range(p.T[s]):
            seen = set()
            for k in range(p.K):
                v = int(ids[s, t, k])
                if 0 <= v < p.E and v not in seen:
                    valid.append(v)
                seen.add(v)
    want_count = np.bincount(np.array(valid, np.int64), minlength=p.E).reshape(p.F, Ef)
    assert np.array_equal(lay["count"], want_count)
    st, en, hc = lay["start"], lay["ends"], lay["host_counts"]
    for f in range(p.F):
        assert st[f, 0] == 0
        assert np.all(st[f] % a == 0)
        assert np.array_equal(en[f] - st[f], want_count[f])
        for l in range(1, Ef):
            # start is the smallest multiple of alpha at or above the previous end
            assert st[f, l] >= en[f, l - 1] and st[f, l] - a < en[f, l - 1]
        assert np.array_equal(hc[f] % a, np.zeros(Ef)) and np.all(hc[f] >= want_count[f])
        assert np.all(hc[f] - want_count[f] < a)
        assert lay["r_exact"][f] == hc[f].sum()
        assert lay["r_exact"][f] % a == 0 and lay["r_exact"][f] >= en[f, -1]


@pytest.mark.parametrize("name", ["tiny", "2A2F", "skew-3A1F", "skew-1A3F"])
def test_layout_invariants_on_workloads(name):
    wl = W.named(name, T=None if name == "tiny" else 128)
    inp = W.make_inputs(wl)
    p = _problem(wl)
    lay = oracle.layout(p, inp.ids)
    _check_ends_convention(p, inp.ids, lay)


def test_layout_random_alignment_and_drops():
    rng = np.random.default_rng(5)
    for trial in range(60):
        F = int(rng.integers(1, 4)); Ef = int(rng.integers(1, 6)); E = F * Ef
        K = int(rng.integers(1, min(E, 5) + 1)); A = int(rng.integers(1, 4))
        B = int(rng.integers(0, 9)); a = int(rng.choice([1, 2, 3, 8, 128]))
        T = [int(rng.integers(0, B + 1)) for _ in range(A)]
        ids = np.stack([np.stack([rng.permutation(E)[:K] for _ in range(B)])
                        if B else np.zeros((0, K), np.int64) for _ in range(A)]).astype(np.int64)
        ids = ids.reshape(A, B, K)
        ids[rng.random(ids.shape) < 0.3] = -1
        p = oracle.Problem(A, F, E, K, 256, a, B, oracle.BF16, T)
        _check_ends_convention(p, ids, oracle.layout(p, ids))


# ----------------------------------------------------------------- dispatch
def _expected_slots_by_stable_sort(p, ids, start):
    """Independent placement: list valid routes in (s, t, k) order, stable-sort
    them by expert (numpy), and give the i-th route of expert e row
    start[e] + i."""
    routes, experts = [], []
    for s in range(p.A):
        for t in range(p.T[s]):
            seen = set()
            for k in range(p.K):
                v = int(ids[s, t, k])
                if 0 <= v < p.E and v not in seen:
                    routes.append((s, t, k)); experts.append(v)
                seen.add(v)
    order = np.argsort(np.array(experts, np.int64), kind="stable")
    slot = np.full((p.A, p.bucket, p.K), -1, np.int64)
    seen_per_e = {}
    flat_start = np.asarray(start).reshape(-1)
    for i in order:
        e = experts[i]
        j = seen_per_e.get(e, 0); seen_per_e[e] = j + 1
        s, t, k = routes[i]
        slot[s, t, k] = flat_start[e] + j
    return slot


def _check_dispatch(p, inp_ids, inp_w, inp_x, inp_xs, r):
    Ef = p.E // p.F
    want_slot = _expected_slots_by_stable_sort(p, inp_ids, r["start"])
    assert np.array_equal(r["slot"], want_slot)
    live = np.zeros(r["row_src"].shape, bool)
    xb = np.ascontiguousarray(inp_x).view(np.uint8).reshape(p.A, p.bucket, -1)
    for s in range(p.A):
        for t in range(p.bucket):
            for k in range(p.K):
                row = int(r["slot"][s, t, k])
                if row < 0:
                    continue
                f = int(inp_ids[s, t, k]) // Ef
                assert not live[f, row], "two routes share a row"
                live[f, row] = True
                assert r["row_src"][f, row] == (s * p.bucket + t) * p.K + k
                assert r["row_w"][f, row].view(np.uint32) == inp_w[s, t, k].view(np.uint32)
                assert np.array_equal(r["rows"][f, row], xb[s, t])
                if p.dtype == oracle.FP8:
                    assert np.array_equal(r["row_scales"][f, row], inp_xs[s, t])
                # the row lies inside its expert's range
                e = int(inp_ids[s, t, k]); l = e % Ef
                assert r["start"][f, l] <= row < r["ends"][f, l]
    for f in range(p.F):
        n = int(r["r_exact"][f])
        pad = ~live[f, :n]
        assert np.all(r["row_src"][f, :n][pad] == -1)
        assert np.all(r["row_w"][f, :n][pad].view(np.uint32) == 0)
        assert live[f].sum() == r["count"][f].sum()


@pytest.mark.parametrize("name,T", [("tiny", None), ("2A2F", 32), ("skew-3A1F", 32),
                                    ("skew-1A3F", 64), ("fp8-2A2F", 16), ("fp8-2A1F", 8)])
def test_dispatch_against_stable_sort(name, T):
    wl = W.named(name, T=T)
    inp = W.make_inputs(wl)
    p = _problem(wl)
    r = oracle.round_trip(p, inp.ids, inp.w, inp.x, inp.x_scales)
    assert r["err"][0] == 0
    _check_dispatch(p, inp.ids, inp.w, inp.x, inp.x_scales, r)


def test_dispatch_exhaustive_tiny():
    """E=4, K=2, A=2, F=2, alpha in {1,2}: every ID pattern (with -1) for two
    live tokens, and a seeded sample of the patterns for three."""
    E, K, F, A = 4, 2, 2, 2
    tok_patterns = [p for p in itertools.product(range(-1, E), repeat=K)
                    if len({v for v in p if v >= 0}) == len([v for v in p if v >= 0])]
    rng = np.random.default_rng(1)
    count = 0
    for alpha in (1, 2):
        for T in ((1, 1), (2, 1), (0, 2)):
            for combo in itertools.product(tok_patterns, repeat=sum(T)):
                if sum(T) > 2 and rng.random() > 0.05:
                    continue
                ids = np.full((A, 2, K), -1, np.int64)
                it = iter(combo)
                for s in range(A):
                    for t in range(T[s]):
                        ids[s, t] = next(it)
                w = rng.random((A, 2, K)).astype(np.float32)
                x = rng.integers(0, 1 << 16, size=(A, 2, 128)).astype(np.uint16)
                p = oracle.Problem(A, F, E, K, 128, alpha, 2, oracle.BF16, list(T))
                r = oracle.round_trip(p, ids, w, x)
                _check_ends_convention(p, ids, r)
                _check_dispatch(p, ids, w, x, None, r)
                count += 1
    assert count > 2000
