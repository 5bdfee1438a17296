"""Seeded synthetic exchanges shaped like the afdEP-comm benchmark workloads.

This module only draws inputs: top-k expert IDs, routing weights and
activations. It holds none of the exchange's arithmetic (no layout, no
placement, no reduction, no rounding code of its own: BF16 and FP8 values are
produced with PyTorch's own conversions). The library's tests feed the same
arrays to the GPU path and to the CPU oracle.

Workloads (afdEP-comm design page, "Result" table: E128, top-k 8, capacity
2,048, hidden 2,048 / 4,096, random or skewed routing, BF16 or FP8 dispatch;
E96 for 1A:3F):

* ``tiny``            2 sources x 16 tokens, 2 workers, E=8, K=2, H=256, alpha=1
* ``uniform``         2A2F, E=128, K=8, H=2048 (or 4096), alpha=128, bucket 2048
* ``skew``            Zipf-like popularity (e+1)^-1.2 sampled without
                      replacement, 10% of top-k slots set to -1; 3A:1F (E128)
                      and 1A:3F (E96)
* ``fp8``             2A2F uniform with E4M3 activations and FP32 block-128
                      scales (absmax / 448), plus a 2A1F layout

Recipe per source s (independent stream seeded from (seed, s, T, kind)):

* IDs, uniform: the first K entries of a uniformly random permutation of the
  E experts (distinct by construction).
* IDs, skew: Gumbel-top-K over log p_e with p_e proportional to (e+1)^-1.2,
  which is the same distribution as drawing K experts one after another
  without replacement in proportion to p_e. Then each slot is set to -1
  independently with probability ``drop``.
* weights: softmax (FP64, stored FP32) of K standard normal logits, taken over
  all K slots before any slot is dropped.
* x: standard normal FP32, rounded to BF16 by PyTorch. FP8: per 128-element
  block, scale = absmax / 448 (1.0 for an all-zero block), q = x / scale
  clamped to [-448, 448] and converted to float8_e4m3fn by PyTorch.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

import numpy as np

_KIND_IDS, _KIND_DROP, _KIND_W, _KIND_X = 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    name: str
    A: int                 # Attention sources
    F: int                 # FFN workers
    E: int                 # experts
    K: int                 # top-k
    H: int                 # hidden
    alpha: int             # expert_alignment
    capacity: int          # max tokens per source (arena sizing)
    bucket: int            # padded tokens per source for this exchange
    T: Tuple[int, ...]     # live tokens per source
    dtype: str = "bf16"    # "bf16" | "fp8"
    routing: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 1.2
    drop: float = 0.0
    seed: int = 0

    @property
    def Ef(self) -> int:
        return self.E // self.F

    @property
    def row_bytes(self) -> int:
        return self.H if self.dtype == "fp8" else 2 * self.H

    def with_tokens(self, T, bucket: Optional[int] = None) -> "Workload":
        if isinstance(T, int):
            T = (T,) * self.A
        return replace(self, T=tuple(T), bucket=self.bucket if bucket is None else bucket)


@dataclass
class Inputs:
    """Arrays padded to ``bucket`` tokens per source (entries t >= T[s] are
    -1 IDs, zero weights and zero activations)."""
    wl: Workload
    ids: np.ndarray                  # int64 [A, bucket, K]
    w: np.ndarray                    # float32 [A, bucket, K]
    x: np.ndarray                    # uint16 BF16 bits or uint8 E4M3 codes [A, bucket, H]
    x_scales: Optional[np.ndarray] = None   # float32 [A, bucket, H/128] (FP8)
    extra: dict = field(default_factory=dict)


# ---------------------------------------------------------------- configs
def tiny(seed: int = 101) -> Workload:
    return Workload("tiny", A=2, F=2, E=8, K=2, H=256, alpha=1, capacity=16, bucket=16,
                    T=(16, 16), seed=seed)


def uniform_2a2f(T: int = 2048, H: int = 2048, seed: Optional[int] = None) -> Workload:
    name = "2A2F" if H == 2048 else f"2A2F-H{H}"
    return Workload(name, A=2, F=2, E=128, K=8, H=H, alpha=128, capacity=2048,
                    bucket=2048, T=(T, T), seed=seed if seed is not None else (202 if H == 2048 else 303))


def skew_3a1f(T: int = 2048, seed: int = 404) -> Workload:
    return Workload("skew-3A1F", A=3, F=1, E=128, K=8, H=2048, alpha=128, capacity=2048,
                    bucket=2048, T=(T,) * 3, routing="zipf", drop=0.1, seed=seed)


def skew_1a3f(T: int = 2048, seed: int = 404) -> Workload:
    return Workload("skew-1A3F", A=1, F=3, E=96, K=8, H=2048, alpha=128, capacity=2048,
                    bucket=2048, T=(T,), routing="zipf", drop=0.1, seed=seed)


def fp8_2a2f(T: int = 2048, seed: int = 505) -> Workload:
    return Workload("fp8-2A2F", A=2, F=2, E=128, K=8, H=2048, alpha=128, capacity=2048,
                    bucket=2048, T=(T, T), dtype="fp8", seed=seed)


def fp8_2a1f(T: int = 2048, seed: int = 505) -> Workload:
    return Workload("fp8-2A1F", A=2, F=1, E=128, K=8, H=2048, alpha=128, capacity=2048,
                    bucket=2048, T=(T, T), dtype="fp8", seed=seed)


def named(name: str, T: Optional[int] = None) -> Workload:
    table = {"tiny": tiny, "2A2F": uniform_2a2f,
             "2A2F-H4096": lambda **kw: uniform_2a2f(H=4096, **kw),
             "skew-3A1F": skew_3a1f, "skew-1A3F": skew_1a3f,
             "fp8-2A2F": fp8_2a2f, "fp8-2A1F": fp8_2a1f}
    wl = table[name]() if T is None or name == "tiny" else table[name](T=T)
    return wl


# ---------------------------------------------------------------- drawing
def _rng(wl: Workload, s: int, kind: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([wl.seed, s, wl.T[s], kind]))


def _draw_ids(wl: Workload, s: int, T: int) -> np.ndarray:
    rng = _rng(wl, s, _KIND_IDS)
    if wl.routing == "uniform":
        keys = rng.random((T, wl.E))
        ids = np.argsort(keys, axis=1, kind="stable")[:, : wl.K]
    elif wl.routing == "zipf":
        logp = -wl.zipf_s * np.log(np.arange(1, wl.E + 1, dtype=np.float64))
        gumbel = -np.log(-np.log(rng.random((T, wl.E))))
        ids = np.argsort(-(logp[None, :] + gumbel), axis=1, kind="stable")[:, : wl.K]
    else:
        raise ValueError(wl.routing)
    ids = ids.astype(np.int64)
    if wl.drop > 0:
        mask = _rng(wl, s, _KIND_DROP).random((T, wl.K)) < wl.drop
        ids[mask] = -1
    return ids


def _draw_weights(wl: Workload, s: int, T: int) -> np.ndarray:
    logits = _rng(wl, s, _KIND_W).standard_normal((T, wl.K))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def _draw_x(wl: Workload, s: int, T: int):
    import torch

    xf = _rng(wl, s, _KIND_X).standard_normal((T, wl.H), dtype=np.float32)
    if wl.dtype == "bf16":
        return torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), None
    blocks = xf.reshape(T, wl.H // 128, 128)
    amax = np.abs(blocks).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = np.clip(blocks / scale[:, :, None], -448.0, 448.0).astype(np.float32).reshape(T, wl.H)
    codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scale


def make_inputs(wl: Workload) -> Inputs:
    A, B, K, H = wl.A, wl.bucket, wl.K, wl.H
    assert len(wl.T) == A and all(0 <= t <= B for t in wl.T)
    ids = np.full((A, B, K), -1, np.int64)
    w = np.zeros((A, B, K), np.float32)
    x = np.zeros((A, B, H), np.uint8 if wl.dtype == "fp8" else np.uint16)
    xs = np.zeros((A, B, H // 128), np.float32) if wl.dtype == "fp8" else None
    for s, T in enumerate(wl.T):
        if T == 0:
            continue
        ids[s, :T] = _draw_ids(wl, s, T)
        w[s, :T] = _draw_weights(wl, s, T)
        xv, sv = _draw_x(wl, s, T)
        x[s, :T] = xv
        if xs is not None:
            xs[s, :T] = sv
    return Inputs(wl, ids, w, x, xs)
