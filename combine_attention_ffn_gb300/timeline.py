"""Where an exchange's time goes, from the phase-timer build.

Builds libafd_timers.so (the same kernels with %globaltimer stamps, see
afd_phase_stamps in include/afd.h), captures one exchange of a synthetic
workload as a CUDA graph, replays it (after an L2 flush, or back to back) and
prints, for every recorded point of every kernel, the median over replays of
the earliest, median and latest block's stamp, in µs from the first dispatch
block's start. The stamps cost a little time themselves; the default library
has none.

    python -m combine_attention_ffn_gb300.timeline --config 2A2F --tokens 2048
"""
from __future__ import annotations

import argparse
import statistics

import numpy as np

POINTS = {
    "dispatch": ("start", "wait passed", "first IDs marked", "counted", "cluster barrier passed",
                 "all counts read", "scan done", "codes written / end"),
    "scatter": ("start", "wait passed", "first row in shared memory", "stores issued",
                "stores complete", "end"),
    "combine": ("start", "wait passed", "sums stored", "end"),
    "combine-early": ("start", "ready to load", "sums stored", "end (after its wait)"),
}


def _exchange(buf, wl, xs, ids, ws, scs, outs, replies):
    for s in range(wl.A):
        buf.source_dispatch(s, xs[s], ids[s], ws[s], scs[s], bucket=wl.bucket)
    for f in range(wl.F):
        r = buf.worker_receive(f, bucket=wl.bucket)
        buf.worker_reply(f, replies[f] if replies else r.rows, r.receipt)
    for s in range(wl.A):
        buf.source_collect(s, out=outs[s])


def run(config: str, tokens: int, replays: int, back_to_back: bool, combine_mode: str) -> list[str]:
    import torch

    from . import afd, build
    from . import workloads as W

    afd.use_library(build.build_timers())
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    wl = W.named(config, T=tokens)
    inp = W.make_inputs(wl)
    modes = {"fused": afd.COMBINE_FUSED, "two-stage": afd.COMBINE_TWO_STAGE,
             "two-stage-fp8": afd.COMBINE_TWO_STAGE_FP8}
    buf = afd.Buffer(wl.A, wl.F, wl.E, wl.K, wl.H, wl.capacity, wl.alpha, wl.dtype,
                     combine_mode=modes[combine_mode])
    fp8 = wl.dtype == "fp8"
    ts = list(enumerate(wl.T))
    if fp8:
        xs = [torch.from_numpy(inp.x[s, :t].copy()).to(dev).view(torch.float8_e4m3fn) for s, t in ts]
        scs = [torch.from_numpy(inp.x_scales[s, :t].copy()).to(dev) for s, t in ts]
    else:
        xs = [torch.from_numpy(inp.x[s, :t].view(np.int16).copy()).to(dev).view(torch.bfloat16)
              for s, t in ts]
        scs = [None] * wl.A
    ids = [torch.from_numpy(inp.ids[s, :t].copy()).to(dev) for s, t in ts]
    ws = [torch.from_numpy(inp.w[s, :t].copy()).to(dev) for s, t in ts]
    outs = [torch.empty((t, wl.H), dtype=torch.bfloat16, device=dev) for _, t in ts]
    replies = None
    if fp8:  # BF16 replies computed once from the received rows (routing does not change)
        for s in range(wl.A):
            buf.source_dispatch(s, xs[s], ids[s], ws[s], scs[s], bucket=wl.bucket)
        replies = []
        for f in range(wl.F):
            r = buf.worker_receive(f, bucket=wl.bucket)
            v = r.rows.float() * r.row_scales.repeat_interleave(128, dim=1)
            replies.append(v.to(torch.bfloat16).contiguous())
            buf.worker_reply(f, replies[f], r.receipt)
        for s in range(wl.A):
            buf.source_collect(s, out=outs[s])
    _exchange(buf, wl, xs, ids, ws, scs, outs, replies)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _exchange(buf, wl, xs, ids, ws, scs, outs, replies)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # afd_l2_flush scratch
    for _ in range(3):
        g.replay()
    samples: dict = {}
    for _ in range(replays):
        if back_to_back:
            g.replay()
            g.replay()
            torch.cuda.synchronize()
            buf.phase_stamps(clear=True)
        else:
            st = afd.load_library().afd_l2_flush(flush.data_ptr(), flush.numel(),
                                                 torch.cuda.current_stream().cuda_stream)
            if st != 0:
                raise afd.AfdError(st, "afd_l2_flush")
            torch.cuda.synchronize()
            buf.phase_stamps(clear=True)
        g.replay()
        st = buf.phase_stamps(clear=False)
        t0 = st[0, :, 0][st[0, :, 0] > 0]
        if t0.size == 0:
            continue
        t0 = int(t0.min())
        for k, kind in enumerate(afd.STAMP_KINDS):
            for i in range(len(POINTS[kind])):
                v = st[k, :, i]
                v = v[v > 0]
                if v.size == 0:
                    continue
                rel = (v.astype(np.int64) - t0) / 1e3
                samples.setdefault((k, i), []).append((rel.min(), float(np.median(rel)), rel.max(), v.size))
    del g
    buf.close()
    lines = [f"{config} T={tokens} per source, {combine_mode}, "
             f"{'back to back' if back_to_back else 'L2 flushed'}, median of {replays} replays "
             f"(µs from the first dispatch block's start)",
             f"{'kernel':14s} {'point':28s} {'first':>8s} {'median':>8s} {'last':>8s} {'blocks':>7s}"]
    for (k, i), ss in sorted(samples.items()):
        kind = afd.STAMP_KINDS[k]
        lines.append(f"{kind:14s} {POINTS[kind][i]:28s} "
                     f"{statistics.median(x[0] for x in ss):8.2f} {statistics.median(x[1] for x in ss):8.2f} "
                     f"{statistics.median(x[2] for x in ss):8.2f} {ss[0][3]:7d}")
    return lines


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--config", default="2A2F")
    ap.add_argument("--tokens", type=int, default=2048)
    ap.add_argument("--replays", type=int, default=10)
    ap.add_argument("--back-to-back", action="store_true")
    ap.add_argument("--combine-mode", default="fused", choices=("fused", "two-stage", "two-stage-fp8"))
    a = ap.parse_args()
    print("\n".join(run(a.config, a.tokens, a.replays, a.back_to_back, a.combine_mode)))


if __name__ == "__main__":
    main()
