"""Benchmark: MoE dispatch + combine round trip on one GB300.

One step is one complete exchange: every source dispatches, every worker
receives and replies (identity expert: the reply is the received rows, as in
the pages' communication-only numbers), every source collects. The exchange
is replayed from one CUDA graph; L2 is flushed (a 256 MB write, then a 256 MB
read) before every timed step, outside the step's events.

Prints ONE JSON line. `value` is microseconds per round trip (lower is
better). With --gpus N > 1 (torchrun), every rank runs an independent replica
(the exchange does not shard across GPUs) and the slowest rank's time is
reported. `--impl reference` times the CPU oracle instead, on this host.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "dispatch+combine µs/round trip; achieved HBM GB/s vs peak (E128 K8 H2048)"
COMBINE_MODES = {"fused": 0, "two-stage": 1, "two-stage-fp8": 2}  # afd_config.combine_mode
FALLBACK_HBM_GBS = 6800.0
# afdEP-comm design page, "Result" table: round trip in us, afdEP-comm (FastAFD M2N),
# 4 x H100 in one NVLink domain, communication only, random routing, CUDA graphs,
# 24 transport SMs, at T = 1, 8, 32, 128, 512, 2048 tokens per source. Context
# for the rows of the same layout, hidden size and dtype; not a target (other
# hardware, a multi-GPU transport).
PAGES_T = (1, 8, 32, 128, 512, 2048)
PAGES_RESULT_US = {
    "2A2F, H2048, BF16": ((20.7, 31.7), (24.8, 34.4), (26.3, 36.0), (35.3, 44.3), (70.6, 78.7), (192.7, 201.0)),
    "2A2F, H4096, BF16": ((28.4, 39.1), (39.2, 47.9), (46.3, 55.7), (61.5, 68.7), (127.3, 136.2), (383.2, 392.6)),
    "3A:1F, H2048, BF16": ((24.8, 36.4), (27.4, 38.6), (33.0, 44.8), (45.9, 55.8), (109.4, 119.5), (367.8, 372.1)),
    "1A:3F (E96), H2048, BF16": ((19.9, 30.5), (21.5, 31.3), (23.1, 32.8), (29.4, 39.7), (59.6, 67.7), (188.3, 197.7)),
    "2A2F, H2048, FP8 dispatch": ((21.3, 32.3), (25.9, 35.6), (26.8, 36.7), (34.5, 43.5), (62.5, 71.8), (159.1, 167.8)),
}
PAGES_ROW_OF = {"2A2F": "2A2F, H2048, BF16", "2A2F-H4096": "2A2F, H4096, BF16",
                "skew-3A1F": "3A:1F, H2048, BF16", "skew-1A3F": "1A:3F (E96), H2048, BF16",
                "fp8-2A2F": "2A2F, H2048, FP8 dispatch"}


def pages_context(name: str, T: int, combine: str = "fused"):
    """The pages' cell for this layout and token count, or None."""
    row = PAGES_ROW_OF.get(name)
    if row is None or T not in PAGES_T:
        return None
    ours, base = PAGES_RESULT_US[row][PAGES_T.index(T)]
    note = "4 x H100 NVLink, communication only, random routing; context, not a target"
    if name.startswith("skew"):
        note += " (this row's routing is skewed)"
    if combine != "fused":
        note += " (the pages' cell rounds per FFN rank like this row)"
    return {"pages_row": row, "afdEP_comm_us": ours, "fastafd_m2n_us": base, "note": note}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="2A2F")
    ap.add_argument("--combine-mode", choices=list(COMBINE_MODES), default="fused",
                    help="fused: one FP32 sum over every route, one rounding; two-stage: BF16 "
                         "partial per worker, then their FP32 sum; two-stage-fp8: the partials as "
                         "E4M3 with one power-of-two scale per 128 values")
    ap.add_argument("--tokens", type=int, default=2048, help="tokens per source")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--under-load", action="store_true",
                    help="time the exchange and a side-stream GEMM batch alone and together "
                         "(the pages' synthetic compute load) and print that record instead")
    ap.add_argument("--all-configs", action="store_true",
                    help="print only the sweep of every workload (no headline)")
    ap.add_argument("--profile-exchanges", type=int, default=0,
                    help="run this many eager exchanges of the workload and exit "
                         "(a short, untimed program for an external profiler)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def algorithmic_bytes(wl, inp) -> dict:
    """Bytes the exchange must move once (read x, write routed rows, read
    replies, write out) plus its metadata, per phase and per launch."""
    valid = 0
    for s, T in enumerate(wl.T):
        valid += int((inp.ids[s, :T] >= 0).sum())
    A, K, H = wl.A, wl.K, wl.H
    toks = sum(wl.T)
    R_in = wl.row_bytes + (4 * (H // 128) if wl.dtype == "fp8" else 0)
    dispatch = toks * R_in + valid * R_in + toks * K * (8 + 4) + valid * (4 + 4) + toks * K * (4 + 8)
    combine = valid * 2 * H + toks * 2 * H + toks * K * 8
    return dict(valid=valid, dispatch=dispatch, combine=combine,
                total=dispatch + combine,
                payload=toks * R_in + valid * R_in + valid * 2 * H + toks * 2 * H)


def host_cpu() -> dict:
    """The host's CPU model and core count, for the CPU-baseline record."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                model = line.split(":", 1)[1].strip()
                if model:
                    break
    except Exception:
        pass
    return {"model": model, "nproc": os.cpu_count()}


def native_digest() -> str:
    """Hash of the library's sources and header: names the native code a
    record was measured with."""
    import glob

    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "combine_attention_ffn_gb300", "csrc", "*")))
    for f in files + [os.path.join(ROOT, "include", "afd.h")]:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel's
    source has not changed since (profiles/traffic.txt)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "combine_attention_ffn_gb300", "csrc",
                       "afd_combine.cu" if kernel == "combine" else "afd_dispatch.cu")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        for line in open(path):
            parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if parts.get("kernel") == kernel and parts.get("source_sha") == sha \
                    and parts.get("workload") == workload:
                return float(parts["bytes_per_launch"])
    except Exception:
        pass
    return None


class L2Flush:
    """Evicts L2 (129 MB) between timed steps, outside the steps' events: a
    256 MB write, then a 256 MB read of another buffer, so that the write's
    dirty lines are written back before the step starts instead of during it.
    The step then finds none of its inputs in L2. Both passes use an L2
    evict-last policy (afd_l2_flush): the scatter writes its rows with that
    policy, and ordinary writes and reads would not evict them."""

    KERNELS = 3  # launches per flush: write, read, discard

    def __init__(self, torch, dev):
        self.scratch = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.torch = torch
        from combine_attention_ffn_gb300 import afd

        self.lib = afd.load_library(afd.LIB_PATH)  # the in-tree library, whichever one is in use
        self.afd = afd

    def __call__(self):
        stream = self.torch.cuda.current_stream(self.scratch.device).cuda_stream
        st = self.lib.afd_l2_flush(self.scratch.data_ptr(), self.scratch.numel(), stream)
        if st != 0:
            raise RuntimeError(f"afd_l2_flush failed (status {st})")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons),
                "window": "1 s of back-to-back replays just before the timed region, and the region"}


def reduce_max(value: float, device) -> float:
    """The slowest rank's value (replicas: every rank timed its own exchange)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ reference arm
def cpu_oracle_round_trip_us(wl, inp, budget_s: float, min_reps: int = 1, combine_mode: str = "fused"):
    """Times the oracle's round trip on this host: validate, layout, dispatch
    and combine. The expert between dispatch and combine is harness work on
    both sides (identity: the replies are the received rows; FP8: the rows
    dequantised to BF16 by the oracle's stand-in) and is not timed, as on the
    GPU side."""
    import oracle

    p = oracle.Problem(wl.A, wl.F, wl.E, wl.K, wl.H, wl.alpha, wl.bucket,
                       oracle.FP8 if wl.dtype == "fp8" else oracle.BF16, list(wl.T))
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < min_reps or time.perf_counter() < t_end:
        t0 = time.perf_counter()
        oracle.validate(p, inp.ids)
        lay = oracle.layout(p, inp.ids)
        r_stride = max(1, int(lay["r_exact"].max()))
        d = oracle.dispatch(p, inp.ids, inp.w, inp.x, inp.x_scales, lay, r_stride)
        t1 = time.perf_counter()
        if wl.dtype == "fp8":
            reply = oracle.expert(p, oracle.EXPERT_IDENTITY, lay, r_stride, d["rows"], d["row_scales"])
        else:
            reply = d["rows"].view(np.uint16).reshape(wl.F, r_stride, wl.H)
        t2 = time.perf_counter()
        if combine_mode == "fused":
            oracle.combine(p, inp.ids, inp.w, d["slot"], r_stride, reply)
        else:
            oracle.combine_two_stage(p, inp.ids, inp.w, d["slot"], r_stride, reply,
                                     fp8=combine_mode == "two-stage-fp8")
        t3 = time.perf_counter()
        times.append(((t1 - t0) + (t3 - t2)) * 1e6)
    return times


def oracle_reps(T: int) -> int:
    """Repeats of the per-row oracle timing: 3, or 5 for small batches."""
    return 5 if T <= 128 else 3


def run_reference(args):
    ws, rank, _ = dist_env()
    from combine_attention_ffn_gb300 import workloads as W

    if rank != 0:
        return 0
    wl = W.named(args.config, T=args.tokens)
    inp = W.make_inputs(wl)
    cpu_oracle_round_trip_us(wl, inp, 0.0, min_reps=args.warmup, combine_mode=args.combine_mode)  # warm-up
    steps = cpu_oracle_round_trip_us(wl, inp, 0.0, min_reps=args.steps, combine_mode=args.combine_mode)
    value = statistics.mean(steps)
    ab = algorithmic_bytes(wl, inp)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": workload_config(wl, combine=args.combine_mode),
        "execution": "CPU oracle (single-threaded C) on the host; the expert stand-in is not timed",
        "l2": "not applicable",
        "gbs": round(ab["total"] / (value * 1e-6) / 1e9, 2),
        "cpu_baseline": {"value": round(value, 1), "unit": "us", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} full round trips of the workload, single-threaded C oracle",
                         "host": host_cpu()},
        "e2e": {"value": round(value, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "native_digest": native_digest(),
    }
    print(json.dumps(line))
    return 0


L2_NOTE = ("flushed before every timed step (256 MB write, then 256 MB read of another buffer so "
           "the write-backs finish first, both with an L2 evict-last policy so that lines of every "
           "priority are evicted; outside the step's events)")


def workload_config(wl, combine: str = "fused") -> dict:
    return {"workload": f"{wl.name}: A={wl.A} sources x T={wl.T[0]} tokens, F={wl.F} workers, "
                        f"E={wl.E}, K={wl.K}, H={wl.H}, {wl.dtype}, alpha={wl.alpha}, "
                        f"bucket={wl.bucket}, {wl.routing} routing",
            "A": wl.A, "F": wl.F, "E": wl.E, "K": wl.K, "H": wl.H, "T_per_source": wl.T[0],
            "bucket": wl.bucket, "expert_alignment": wl.alpha, "routing": wl.routing,
            "expert": "identity (reply = received rows)" if wl.dtype == "bf16" else
                      "BF16 replies computed once from the received rows, outside the timed graph",
            "combine": combine}


# ------------------------------------------------------------------ our arm
class Rig:
    """One workload's exchange, ready to replay: inputs resident in device
    memory, the context, and the BF16 replies. BF16 replies are the received
    rows (identity expert, as in the pages' communication-only numbers); FP8
    replies are the received rows dequantised to BF16 once, from a first
    exchange outside any timed region (routing and rows do not change between
    replays, so they stay the right replies)."""

    def __init__(self, torch, afd, W, name, T, dev, combine="fused", num_sms=0):
        self.torch = torch
        wl = self.wl = W.named(name, T=T)
        inp = self.inp = W.make_inputs(wl)
        self.buf = afd.Buffer(wl.A, wl.F, wl.E, wl.K, wl.H, wl.capacity, wl.alpha, wl.dtype,
                              num_sms=num_sms, combine_mode=COMBINE_MODES[combine])
        fp8 = self.fp8 = wl.dtype == "fp8"
        if fp8:
            self.xs = [torch.from_numpy(inp.x[s, :t].copy()).to(dev).view(torch.float8_e4m3fn)
                       for s, t in enumerate(wl.T)]
            self.scs = [torch.from_numpy(inp.x_scales[s, :t].copy()).to(dev) for s, t in enumerate(wl.T)]
        else:
            self.xs = [torch.from_numpy(inp.x[s, :t].view(np.int16).copy()).to(dev).view(torch.bfloat16)
                       for s, t in enumerate(wl.T)]
            self.scs = [None] * wl.A
        self.ids = [torch.from_numpy(inp.ids[s, :t].copy()).to(dev) for s, t in enumerate(wl.T)]
        self.ws = [torch.from_numpy(inp.w[s, :t].copy()).to(dev) for s, t in enumerate(wl.T)]
        self.outs = [torch.empty((t, wl.H), dtype=torch.bfloat16, device=dev) for t in wl.T]
        self.replies = None
        if fp8:
            replies = {}

            def expert(f, r):
                v = r.rows.float() * r.row_scales.repeat_interleave(128, dim=1)
                replies[f] = v.to(torch.bfloat16).contiguous()
                return replies[f]

            self.exchange(expert=expert)
            torch.cuda.synchronize()
            self.replies = replies

    def exchange(self, view=False, cached=False, batched=False, expert=None):
        wl, buf = self.wl, self.buf
        for s in range(wl.A):
            if cached:
                buf.source_dispatch_cached(s, self.xs[s], self.ws[s], self.scs[s], bucket=wl.bucket)
            else:
                buf.source_dispatch(s, self.xs[s], self.ids[s], self.ws[s], self.scs[s], bucket=wl.bucket)
        for f in range(wl.F):
            r = buf.worker_receive(f, bucket=wl.bucket)
            reply = expert(f, r) if expert else (self.replies[f] if self.fp8 else r.rows)
            buf.worker_reply(f, reply, r.receipt)
        if batched:
            buf.source_collect_all(view=view, outs=None if view and wl.F == 1 else self.outs)
        else:
            for s in range(wl.A):
                buf.source_collect(s, out=None if view and wl.F == 1 else self.outs[s], view=view)

    def graph(self, **kw):
        """One exchange captured as a CUDA graph (after one eager exchange)."""
        torch = self.torch
        self.exchange(**kw)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.exchange(**kw)
        return g

    def close(self):
        self.buf.close()


def replay_stats(torch, g, flush, n_flushed: int = 20, n_btb: int = 50):
    """Mean µs of one replay with L2 flushed before it (outside its events),
    and mean µs of n_btb replays back to back. Event timestamps fall on a
    grid of about 2 µs on this hardware, so a median of single replays sits
    on a grid point; the mean of many resolves finer."""
    for _ in range(3):
        g.replay()
    times = []
    for _ in range(n_flushed):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n_btb):
        g.replay()
    b.record()
    b.synchronize()
    return statistics.mean(times), a.elapsed_time(b) * 1e3 / n_btb


# Rows of the default run: every workload at the token counts of its
# benchmark, and the pages' per-worker rounding (two-stage combine).
SWEEP = (("tiny", (16,), "fused"), ("2A2F", (1, 8, 32, 128, 512, 2048), "fused"),
         ("2A2F-H4096", (1, 128, 2048), "fused"), ("skew-3A1F", (1, 32, 512, 2048), "fused"),
         ("skew-1A3F", (1, 32, 512, 2048), "fused"), ("fp8-2A2F", (1, 128, 2048), "fused"),
         ("fp8-2A1F", (1, 128, 2048), "fused"),
         ("2A2F", (1, 128, 512, 2048), "two-stage"), ("2A2F", (1, 128, 512, 2048), "two-stage-fp8"))


def measure_sweep(torch, afd, W, dev, flush, peak, with_oracle=True):
    """Every row of SWEEP, one CUDA graph replay per round trip: mean µs after
    an L2 flush and back to back (median of three such measurements),
    algorithmic bytes, GB/s and the fraction of
    the HBM peak (from 512 tokens per source; below, the round trip is bound
    by latency), the pages' cell for the same layout as context, and the
    oracle's time for the same round trip on this host. Single-worker
    layouts also collect through the view; the 2A2F layouts also with a
    cached dispatch and with one batched collect."""
    rows = []
    for name, Ts, mode in SWEEP:
        for T in Ts:
            rig = Rig(torch, afd, W, name, T, dev, combine=mode)
            wl, inp = rig.wl, rig.inp
            variants = [("full", {})]
            if wl.F == 1:
                variants.append(("view", dict(view=True)))
            if name in ("2A2F", "2A2F-H4096") and mode == "fused":
                variants += [("cached", dict(cached=True)), ("batched collect", dict(batched=True))]
            for label, kw in variants:
                g = rig.graph(**kw)
                # median of three measurements: single replays fall on a ~2 µs grid, and
                # a back-to-back run settles on one grid step or the next
                stats = [replay_stats(torch, g, flush) for _ in range(3)]
                us = statistics.median(x[0] for x in stats)
                btb = statistics.median(x[1] for x in stats)
                del g
                ab = algorithmic_bytes(wl, inp)
                gbs = ab["total"] / (us * 1e-6) / 1e9
                row = {"config": name, "T": T, "combine": mode, "variant": label, "us": round(us, 2),
                       "us_back_to_back": round(btb, 2), "bytes": int(ab["total"]), "gbs": round(gbs, 1),
                       "frac": round(gbs / peak, 4) if T >= 512 else None}
                if label == "full":
                    row["context"] = pages_context(name, T, mode)
                    if with_oracle:
                        n = oracle_reps(T)
                        row["oracle_us"] = round(statistics.median(
                            cpu_oracle_round_trip_us(wl, inp, 0.0, min_reps=n, combine_mode=mode)), 1)
                        row["oracle_reps"] = n
                rows.append(row)
            torch.cuda.synchronize()
            rig.close()
    return rows


def measure_under_load(torch, afd, W, dev, name="2A2F", Ts=(512, 2048), settings=((0, False), (24, False)),
                       n_ex: int = 100, n_gemm: int = 100):
    """The exchange under compute load (afdEP-comm design page, section 14:
    a fixed batch of 2,048^3 BF16 GEMMs on a side stream while the exchanges
    replay). Per token count and (SM cap, exchange stream priority): GEMM time
    alone and under the exchanges, exchange time alone and under the GEMMs,
    and the makespan of both."""
    side_s = torch.cuda.Stream()
    a = torch.randn(2048, 2048, device=dev, dtype=torch.bfloat16)
    b = torch.randn(2048, 2048, device=dev, dtype=torch.bfloat16)
    c = torch.empty(2048, 2048, device=dev, dtype=torch.bfloat16)

    def gemms():
        for _ in range(n_gemm):
            torch.matmul(a, b, out=c)

    rows = []
    for T in Ts:
        for sms, prio in settings:
            rig = Rig(torch, afd, W, name, T, dev, num_sms=sms)
            main_s = torch.cuda.Stream(priority=torch.cuda.Stream.priority_range()[1]) if prio \
                else torch.cuda.default_stream()
            torch.cuda.set_stream(main_s)

            def span(fn_main, fn_side):
                e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                torch.cuda.synchronize()
                e[0].record(main_s)
                side_s.wait_event(e[0])
                if fn_side:
                    with torch.cuda.stream(side_s):
                        e[2].record(side_s)
                        fn_side()
                        e[3].record(side_s)
                if fn_main:
                    fn_main()
                e[1].record(main_s)
                torch.cuda.synchronize()
                t_main = e[0].elapsed_time(e[1]) * 1e3 if fn_main else None
                t_side = e[2].elapsed_time(e[3]) * 1e3 if fn_side else None
                make = max(e[0].elapsed_time(e[1]), e[0].elapsed_time(e[3]) if fn_side else 0) * 1e3
                return t_main, t_side, make

            g = rig.graph()

            def replays():
                for _ in range(n_ex):
                    g.replay()

            span(replays, gemms)  # warm-up
            ex_alone, _, _ = span(replays, None)
            _, gemm_alone, _ = span(None, gemms)
            ex_load, gemm_load, make = span(replays, gemms)
            rows.append({"T": T, "num_sms": sms, "exchange_stream": "high priority" if prio else "default",
                         "exchange_us_alone": round(ex_alone / n_ex, 2),
                         "exchange_us_under_load": round(ex_load / n_ex, 2),
                         "gemm_us_alone": round(gemm_alone / n_gemm, 2),
                         "gemm_us_under_load": round(gemm_load / n_gemm, 2),
                         "gemm_slowdown": round(gemm_load / gemm_alone - 1, 4),
                         "makespan_ms": round(make / 1e3, 3)})
            del g
            rig.close()
            torch.cuda.set_stream(torch.cuda.default_stream())
    return rows


def run_under_load(args):
    """The full under-load table (more token counts and settings than the
    default run's block)."""
    import torch

    from combine_attention_ffn_gb300 import afd
    from combine_attention_ffn_gb300 import build as libbuild
    from combine_attention_ffn_gb300 import workloads as W

    libbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    rows = measure_under_load(torch, afd, W, dev, args.config, Ts=(1, 32, 512, 2048),
                              settings=((0, False), (64, False), (24, False), (0, True)),
                              n_ex=200, n_gemm=200)
    print(json.dumps({"metric": "exchange and side-stream GEMM under load", "mode": "under_load",
                      "config": {"workload": args.config, "gemm": "2048^3 BF16 (torch.matmul) x 200",
                                 "exchanges": 200, "execution": "one CUDA graph per exchange"},
                      "rows": rows}))
    return 0


def run_sweep_only(args):
    """Only the sweep of every workload (no headline), as one JSON line."""
    import torch

    from combine_attention_ffn_gb300 import afd
    from combine_attention_ffn_gb300 import build as libbuild
    from combine_attention_ffn_gb300 import workloads as W

    libbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peak, peak_kind = load_peaks()
    rows = measure_sweep(torch, afd, W, dev, L2Flush(torch, dev), peak, with_oracle=not args.no_cpu_baseline)
    print(json.dumps({"metric": METRIC, "mode": "sweep", "unit": "us", "peak_gbs": peak,
                      "peak_kind": peak_kind, "native_digest": native_digest(), "l2": L2_NOTE,
                      "host": host_cpu(), "rows": rows}))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.under_load:
        return run_under_load(args)
    if args.all_configs:
        return run_sweep_only(args)

    import warnings

    import torch

    # the receive/reply phase graph holds no kernel (only host checks)
    warnings.filterwarnings("ignore", message="The CUDA Graph is empty")
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from combine_attention_ffn_gb300 import afd
    from combine_attention_ffn_gb300 import build as libbuild
    from combine_attention_ffn_gb300 import workloads as W

    # one rank builds (if the sources are newer than the library), the others wait
    if rank == 0:
        libbuild.build()
    if ws > 1:
        torch.distributed.barrier()
    wl = W.named(args.config, T=args.tokens)
    if wl.dtype == "fp8":
        if not args.profile_exchanges:
            raise SystemExit("the headline times the BF16 identity-expert round trip; FP8 rows are in the sweep")
        # an untimed program for an external profiler: the sweep's FP8 exchange
        # (its replies computed once by the stand-in expert), repeated
        rig = Rig(torch, afd, W, args.config, args.tokens, dev, combine=args.combine_mode)
        for _ in range(args.profile_exchanges):
            rig.exchange()
        torch.cuda.synchronize()
        rig.close()
        print(f"ran {args.profile_exchanges} exchanges of {wl.name} T={wl.T[0]}")
        return 0
    inp = W.make_inputs(wl)
    buf = afd.Buffer(wl.A, wl.F, wl.E, wl.K, wl.H, wl.capacity, wl.alpha, wl.dtype,
                     combine_mode=COMBINE_MODES[args.combine_mode])
    buf_small = sum(wl.T) * wl.K <= 2048 or sum(wl.T) <= 32  # one-kernel dispatch (afd_dispatch.cu)

    xs = [torch.from_numpy(inp.x[s, :T].view(np.int16).copy()).to(dev).view(torch.bfloat16)
          for s, T in enumerate(wl.T)]
    ids = [torch.from_numpy(inp.ids[s, :T].copy()).to(dev) for s, T in enumerate(wl.T)]
    ws_ = [torch.from_numpy(inp.w[s, :T].copy()).to(dev) for s, T in enumerate(wl.T)]
    outs = [torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev) for T in wl.T]

    def dispatch_all():
        for s in range(wl.A):
            buf.source_dispatch(s, xs[s], ids[s], ws_[s], bucket=wl.bucket)

    def receive_reply_all():
        for f in range(wl.F):
            r = buf.worker_receive(f, bucket=wl.bucket)
            buf.worker_reply(f, r.rows, r.receipt)  # identity expert

    def collect_all():
        for s in range(wl.A):
            buf.source_collect(s, out=outs[s])

    def exchange():
        dispatch_all()
        receive_reply_all()
        collect_all()

    if args.profile_exchanges:
        for _ in range(args.profile_exchanges):
            exchange()
        torch.cuda.synchronize()
        buf.close()
        print(f"ran {args.profile_exchanges} exchanges of {wl.name} T={wl.T[0]}")
        return 0

    # warm up eagerly, then capture one round trip as one graph (the headline),
    # and one more exchange as three graphs, one per phase, for the per-kernel
    # times (an event between kernels inside one graph would cut the
    # programmatic-launch edges and slow the headline down)
    for _ in range(2):
        exchange()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        exchange()
    def exchange_batched():
        dispatch_all()
        receive_reply_all()
        buf.source_collect_all(outs=outs)

    exchange_batched()
    torch.cuda.synchronize()
    g_batched = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_batched):
        exchange_batched()
    g_phase = []
    for fn in (dispatch_all, receive_reply_all, collect_all):
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp):
            fn()
        g_phase.append(gp)
    flush = L2Flush(torch, dev)
    for _ in range(max(3, args.warmup)):
        flush()
        g.replay()
        for gp in g_phase:
            gp.replay()
    torch.cuda.synchronize()
    # The timed region is short next to nvidia-smi's sampling period, so the
    # sampler also covers one second of back-to-back replays just before it.
    clocks = ClockSampler(dev.index)
    clocks.start()
    soak_end = time.perf_counter() + 1.0
    while time.perf_counter() < soak_end:
        for _ in range(200):
            g.replay()
        torch.cuda.synchronize()

    # timed region: each step is one replay of the round trip, L2 flushed
    # before it; after it (outside the step's events) the same exchange runs
    # phase by phase for the per-kernel times
    def ev():
        return torch.cuda.Event(enable_timing=True)

    steps_ev = [(ev(), ev()) for _ in range(args.steps)]
    batched_ev = [(ev(), ev()) for _ in range(args.steps)]
    phase_ev = [[ev() for _ in range(4)] for _ in range(args.steps)]
    cold_ev = [[(ev(), ev()) for _ in range(3)] for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush()
        steps_ev[i][0].record()
        g.replay()
        steps_ev[i][1].record()
        flush()
        pe = phase_ev[i]
        pe[0].record()
        for j, gp in enumerate(g_phase):
            gp.replay()
            pe[j + 1].record()
        for j, gp in enumerate(g_phase):  # each phase alone, L2 flushed before it
            flush()
            cold_ev[i][j][0].record()
            gp.replay()
            cold_ev[i][j][1].record()
        flush()
        batched_ev[i][0].record()
        g_batched.replay()
        batched_ev[i][1].record()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in steps_ev]
    ms = reduce_max(sum(step_ms) / len(step_ms), dev)
    batched_us = statistics.mean(a.elapsed_time(b) for a, b in batched_ev) * 1e3

    # the same round trip replayed back to back (L2 not flushed) and issued
    # eagerly call by call (L2 flushed), outside the timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(50):
        g.replay()
    e1.record()
    e1.synchronize()
    btb_us = e0.elapsed_time(e1) * 1e3 / 50
    eager = []
    for _ in range(10):
        flush()
        e0.record()
        exchange()
        e1.record()
        e1.synchronize()
        eager.append(e0.elapsed_time(e1) * 1e3)
    eager_us = statistics.median(eager)
    d_ms = statistics.mean(pe[0].elapsed_time(pe[1]) for pe in phase_ev)
    r_ms = statistics.mean(pe[1].elapsed_time(pe[2]) for pe in phase_ev)
    c_ms = statistics.mean(pe[2].elapsed_time(pe[3]) for pe in phase_ev)
    d_cold, r_cold, c_cold = (statistics.mean(ce[j][0].elapsed_time(ce[j][1]) for ce in cold_ev)
                              for j in range(3))

    ab = algorithmic_bytes(wl, inp)
    peak, peak_kind = load_peaks()
    us = ms * 1e3
    launches_per_step = (1 if buf_small else 2) + wl.A

    # dominant kernel: the combine has the largest share of the launch list
    # (profiles/launches_*.md), one launch per source, all in the collect
    # phase; the receive/reply phase launches no kernel at all. The dispatch
    # phase (layout + scatter) is reported too.
    n_launch = wl.A
    per_launch_s = c_ms / n_launch * 1e-3
    per_launch_bytes = ab["combine"] / n_launch
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kname = "combine_token_kernel" if sum(wl.T) // n_launch >= 4 * n_sms else (
        "combine_kernel" if args.combine_mode == "fused" else "combine_two_stage_kernel")
    if args.combine_mode != "fused":
        kname += f" ({args.combine_mode})"
    achieved = per_launch_bytes / per_launch_s / 1e9
    traffic = kernel_traffic("combine", f"{wl.name}-T{wl.T[0]}") if args.combine_mode == "fused" else None
    d_gbs = ab["dispatch"] / (d_ms * 1e-3) / 1e9
    comb_cold_s = c_cold / n_launch * 1e-3
    cold_achieved = per_launch_bytes / comb_cold_s / 1e9
    d_cold_gbs = ab["dispatch"] / (d_cold * 1e-3) / 1e9
    roofline = {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "bytes_per_launch": int(per_launch_bytes),
                "us_per_launch": round(per_launch_s * 1e6, 2),
                "phase_us": {"dispatch": round(d_ms * 1e3, 2),
                             "receive_reply": round(r_ms * 1e3, 2),
                             "collect": round(c_ms * 1e3, 2)},
                "dispatch_phase": {"us": round(d_ms * 1e3, 2), "bytes": int(ab["dispatch"]),
                                   "achieved": round(d_gbs, 1), "frac": round(d_gbs / peak, 4)},
                "cold": {"us_per_launch": round(comb_cold_s * 1e6, 2), "achieved": round(cold_achieved, 1),
                         "frac": round(cold_achieved / peak, 4),
                         "phase_us": {"dispatch": round(d_cold * 1e3, 2), "receive_reply": round(r_cold * 1e3, 2),
                                      "collect": round(c_cold * 1e3, 2)},
                         "dispatch_phase_frac": round(d_cold_gbs / peak, 4),
                         "note": "each phase's graph replayed alone with L2 flushed before it: the "
                                 "combine finds none of the replies in L2"},
                "note": "us_per_launch/frac: the per-phase graphs replayed one after another after "
                        "each timed step, L2 flushed before the first (dispatch) phase only, as in "
                        "the round trip: the combine finds the part of the scatter's rows that is "
                        "still in L2"}

    # end to end through the public API, host buffers, copies inside the region
    e2e = None
    if rank == 0 or ws > 1:
        e2e = measure_e2e(torch, buf, wl, inp, dev, steps=max(5, args.steps // 2), flush=flush)
        if ws > 1:  # the slowest rank, as for the headline
            e2e["value"] = round(reduce_max(e2e["value"], dev), 2)

    sweep = under_load = None
    if not args.no_sweep and rank == 0:
        sweep = measure_sweep(torch, afd, W, dev, flush, peak, with_oracle=not args.no_cpu_baseline)
        under_load = {"rows": measure_under_load(torch, afd, W, dev),
                      "note": "100 replays of the exchange (one CUDA graph each) and 100 BF16 "
                              "2048^3 GEMMs (torch.matmul) on a side stream, alone and together; "
                              "num_sms caps the exchange's kernels"}

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and ws == 1:  # the oracle runs at N = 1 only
        times = cpu_oracle_round_trip_us(wl, inp, args.cpu_seconds, combine_mode=args.combine_mode)
        cpu = {"value": round(statistics.median(times), 1), "unit": "us", "cores": 1, "kind": "oracle",
               "sample": f"{len(times)} full round trips of the same workload "
                         f"(validate, layout, dispatch, combine; the expert stand-in untimed), "
                         f"single-threaded C",
               "host": host_cpu()}

    buf.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(us, 2), "unit": "us", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic", "config": workload_config(wl, combine=args.combine_mode),
            "execution": "one CUDA graph per round trip", "l2": L2_NOTE,
            "gbs": round(ab["total"] / (us * 1e-6) / 1e9, 1),
            "hbm_frac_of_peak": round(ab["total"] / (us * 1e-6) / 1e9 / peak, 4),
            "peak_gbs": peak, "peak_kind": peak_kind,
            "algorithmic_bytes": ab["total"],
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": (4 * launches_per_step - (wl.A - 1) + 6 * L2Flush.KERNELS) * args.steps,
            "gpu_launches_note": "per step: the round-trip graph, the same exchange phase by phase "
                                 "(one after another, then each after an L2 flush), the round trip "
                                 "with one batched collect, and the six L2 flushes between them "
                                 "(afd_l2_flush: three kernels each, outside every event pair)",
            "back_to_back_us": round(btb_us, 2),
            "eager_us": round(eager_us, 2),
            "collect_all_us": round(batched_us, 2),
            "collect_all_note": "the same round trip with afd_source_collect_all (one combine "
                                "launch for every source) in place of one collect per source",
            "wall_s": round(wall, 3),
            "context": pages_context(args.config, wl.T[0], args.combine_mode),
            "sweep": sweep,
            "under_load": under_load,
            "native_digest": native_digest(),
        }
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def measure_e2e(torch, buf, wl, inp, dev, steps: int, flush):
    """Host buffers in, host result out: pinned H2D of x, ids and weights,
    the four calls, D2H of the outputs, every step."""
    hx = [torch.from_numpy(inp.x[s, :T].view(np.int16).copy()).pin_memory() for s, T in enumerate(wl.T)]
    hid = [torch.from_numpy(inp.ids[s, :T].copy()).pin_memory() for s, T in enumerate(wl.T)]
    hw = [torch.from_numpy(inp.w[s, :T].copy()).pin_memory() for s, T in enumerate(wl.T)]
    hout = [torch.empty((T, wl.H), dtype=torch.int16).pin_memory() for T in wl.T]
    dx = [torch.empty((T, wl.H), dtype=torch.int16, device=dev) for T in wl.T]
    did = [torch.empty((T, wl.K), dtype=torch.int64, device=dev) for T in wl.T]
    dw = [torch.empty((T, wl.K), dtype=torch.float32, device=dev) for T in wl.T]
    dout = [torch.empty((T, wl.H), dtype=torch.bfloat16, device=dev) for T in wl.T]
    h2d = sum(t.numel() * t.element_size() for t in hx + hid + hw)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def step():
        for s in range(wl.A):
            dx[s].copy_(hx[s], non_blocking=True)
            did[s].copy_(hid[s], non_blocking=True)
            dw[s].copy_(hw[s], non_blocking=True)
        for s in range(wl.A):
            buf.source_dispatch(s, dx[s].view(torch.bfloat16), did[s], dw[s], bucket=wl.bucket)
        for f in range(wl.F):
            r = buf.worker_receive(f, bucket=wl.bucket)
            buf.worker_reply(f, r.rows, r.receipt)
        for s in range(wl.A):
            buf.source_collect(s, out=dout[s])
            hout[s].copy_(dout[s].view(torch.int16), non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()

    def timed(run):
        times = []
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        return statistics.mean(times) * 1e3

    def replayed(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        us = timed(g.replay)
        del g
        return us

    eager_us = timed(step)
    # the same step, copies included, captured once and replayed
    graph_us = replayed(step)
    copied = [o.clone() for o in hout]

    # zero-copy: the pinned host buffers go to the calls as they are; the
    # dispatch kernels read x, ids and weights over the host link and the
    # combine writes the results there
    hout_bf = [o.view(torch.bfloat16) for o in hout]
    for o in hout:
        o.zero_()

    def step_zero_copy():
        for s in range(wl.A):
            buf.source_dispatch(s, hx[s].view(torch.bfloat16), hid[s], hw[s], bucket=wl.bucket)
        for f in range(wl.F):
            r = buf.worker_receive(f, bucket=wl.bucket)
            buf.worker_reply(f, r.rows, r.receipt)
        for s in range(wl.A):
            buf.source_collect(s, out=hout_bf[s])

    for _ in range(3):
        step_zero_copy()
    torch.cuda.synchronize()
    if not all(torch.equal(a, b) for a, b in zip(copied, hout)):
        raise RuntimeError("zero-copy results differ from the copied ones")
    zc_eager_us = timed(step_zero_copy)
    zc_graph_us = replayed(step_zero_copy)
    best = "zero-copy" if zc_graph_us < graph_us else "copies"
    return {"value": round(min(graph_us, zc_graph_us), 2), "unit": "us",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "method": best,
            "copies_us": round(graph_us, 2), "copies_eager_us": round(eager_us, 2),
            "zero_copy_us": round(zc_graph_us, 2), "zero_copy_eager_us": round(zc_eager_us, 2),
            "note": "per step, from pinned host inputs to pinned host results, through the "
                    "four calls. copies: cudaMemcpyAsync of x, ids and weights to the device, "
                    "the calls on device buffers, the outputs copied back. zero-copy: the "
                    "pinned buffers passed to the calls, which read and write them over the "
                    "host link. *_us = the step captured once as a CUDA graph and replayed, "
                    "*_eager_us = issued call by call; value = the faster method"}


if __name__ == "__main__":
    sys.exit(main())
