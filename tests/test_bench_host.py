"""Host-side logic of bench.py: the max-over-ranks reduction of the replica
path (world_size 2 over gloo on CPU), the reference arm's rank rule, and the
algorithmic byte count."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch, torch.distributed as dist
import bench
dist.init_process_group("gloo", rank=int(os.environ["RANK"]), world_size=2)
rank = dist.get_rank()
v = bench.reduce_max(10.0 + 5.0 * rank, torch.device("cpu"))
dist.barrier()
print("RESULT", rank, v, flush=True)
dist.destroy_process_group()
"""


def test_reduce_max_over_two_gloo_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    vals = sorted(line.split()[1:] for o, _ in outs for line in o.splitlines() if line.startswith("RESULT"))
    assert vals == [["0", "15.0"], ["1", "15.0"]]


def test_reduce_max_single_process_is_identity():
    import torch
    import bench

    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_algorithmic_bytes_match_the_formula():
    import bench
    from combine_attention_ffn_gb300 import workloads as W

    wl = W.named("2A2F", T=2048)
    inp = W.make_inputs(wl)
    ab = bench.algorithmic_bytes(wl, inp)
    V = 2 * 2048 * 8  # uniform routing: every slot valid
    assert ab["valid"] == V
    # payload: read x, write the routed rows, read the replies, write out
    assert ab["payload"] == 2 * 2048 * 4096 + V * 4096 + V * 4096 + 2 * 2048 * 4096
    assert ab["payload"] == 147456 * 2048


@pytest.mark.parametrize("mode", ["fused", "two-stage", "two-stage-fp8"])
def test_reference_arm_reports_the_combine_mode(mode):
    import json

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--tokens", "16", "--steps", "1", "--warmup", "1",
                        "--combine-mode", mode], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"]["combine"] == mode
    assert line["value"] > 0 and line["cpu_baseline"]["cores"] == 1


def test_pages_context_cells():
    """The pages' "Result" cells attached to sweep rows: the layout, hidden
    size and dtype must match, and only the pages' token counts have one."""
    import bench

    c = bench.pages_context("2A2F", 1)
    assert (c["afdEP_comm_us"], c["fastafd_m2n_us"]) == (20.7, 31.7)
    assert bench.pages_context("2A2F-H4096", 2048)["afdEP_comm_us"] == 383.2
    assert bench.pages_context("skew-3A1F", 512)["afdEP_comm_us"] == 109.4
    assert bench.pages_context("skew-1A3F", 32)["fastafd_m2n_us"] == 32.8
    assert bench.pages_context("fp8-2A2F", 128)["afdEP_comm_us"] == 34.5
    assert bench.pages_context("fp8-2A1F", 128) is None      # no such layout on the pages
    assert bench.pages_context("2A2F", 16) is None            # no such token count
    assert bench.pages_context("tiny", 16) is None
    for name, Ts, _ in bench.SWEEP:                          # every row's T is a workload's own
        assert all(T >= 1 for T in Ts)


def test_reference_arm_config_equals_ours_and_runs_fp8():
    """Both arms describe the workload with the same config dict; the
    reference arm also times the FP8 round trip (its expert stand-in untimed)."""
    import json

    import bench
    from combine_attention_ffn_gb300 import workloads as W

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "fp8-2A2F", "--tokens", "1", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    wl = W.named("fp8-2A2F", T=1)
    assert line["config"] == bench.workload_config(wl)
    assert line["dtype"] == "fp8" and line["value"] > 0
