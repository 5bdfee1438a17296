"""Builds libafd.so (the C-ABI library) for sm_103a with nvcc.

Each translation unit compiles in parallel to an object under ``_build/``;
they are then linked into ``libafd.so`` next to this file. No GPU is needed
to build. ``python -m combine_attention_ffn_gb300.build`` runs it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libafd.so")
# The diagnostic phase-timer build (-DAFD_PHASE_TIMERS=1), kept apart.
BUILD_TIMERS = os.path.join(HERE, "_build", "timers")
LIB_TIMERS = os.path.join(HERE, "libafd_timers.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _compile(src: str, extra: list[str], build_dir: str = BUILD) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          out: str = LIB, build_dir: str = BUILD) -> str:
    """Compiles every csrc/*.cu and links libafd.so. Returns the library path."""
    os.makedirs(build_dir, exist_ok=True)
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(p) for p in _deps())
        if os.path.getmtime(out) >= newest:
            return out
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra or [], build_dir), srcs))
    log = "\n".join(r[1] for r in results)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as fh:
        fh.write(log)
    if verbose:
        print(log)
    tmp = out + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[r[0] for r in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def build_timers(force: bool = False) -> str:
    """The diagnostic library with phase timers (libafd_timers.so): the same
    kernels plus %globaltimer stamps (see afd_phase_stamps in afd.h)."""
    return build(force=force, extra=["-DAFD_PHASE_TIMERS=1"], out=LIB_TIMERS, build_dir=BUILD_TIMERS)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
