"""The C-ABI library builds, loads and exports every entry point that
include/afd.h declares. No compute calls: these run without a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "afd.h")


@pytest.fixture(scope="module")
def lib_path():
    from combine_attention_ffn_gb300 import build

    return build.build()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^AFD_API\s+[\w\s\*]+?\b(afd_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("afd_source_dispatch", "afd_worker_receive", "afd_worker_reply", "afd_source_collect",
              "afd_create", "afd_destroy", "afd_get_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (afd_\w+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported
    lib = ctypes.CDLL(lib_path)
    for n in declared_functions():
        assert hasattr(lib, n)


def test_binding_signatures_cover_the_header(lib_path):
    from combine_attention_ffn_gb300 import afd

    assert set(afd.EXPORTS) == set(declared_functions())
    lib = afd.load_library(lib_path)
    assert lib.afd_version() >> 16 == 0


def test_status_strings_and_no_device(lib_path):
    from combine_attention_ffn_gb300 import afd
    import torch

    lib = afd.load_library(lib_path)
    assert lib.afd_status_string(0) == b"ok"
    assert b"receipt" in lib.afd_status_string(afd.ERR_RECEIPT)
    assert b"wait" in lib.afd_status_string(afd.ERR_TIMEOUT)
    for code in range(12):  # every status has its own text
        assert lib.afd_status_string(code) != lib.afd_status_string(99)
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the no-device path is not reachable")
    cfg = afd.Config(2, 2, 8, 2, 256, 16, 1, 0, 0)
    h = ctypes.c_void_p()
    st = lib.afd_create(ctypes.byref(cfg), 0, ctypes.byref(h))
    assert st == afd.ERR_CUDA and not h.value


def test_bad_configs_rejected_before_any_device_work(lib_path):
    from combine_attention_ffn_gb300 import afd

    lib = afd.load_library(lib_path)
    bad = [
        afd.Config(2, 3, 8, 2, 256, 16, 1, 0, 0),     # E not a multiple of F
        afd.Config(2, 2, 8, 9, 256, 16, 1, 0, 0),     # K > E
        afd.Config(2, 2, 64, 33, 256, 16, 1, 0, 0),   # K > 32
        afd.Config(2, 2, 8, 2, 200, 16, 1, 0, 0),     # H not a multiple of 256
        afd.Config(2, 2, 8, 2, 256, 16, 0, 0, 0),     # alignment 0
        afd.Config(0, 2, 8, 2, 256, 16, 1, 0, 0),     # no sources
        afd.Config(2, 2, 8, 2, 256, 16, 1, 7, 0),     # unknown dtype
        afd.Config(2, 2, 2048, 2, 256, 16, 1, 0, 0),  # E above this build's limit
    ]
    for cfg in bad:
        h = ctypes.c_void_p()
        st = lib.afd_create(ctypes.byref(cfg), 0, ctypes.byref(h))
        assert st in (afd.ERR_ARG, afd.ERR_UNSUPPORTED), (cfg.num_experts, st)
        assert not h.value


def test_missing_library_fails_loudly(tmp_path):
    from combine_attention_ffn_gb300 import afd

    with pytest.raises(afd.AfdError):
        afd.load_library(str(tmp_path / "libafd.so"))


def test_noalloc_size_limits_are_host_checks(lib_path):
    """afd_route_layout_noalloc refuses sizes beyond its fixed scratch, and
    alignments whose largest row index would overflow int32, on the host
    before any CUDA call (so this runs without a GPU)."""
    from combine_attention_ffn_gb300 import afd

    lib = afd.load_library(lib_path)
    bogus = ctypes.c_void_p(16)
    for T, K, E, F, alpha in ((8193, 1, 16, 2, 4), (4096, 17, 32, 2, 1), (64, 8, 1025, 1, 1),
                              (8192, 8, 1024, 1, 1 << 21), (0, 1, 1024, 1, (1 << 31) - 1)):
        st = lib.afd_route_layout_noalloc(bogus, T, K, E, F, alpha, bogus, bogus, bogus, None)
        assert st == afd.ERR_UNSUPPORTED, (T, K, E, F, alpha)
    for T, K, E, F, alpha in ((-1, 1, 8, 1, 1), (4, 0, 8, 1, 1), (4, 9, 8, 1, 1), (4, 2, 9, 2, 1),
                              (4, 2, 8, 2, 0)):
        st = lib.afd_route_layout_noalloc(bogus, T, K, E, F, alpha, bogus, bogus, bogus, None)
        assert st == afd.ERR_ARG, (T, K, E, F, alpha)


def test_phase_stamps_only_in_the_timer_build(lib_path):
    """The default build has no phase timers: afd_phase_stamps answers
    AFD_ERR_UNSUPPORTED without touching a device. The timer build compiles
    (for sm_103a, here without a GPU) and exports the same entry points."""
    from combine_attention_ffn_gb300 import afd, build

    lib = afd.load_library(lib_path)
    assert lib.afd_phase_stamps(None, None, 0, 0) == afd.ERR_UNSUPPORTED
    timers = build.build_timers()
    assert timers != lib_path and os.path.exists(timers)
    out = subprocess.run(["nm", "-D", "--defined-only", timers], capture_output=True, text=True,
                         check=True).stdout
    assert set(declared_functions()) <= set(re.findall(r"\bT (afd_\w+)$", out, flags=re.M))


def test_l2_flush_checks_arguments_on_the_host(lib_path):
    """afd_l2_flush refuses a null, unaligned or badly sized scratch before
    it touches a device."""
    from combine_attention_ffn_gb300 import afd

    lib = afd.load_library(lib_path)
    assert lib.afd_l2_flush(None, 1 << 20, None) == afd.ERR_ARG
    assert lib.afd_l2_flush(ctypes.c_void_p(0x1000), 0, None) == afd.ERR_ARG
    assert lib.afd_l2_flush(ctypes.c_void_p(0x1000), 48, None) == afd.ERR_ARG      # not a multiple of 32
    assert lib.afd_l2_flush(ctypes.c_void_p(0x1008), 1 << 20, None) == afd.ERR_ARG  # not 16-byte aligned
