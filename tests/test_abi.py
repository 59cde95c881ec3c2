"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks answer without a GPU."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def _declared():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(ft_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    import moe_expert_cache_gb300 as ft
    if not os.path.exists(ft.LIB_PATH):
        from moe_expert_cache_gb300 import build
        build.build()
    return ft


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "ft_layer_init" in names and "ft_route_ctl" in names and "ft_moe_forward" in names
    assert "ft_prefill_layer" in names and "ft_cache_resize" in names
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing
    # and the binding wraps each of them
    assert set(names) <= set(lib._SIGS), set(names) - set(lib._SIGS)


def test_exported_symbols_are_c_linkage(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ft_[a-z0-9_]+)$", out, flags=re.M))
    assert set(_declared()) <= exported


def test_host_only_calls(lib):
    assert lib.abi_version() == 1
    assert lib.status_str(0) == "ok"
    assert lib.status_str(lib.FT_ERR_CAPACITY).startswith("cache too small")
    assert lib.record_bytes(2048, 768, lib.FT_FMT_BF16) == 9437184
    assert lib.record_bytes(64, 128, lib.FT_FMT_BF16) == 49152
    assert lib.record_bytes(4096, 2048, lib.FT_FMT_NVFP4) == 14155776
    import synth
    assert lib.record_bytes(4096, 2048, 1) == synth.record_bytes(4096, 2048, synth.FMT_NVFP4)
    assert lib.record_bytes(4096, 2048, lib.FT_FMT_MXFP4) == 13369344
    assert lib.record_bytes(4096, 2048, 2) == synth.record_bytes(4096, 2048, synth.FMT_MXFP4)
    assert lib.record_bytes(4096, 2048, lib.FT_FMT_FP8) == 3 * 4096 * 2048 + 12 * 32 * 16
    assert lib.record_bytes(4096, 2048, 3) == synth.record_bytes(4096, 2048, synth.FMT_FP8)
    assert lib.record_bytes(4096, 2048, 4) == 0


def test_argument_checks_need_no_gpu(lib):
    # each of these fails the host-side checks before any CUDA call
    assert lib.layer_init(0, 8, 2, 64, 128, 4, 0, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 9, 64, 128, 4, 0, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 60, 128, 4, 0, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 64, 128, 4, 0, 4, 0, None, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 64, 128, 0, 0, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    # record formats: unknown; MXFP4 with F % 512 != 0 or with a global; NVFP4 without one
    assert lib.layer_init(1, 8, 2, 256, 512, 4, 4, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 192, 256, 4, lib.FT_FMT_FP8, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 256, 256, 4, lib.FT_FMT_FP8, 4, 0, 1024, 4096, None, None)[0] == lib.FT_ERR_ARG
    # FP8 shapes whose records would not start on 16-byte boundaries: (H/128)*(F/128) = 1, 2, 3, 6
    for H, F in ((128, 128), (256, 128), (384, 128), (384, 256)):
        assert lib.layer_init(1, 8, 2, H, F, 4, lib.FT_FMT_FP8, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 256, 256, 4, lib.FT_FMT_MXFP4, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 256, 512, 4, lib.FT_FMT_MXFP4, 4, 0, 1024, 4096, None, None)[0] == lib.FT_ERR_ARG
    assert lib.layer_init(1, 8, 2, 256, 512, 4, lib.FT_FMT_NVFP4, 4, 0, 1024, None, None, None)[0] == lib.FT_ERR_ARG
    assert lib.route_ctl(None, 0, 1, None, None, None, 1.0, 1.0) == lib.FT_ERR_ARG
    assert lib.moe_forward(None, None, None, None) == lib.FT_ERR_ARG
    assert lib.cache_resize(None, 4) == lib.FT_ERR_ARG
    assert lib.get_status(None) == lib.FT_ERR_ARG
    lib.destroy(None)


def test_product_path_does_not_import_oracle():
    code = ("import sys, moe_expert_cache_gb300 as ft; ft.load(); "
            "bad=[m for m in sys.modules if m=='oracle' or m.startswith('oracle.')]; print(bad); "
            "sys.exit(1 if bad else 0)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_oracle_does_not_import_product():
    code = ("import sys, oracle.control, oracle.numerics, oracle.nvfp4; "
            "bad=[m for m in sys.modules if m.startswith('moe_expert_cache_gb300')]; "
            "sys.exit(1 if bad else 0)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
