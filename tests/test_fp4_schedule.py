"""The FP4 decode kernel's step order and fill-share arithmetic, checked on
the host (no GPU): a C++ program built from the kernel's own header
(moe_expert_cache_gb300/csrc/fp4_steps.cuh) checks that every phase-A item is
taken once, that each CTA seals each group after its phase-A items and before
the group's phase-B items, that the cross-CTA waits always complete, and that
the CTAs' fill shares tile every record exactly once in 16-byte-aligned
chunks (deepmox, "How residency follows demand without leaving the device":
a fill copies the complete record).  See the program's header for the list."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fp4_schedule_and_fill_shares(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "fp4_schedule_check"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "moe_expert_cache_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "csrc", "fp4_schedule_check.cpp"), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
