"""bench.py's host-side accounting on CPU: the algorithmic bytes of a decode
launch, the choice of the bounding side of the roofline, and the DRAM
traffic taken from a committed capture (scaled by records read, dropped once
the kernel source changes)."""
import hashlib
import json
import os
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_kernel_bytes_counts_fills_hits_and_activations():
    sh = synth.Shape(L=1, E=8, k=2, H=64, F=128)
    rb = sh.record_bytes
    d = {"calls": 3, "fills": 2, "hits": 4, "assign": 10}
    T = 2
    kb = bench.kernel_bytes(sh, T, d)
    link = 2 * rb
    assert kb["expert_ffn"]["link"] == link
    # fills written + hit records read + x (bf16) + h written and read (fp32) + partial_C and y (fp32)
    assert kb["expert_ffn"]["hbm"] == link + 4 * rb + 3 * T * 64 * 2 + 2 * 10 * 128 * 4 + 3 * T * 64 * 4 * 2
    assert kb["route_ctl"]["hbm"] == 3 * (T * 8 * 4 + 2 * T * 2 * 4)


def _kernels(link_bytes, hbm_bytes, us):
    gbs = lambda b: b / (us * 1e-6) / 1e9  # noqa: E731
    return {"expert_ffn": {"us_per_launch": us,
                           "link": {"bytes_per_launch": link_bytes, "achieved_GBps": gbs(link_bytes),
                                    "peak_GBps": 200.0, "frac": gbs(link_bytes) / 200.0},
                           "hbm": {"bytes_per_launch": hbm_bytes, "achieved_GBps": gbs(hbm_bytes),
                                   "peak_GBps": 6000.0, "frac": gbs(hbm_bytes) / 6000.0}}}


def test_roofline_is_against_measured_hbm_and_names_the_binding_side():
    peaks = {"hbm_gbs": 6000.0, "source": "measured"}
    # 10 MB over a 200 GB/s link (50 us) outweighs 60 MB of HBM (10 us)
    r = bench.roofline_entry("expert_ffn", _kernels(10e6, 60e6, 80.0), peaks, 200.0, traffic=123)
    assert r["bound"] == "hbm" and r["peak"] == 6000.0 and r["unit"] == "GB/s" and r["traffic"] == 123
    assert abs(r["frac"] - (60e6 / 80e-6 / 1e9) / 6000.0) < 1e-12
    assert r["binding"] == "link" and abs(r["link"]["frac"] - (10e6 / 80e-6 / 1e9) / 200.0) < 1e-12
    # no link bytes: HBM only
    r = bench.roofline_entry("expert_ffn", _kernels(0, 60e6, 20.0), peaks, 200.0)
    assert r["bound"] == "hbm" and "link" not in r and "binding" not in r


def test_kernel_table_shares_and_rates():
    prof = {"expert_ffn": {"ms": 3.0, "launches": 30}, "route_ctl": {"ms": 1.0, "launches": 30}}
    kb = {"expert_ffn": {"link": 30 * 1e6, "hbm": 30 * 5e6}}
    t = bench.kernel_table(prof, kb, 30, {"hbm_gbs": 5000.0}, 100.0)
    assert t["expert_ffn"]["share"] == 0.75 and t["route_ctl"]["share"] == 0.25
    assert t["expert_ffn"]["us_per_launch"] == 100.0
    assert t["expert_ffn"]["hbm"]["achieved_GBps"] == 50.0 and t["expert_ffn"]["hbm"]["frac"] == 0.01
    assert t["expert_ffn"]["link"]["achieved_GBps"] == 10.0 and t["expert_ffn"]["link"]["frac"] == 0.1


def test_traffic_is_scaled_by_algorithmic_bytes_and_dropped_when_a_source_changes(tmp_path, monkeypatch):
    src, src2 = tmp_path / "k.cu", tmp_path / "h.cuh"
    src.write_text("kernel v1")
    src2.write_text("helpers v1")
    import hashlib as hl
    h = hl.sha256()
    h.update(src.read_bytes())
    h.update(src2.read_bytes())
    sha = h.hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "scaled": {"sources": ["k.cu", "h.cuh"], "source_sha": sha, "dram_bytes": 800, "alg_bytes": 400},
        "per_launch": {"sources": ["k.cu", "h.cuh"], "source_sha": sha, "dram_bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("scaled", 1000) == 2000
    assert bench.traffic_from_profiles("scaled") is None        # nothing to scale to
    assert bench.traffic_from_profiles("per_launch") == 1234
    assert bench.traffic_from_profiles("absent", 3) is None
    src2.write_text("helpers v2")                                # a listed source changed since
    assert bench.traffic_from_profiles("scaled", 1000) is None


def test_committed_traffic_entries_name_existing_sources():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for k, v in d.items():
        if k.startswith("_"):
            continue
        for src in v["sources"]:
            assert os.path.exists(os.path.join(ROOT, src)), (k, src)
        if "alg_bytes" in v:
            assert v["dram_bytes"] > 0 and v["alg_bytes"] > 0
        else:
            assert v["dram_bytes_per_launch"] > 0


def test_cli_help_needs_no_gpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    for flag in ("--gpus", "--steps", "--warmup", "--impl", "--no-fp4", "--leg", "--ncu-quant", "--ncu-case",
                 "--windows"):
        assert flag in r.stdout


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0 and "--warmup must be >= 3" in (r.stderr + r.stdout)


def test_clock_sampler_summary_from_a_stand_in_nvidia_smi(tmp_path, monkeypatch):
    # a stand-in for nvidia-smi on PATH that checks it is asked for the GPU
    # by UUID: one idle sample before the span, two under load inside it (one
    # with the power cap active), then it idles until the sampler stops it
    import time
    now = time.time()
    stamp = lambda t: time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".000"  # noqa: E731
    exe = tmp_path / "bin" / "nvidia-smi"
    exe.parent.mkdir()
    exe.write_text("#!/bin/sh\n"
                   "[ \"$2\" = GPU-0123 ] || exit 3\n"
                   f"echo '{stamp(now - 30)}, 1000, 2070, 100.0, 0x0, Not Active, Active, Not Active, Not Active'\n"
                   f"echo '{stamp(now + 2)}, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                   f"echo '{stamp(now + 3)}, 2040, 2070, 1399.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
                   "exec sleep 30\n")
    exe.chmod(0o755)
    monkeypatch.setenv("PATH", f"{exe.parent}:{os.environ['PATH']}")
    monkeypatch.setenv("FT_CLOCKS_DIR", str(tmp_path / "clocks"))
    cs = bench.ClockSampler("GPU-0123", "0")
    time.sleep(0.5)
    got = cs.stop(now + 1, now + 4)
    assert got["sm_mhz"] == 2055.0 and got["sm_max_mhz"] == 2070.0 and got["samples"] == 2
    assert got["reasons"] == ["sw_power_cap"] and got["power_w_max"] == 1399.0
    assert (tmp_path / "clocks" / "ft_clocks_rank0.csv").exists()
