"""Host-side logic of the library, compiled with g++ and run on the CPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "rope_tcgen05_mxfp8_gb300", "csrc")


@pytest.fixture(scope="module")
def bands_bin(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    out = str(tmp_path_factory.mktemp("host") / "bands_check")
    cmd = [gxx, "-std=c++17", "-O1", "-I", CSRC, "-I", "/usr/local/cuda/include",
           os.path.join(ROOT, "tests", "host", "bands_check.cpp"), "-o", out]
    subprocess.run(cmd, check=True)
    return out


@pytest.mark.parametrize("T,H,I,tile_n,k_end,band,chunks", [
    (32760, 5120, 15360, 240, 10240, 45, 1),   # Wan 480p: one V band, one Q/K band
    (32760, 5120, 15360, 240, 10240, 10, 1),
    (32760, 5120, 15360, 240, 10240, 23, 4),   # 28 MB bands, Q/K bands over four row-panel ranges
    (32760, 5120, 15360, 240, 10240, 23, 20),  # more chunks than the segment cap allows
    (75600, 5120, 15360, 256, 10240, 1, 1),    # one N tile per band: capped at 16 bands
    (256, 512, 1536, 240, 1024, 3, 1),
    (256, 512, 1536, 240, 1024, 3, 3),         # more chunks than row panels
    (1, 256, 640, 128, 512, 2, 2),
    (4096, 5120, 5120, 240, 5120, 45, 1),      # separate mode: every tile is Q
    (4096, 5120, 5120, 240, 5120, 45, 5),
    (129, 384, 576, 192, 448, 1000, 1),
])
def test_banded_tile_order_covers_every_tile_once(bands_bin, T, H, I, tile_n, k_end, band, chunks):
    r = subprocess.run([bands_bin, str(T), str(H), str(I), str(tile_n), str(k_end), str(band), str(chunks)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")


@pytest.fixture(scope="module")
def schedule_bin(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    out = str(tmp_path_factory.mktemp("host") / "schedule_check")
    cmd = [gxx, "-std=c++17", "-O1", "-I", CSRC, "-I", "/usr/local/cuda/include",
           os.path.join(ROOT, "tests", "host", "schedule_check.cpp"), "-o", out]
    subprocess.run(cmd, check=True)
    return out


@pytest.mark.parametrize("num_tiles,pairs,seed", [
    (8192, 76, 1),    # Wan 480p: 107 full waves, the last six and the partial one claimed
    (8192, 76, 7),
    (1024, 76, 3),    # 4096 tokens: 13 waves
    (88, 76, 5),      # the K|V call: one wave and a bit, all claimed
    (7, 7, 2),        # fewer tiles than pairs (the grid shrinks to the tiles)
    (456, 76, 4),     # exactly six waves: nothing static
    (532, 76, 9),     # exactly seven waves: one static
])
def test_pair_schedule_covers_every_tile_once(schedule_bin, num_tiles, pairs, seed):
    r = subprocess.run([schedule_bin, str(num_tiles), str(pairs), str(seed)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")


def test_clock_samples_are_kept_only_inside_the_timed_region():
    """bench.py reports clocks from the nvidia-smi samples taken while the timed steps
    ran; idle samples before or after them must not enter the median."""
    import datetime
    import sys

    sys.path.insert(0, ROOT)
    import bench

    def row(t, mhz, cap="Not Active"):
        stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return [stamp, "0", str(mhz), "2070", "900.0", "0x0", "Not Active", "Not Active", "Not Active", cap]

    t0 = 1_800_000_000.0
    rows = [row(t0 - 0.2, 345), row(t0 + 0.01, 2070), row(t0 + 0.03, 2055, "Active"), row(t0 + 0.05, 2070),
            row(t0 + 0.4, 345)]
    out = bench.ClockSampler.summarise(rows, t0, t0 + 0.1)
    assert out["samples"] == 3 and out["window"] == "timed region"
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    # nothing inside the window: every sample, and the line says so
    out = bench.ClockSampler.summarise(rows, t0 + 0.06, t0 + 0.07)
    assert out["samples"] == 5 and out["window"].startswith("no sample")


def test_bench_traffic_only_from_a_profile_of_the_current_kernel(tmp_path, monkeypatch):
    """bench.py reports the GEMM's DRAM traffic from the committed ncu summary only while
    that summary's source hash matches the kernel sources; otherwise traffic is null."""
    import shutil
    import sys

    sys.path.insert(0, ROOT)
    import bench

    name = "qkv_gemm_mxf8_pair_wan480p.md"
    src = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(src):
        pytest.skip("no committed GEMM profile")
    fake_root = tmp_path / "repo"
    (fake_root / "profiles").mkdir(parents=True)
    shutil.copy(src, fake_root / "profiles" / name)
    rec = {}
    for line in open(src):
        if ":" in line and not line.startswith(("|", " ", "#", "-")):
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    for rel in rec["sources"].split():
        (fake_root / rel).parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), fake_root / rel)
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    import hashlib

    h = hashlib.sha256()
    for rel in rec["sources"].split():
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    current = h.hexdigest() == rec["source_sha256"]  # False while a kernel change awaits a new capture
    expect = int(rec["dram_bytes_per_launch"]) if current else None
    assert bench._k1_traffic("wan480p", 240, True) == expect
    assert bench._k1_traffic("wan480p", 192, True) is None       # another tile width
    assert bench._k1_traffic("short", 240, True) is None         # another workload
    first = rec["sources"].split()[0]
    with open(fake_root / first, "a") as f:                      # the kernel changed since the capture
        f.write("\n// changed\n")
    assert bench._k1_traffic("wan480p", 240, True) is None
