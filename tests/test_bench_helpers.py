"""bench.py's accounting (CPU only): algorithmic bytes, launch counts, the
reported-traffic gate, and the oracle reference arm's JSON line."""
import json
import subprocess
import sys
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_lower_sector_bytes_and_algorithmic_bytes():
    # 16x16 fp32: rows 0-7 need one 32-byte sector, rows 8-15 two
    assert bench.lower_sector_bytes(16, 4) == 8 * 32 + 8 * 64
    fwd, adj = bench.algorithmic_bytes(16, 4)
    assert fwd == 768 + 1024 + 4 and adj == 4 * 768 + 4
    assert bench.algorithmic_bytes(64, 4) == (25604, 36868)
    assert bench.lower_sector_bytes(512, 8) == 1056768


def test_launch_counts():
    assert bench.launches_per_step(16, 0) == 2
    # FMA-pipe tiles, nt = 4: forward 1 + 4 + 6, adjoint 5 * 4 - 3
    assert bench.launches_per_step(512, 128, 1, False) == 11 + 17
    assert bench.launches_per_step(100, 128) == 1 + 1 + 0 + 3
    # float64, 128-wide tiles, one 8192 x 8192 matrix: 1081 kernels per step
    # without the lookaheads' 62 + 62 extra launches (ncu launch lists of one
    # step counted 1081 before the lookahead, 1143 with the forward's and
    # 1205 with both), less the 63 inverses the cluster factor now makes, plus
    # the adjoint row update's side-stream part (61) and its reductions (60)
    # (1263 in the launch list), less the 63 inverse slicings that share the
    # panel's slicing launch
    assert bench.launches_per_step(8192, 128, 1, True) == 1081 + 62 + 62 - 63 + 61 + 60 - 63
    # many matrices: no literal diagonal adjoint, no split reduction
    nt = 4
    fwd = 1 + nt + 3 * 5 + 2 * 1          # lookahead: 2 extra launches (k = 0, 1)
    adj = 6 + 3 * 4 + nt * 1 + 3 * 2 + 2 + 1   # lookahead: J = 3, 2; row rest of J = 2
    assert bench.launches_per_step(512, 128, 256, True) == fwd + adj


def test_default_tile_mirrors_the_library_rule():
    assert bench.default_tile(8192, 1) == 128
    assert bench.default_tile(512, 1) == 32
    assert bench.default_tile(512, 1, 152, True) == 128
    assert bench.default_tile(128, 1, 152, True) == 32
    assert bench.default_tile(512, 19, 152, True) == 128
    assert bench.default_tile(512, 20, 152, True) == 64
    assert bench.default_tile(512, 256) == 64


def test_traffic_is_reported_only_for_the_captured_kernel_source():
    rec = bench.MEASURED_TRAFFIC["batched_16"]
    got = bench.measured_traffic("batched_16", rec["kernel"])
    assert got is None or got == rec["bytes"]
    assert bench.measured_traffic("batched_16", "fwd" if rec["kernel"] == "adj" else "adj") is None
    assert bench.measured_traffic("banded_8192", "adj") is None
    # the tensor-core update's record holds while ozaki.cu's code is the captured one
    rec = bench.MEASURED_TRAFFIC["banded_8192"]
    assert bench.measured_traffic("banded_8192", "tc_update") in (None, rec["bytes"])


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "matrices/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_code_hash_ignores_comments_but_not_code():
    import bench
    src = "int f(int x) {  // doubles x\n    /* block\n comment */ return 2 * x;\n}\n"
    same = "// a new header line\nint f(int x) {\n\n    return 2 * x;   // still doubles\n}\n"
    other = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench.code_sha256(src) == bench.code_sha256(same)
    assert bench.code_sha256(src) != bench.code_sha256(other)


def test_traffic_record_follows_the_kernel_source_hash():
    import bench
    for wl, rec in bench.MEASURED_TRAFFIC.items():
        with open(os.path.join(ROOT, rec["source"])) as f:
            live = bench.code_sha256(f.read()) == rec["code_sha256"]
        got = bench.measured_traffic(wl, rec["kernel"])
        assert (got == rec["bytes"]) if live else (got is None)
