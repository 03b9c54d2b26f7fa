"""Host-side helpers of bench.py (CPU): the traffic record is tied to the
kernel's code, not to its comments."""

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "fp4_moe_expert_gb300", "csrc", "fme_routed_fp8.cu")


def _write(path, text):
    with open(path, "w") as f:
        f.write(text)
    return path


def test_code_hash_ignores_comment_lines_only(tmp_path):
    base = "// header\nint f() {\n  return 1;  // one\n}\n"
    h = bench.kernel_code_sha256(_write(tmp_path / "a.cu", base))
    assert bench.kernel_code_sha256(_write(tmp_path / "b.cu", "// other header\n\n" + base[10:])) == h
    assert bench.kernel_code_sha256(_write(tmp_path / "c.cu", base.replace("return 1", "return 2"))) != h
    assert bench.kernel_code_sha256(_write(tmp_path / "d.cu", base.replace("// one", "// two"))) != h


def test_committed_traffic_record_matches_the_kernel():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    assert d["kernel_code_sha256"] == bench.kernel_code_sha256(SRC)
    assert bench.load_traffic() == d["fp8_moe_kernel_dsv3_bytes_per_launch"]
    assert 1.0 <= d["fp8_moe_kernel_dsv3_bytes_per_launch"] / d["algorithmic_bytes_per_launch"] < 1.05


def test_parallel_oracle_leg_runs_every_process_over_one_window():
    out = bench.run_oracle_parallel(0.2, 2, steps=2)
    assert len(out) == 2
    for step in out:
        assert step["workers"] == 2 and step["routes"] >= 2 and step["seconds"] > 0
        assert abs(step["gbs"] - step["routes"] * bench.EXPERT_BYTES / step["seconds"] / 1e9) < 1e-9
