"""CPU check of the routed FP8 kernel's work decomposition: compiles
tests/plan_walk_check.cpp against the kernel's own schedule header
(fme_plan.cuh, host and device code) and runs it. Every CTA's chunk walk must
cover each (phase, unit, tile, K block) slot of the launched phases exactly
once, for one launch and for the two-kernel chain's phase ranges, with slices by
slot count and by cost; and the fill warps' division-free walk over a chunk's
(row, K block) items must match p % r, p / r."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_slot_walked_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "plan_walk_check"
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "fp4_moe_expert_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "plan_walk_check.cpp"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr
