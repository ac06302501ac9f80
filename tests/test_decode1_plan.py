"""The batch-1 decode kernel's work split, checked on the host (no GPU needed):
tests/decode1_plan_check.cu includes the kernel's source, builds every CTA's
plan and block layouts for several shapes and grids, and checks coverage (each
half-row tile, router unit and head task owned exactly once) and bounds (every
copy inside its source matrix, 16-byte aligned, inside its block and the ring)."""
import os
import shutil
import subprocess

import pytest

from int4_routed_expert_prerouter_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode1_plans_cover_every_tile_once(tmp_path):
    nvcc = build.nvcc()
    if shutil.which(nvcc) is None and not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "decode1_plan_check")
    # device code only as PTX (no ptxas): the check runs the host functions
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=compute_103a", "-std=c++17", "-O1",
                           "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(ROOT, "int4_routed_expert_prerouter_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "decode1_plan_check.cu"), "-o", exe])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-4000:] + out.stderr[-2000:]
    assert "ALL OK" in out.stdout
