"""The persistent engine's work split, checked on the host (no GPU needed):
tests/engine_plan_check.cu includes the engine's source, builds every CTA
pair's plan and copy items and the head flush's tables for several layer kinds
and grids, and checks coverage (each tile, unit, row tile and task owned exactly
once) and bounds (every copy inside its source matrix and its ring)."""
import os
import shutil
import subprocess

import pytest

from int4_routed_expert_prerouter_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_engine_plans_cover_every_tile_once(tmp_path):
    nvcc = build.nvcc()
    if shutil.which(nvcc) is None and not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "engine_plan_check")
    # device code only as PTX (no ptxas): the check runs the host functions
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=compute_103a", "-std=c++17", "-O1",
                           "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(ROOT, "int4_routed_expert_prerouter_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "engine_plan_check.cu"), "-o", exe])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-4000:] + out.stderr[-2000:]
    assert "ALL OK" in out.stdout
