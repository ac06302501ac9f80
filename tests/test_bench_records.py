"""Host-side checks of bench.py's use of committed measurements: the kernel's
DRAM traffic from an ncu capture is reported only while the kernel's code is the
code that was captured (comment edits do not count as changes)."""
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    for f in bench.KERNEL_SOURCES + ("profiles/" + bench.TRAFFIC_RECORD,):
        dst = tmp_path / f
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(ROOT, f), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_recorded_traffic_matches_the_committed_kernel():
    # the committed record was taken on the committed kernel code
    assert bench.profiled_traffic() is not None
    assert bench.profiled_traffic() >= 484_978_688   # at least the algorithmic bytes


def test_comment_edits_keep_the_record(fake_root):
    before = bench.kernel_source_hash()
    p = fake_root / bench.KERNEL_SOURCES[0]
    p.write_text("// a new comment line\n" + p.read_text().replace("//", "//  edited:", 3))
    assert bench.kernel_source_hash() == before
    assert bench.profiled_traffic() is not None


def test_code_edits_drop_the_record(fake_root):
    p = fake_root / bench.KERNEL_SOURCES[0]
    p.write_text(p.read_text() + "\nnamespace edge0 { constexpr int kProbeOnly = 1; }\n")
    assert bench.profiled_traffic() is None
