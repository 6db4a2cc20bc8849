"""bench.py's roofline.traffic gate: the DRAM bytes per parameter recorded in
the committed ncu summary are reported only while the update kernel's
sources, comments and whitespace aside, are those the capture was taken on.
CPU only."""
import os
import shutil

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture
def tree(tmp_path, monkeypatch):
    for rel in bench.KERNEL_SOURCES + (bench.TRAFFIC_SUMMARY,):
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _edit(path, fn):
    text = path.read_text()
    path.write_text(fn(text))


def test_committed_summary_matches_the_sources(tree):
    assert bench.update_traffic_per_param() == pytest.approx(10.757)


def test_comments_and_whitespace_keep_the_digest(tree):
    before = bench.kernel_source_digest()
    src = tree / bench.KERNEL_SOURCES[0]
    _edit(src, lambda t: "// a new leading comment\n/* and a block\n   comment */\n"
          + t.replace("\n", "\n\n", 3) + "\n   \n")
    assert bench.kernel_source_digest() == before
    assert bench.update_traffic_per_param() is not None


@pytest.mark.parametrize("which", range(3))
def test_a_code_edit_drops_the_traffic(tree, which):
    before = bench.kernel_source_digest()
    _edit(tree / bench.KERNEL_SOURCES[which], lambda t: t + "\nstatic int fp8opt_x;\n")
    assert bench.kernel_source_digest() != before
    assert bench.update_traffic_per_param() is None


def test_a_missing_summary_drops_the_traffic(tree):
    os.remove(tree / bench.TRAFFIC_SUMMARY)
    assert bench.update_traffic_per_param() is None
