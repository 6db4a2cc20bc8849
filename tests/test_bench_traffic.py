"""bench.py's roofline.traffic gate: the DRAM bytes per parameter recorded
from an ncu capture of step_update (profiles/step_update_traffic.json,
written by ``bench.py --record-traffic``) are reported only while the update
kernel's sources, comments and whitespace aside, are those the capture was
taken on.  CPU only; the ncu CSV here is a synthetic one in ncu's raw-page
layout (a header row of metric names, a row of units, a row per launch)."""
import json
import os
import shutil

import pytest

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture
def tree(tmp_path, monkeypatch):
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, rel), dst)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def ncu_csv(path, launches):
    """launches: (kernel name, read, read unit, write, write unit, ns)."""
    head = ['"ID"', '"Kernel Name"', '"dram__bytes_read.sum"',
            '"dram__bytes_write.sum"', '"gpu__time_duration.sum"']
    lines = [",".join(head)]
    # ncu prints one units row; the tests give every launch the same units
    units = launches[0]
    lines.append(",".join(['""', '""', f'"{units[2]}"', f'"{units[4]}"', '"nsecond"']))
    for i, (name, rd, _, wr, _, ns) in enumerate(launches):
        lines.append(",".join([f'"{i}"', f'"{name}"', f'"{rd}"', f'"{wr}"', f'"{ns}"']))
    path.write_text("\n".join(lines) + "\n")


def tiny_record(tree):
    wl = synth.tiny()
    csv = tree / "launches.csv"
    name = "void fp8opt::<unnamed>::step_update_kernel<0, 0, 0>(...)"
    ncu_csv(csv, [("cast_amax_kernel", "1.0", "Mbyte", "0", "Mbyte", "1000"),
                  (name, "0.1", "Mbyte", "0.12", "Mbyte", "5000"),
                  (name, "0.14", "Mbyte", "0.08", "Mbyte", "7000")])
    return wl, bench.record_traffic(str(csv), wl, "ncu ... python bench.py ...")


def test_record_from_a_capture(tree):
    wl, rec = tiny_record(tree)
    assert rec["launches"] == 2
    assert rec["dram_bytes_read"] == pytest.approx(0.12e6)
    assert rec["dram_bytes_write"] == pytest.approx(0.10e6)
    assert rec["duration_us"] == pytest.approx(6.0)
    assert rec["traffic_bytes_per_param"] == pytest.approx(0.22e6 / wl.n_params, abs=1e-4)
    on_disk = json.loads((tree / bench.TRAFFIC_RECORD).read_text())
    assert on_disk == rec
    assert bench.update_traffic_per_param() == rec["traffic_bytes_per_param"]


def test_units_are_converted(tree):
    csv = tree / "u.csv"
    ncu_csv(csv, [("step_update_kernel", "2", "Gbyte", "1500", "Kbyte", "3")])
    (x,) = bench.ncu_launches(str(csv))
    assert x == pytest.approx({"dram_read": 2e9, "dram_write": 1.5e6, "seconds": 3e-9})


def test_comments_and_whitespace_keep_the_digest(tree):
    tiny_record(tree)
    before = bench.kernel_source_digest()
    src = tree / bench.KERNEL_SOURCES[0]
    text = src.read_text()
    src.write_text("// a new leading comment\n/* and a block\n   comment */\n"
                   + text.replace("\n", "\n\n", 3) + "\n   \n")
    assert bench.kernel_source_digest() == before
    assert bench.update_traffic_per_param() is not None


@pytest.mark.parametrize("which", range(3))
def test_a_code_edit_drops_the_traffic(tree, which):
    tiny_record(tree)
    before = bench.kernel_source_digest()
    src = tree / bench.KERNEL_SOURCES[which]
    src.write_text(src.read_text() + "\nstatic int fp8opt_x;\n")
    assert bench.kernel_source_digest() != before
    assert bench.update_traffic_per_param() is None


def test_a_missing_or_broken_record_drops_the_traffic(tree):
    assert bench.update_traffic_per_param() is None
    (tree / bench.TRAFFIC_RECORD).write_text("{not json")
    assert bench.update_traffic_per_param() is None


def test_no_launch_of_the_kernel_is_an_error(tree):
    csv = tree / "n.csv"
    ncu_csv(csv, [("cast_amax_kernel", "1", "byte", "1", "byte", "1")])
    with pytest.raises(SystemExit):
        bench.record_traffic(str(csv), synth.tiny(), "")
