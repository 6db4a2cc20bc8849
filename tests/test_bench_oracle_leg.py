"""The benchmark's oracle leg (host logic only): the bounded sample, the split
of its tensors over processes, and a short parallel run on the tiny list."""
import dataclasses
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _big():
    return dataclasses.replace(synth.WORKLOADS["o2_6p7b_tail"](), inf_site=None)


def test_sample_respects_budget_and_share():
    wl = _big()
    for budget, parts in ((2.0, 1), (60.0, 8), (120.0, 16)):
        entries, total = bench.oracle_sample(wl, budget, parts)
        limit = int(budget * 5e6)
        assert total == sum(n for _, n in entries)
        assert total <= limit
        assert max(n for _, n in entries) <= limit // parts
        idx = [i for i, _ in entries]
        assert idx == sorted(set(idx))
        # whole tensors, or (split samples only) a leading slice of one share
        for i, n in entries:
            assert n == wl.numels[i] or (parts > 1 and n == limit // parts
                                         and n < wl.numels[i])
        if parts > 1:
            # the budget is filled to within one share
            assert total > limit - limit // parts


def test_split_covers_each_tensor_once_and_balances():
    wl = _big()
    entries, _ = bench.oracle_sample(wl, 60.0, 8)
    parts = bench._split_by_size(entries, 8)
    flat = sorted(e for p in parts for e in p)
    assert flat == entries
    loads = [sum(n for _, n in p) for p in parts]
    # greedy largest-first: no list exceeds the lightest by more than its
    # largest entry
    biggest = max(n for _, n in entries)
    assert max(loads) - min(loads) <= biggest


def test_split_drops_empty_lists():
    wl = dataclasses.replace(synth.tiny(), inf_site=None)
    entries = [(i, n) for i, n in enumerate(wl.numels)]
    parts = bench._split_by_size(entries, 8)
    assert len(parts) == len(wl.shapes)
    assert sorted(e for p in parts for e in p) == entries


def test_parallel_run_on_tiny_list():
    wl = dataclasses.replace(synth.tiny(), inf_site=None)
    entries = [(i, n) for i, n in enumerate(wl.numels)]
    times, used = bench.oracle_parallel_times(wl, entries, 2, 2)
    assert used == 2
    assert len(times) == 2 and all(t > 0 for t in times)
