"""The sharded data-parallel step on 2 CPU ranks over gloo, with the oracle as
its engine: the tensor partition, the all-to-all of gradient codes and scales,
the FP8 mean of the ranks' shards, found_inf combined over ranks, the global
clip norm and the owners' weight broadcasts give, on every rank, the result of
the same pipeline run whole in one process, bit for bit."""
import os
import socket
import sys

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import host_src

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def workload():
    return synth.fp8_reduce(ranks=2, n_layer=1, d=64, ffn=256, vocab=500, ctx=32)


def local_grads(wl, step, rank, inf_at=None):
    grads = [wl.rank_grad(i, step, rank) for i in range(len(wl.shapes))]
    if inf_at is not None and inf_at[:2] == (step, rank):
        grads[inf_at[2]][inf_at[3]] = float("inf")
    return grads


def worker(rank, world, port, cfg, out_dir):
    sys.path[:0] = [ROOT, HERE]
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    from bit_optimizer_gb300.sharded import ShardedFp8AdamW, TorchDistComm
    from oracle_engine import OracleEngine
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = workload()
    opt = ShardedFp8AdamW(wl.weights(), TorchDistComm(), lr=wl.lr,
                          betas=(wl.beta1, wl.beta2), eps=wl.eps,
                          weight_decay=wl.wd, level=cfg["level"],
                          l2=cfg["l2"], scaled_v=cfg["scaled_v"],
                          max_grad_norm=cfg["max_norm"], engine=OracleEngine(),
                          device="cpu")
    found, norms = [], []
    for t in range(1, cfg["steps"] + 1):
        found.append(opt.step(local_grads(wl, t, rank, cfg["inf_at"])))
        norms.append(opt.last_grad_norm if cfg["max_norm"] is not None else 0.0)
    out = {"found": np.array(found), "norms": np.array(norms),
           "ranges": np.array(opt.ranges)}
    for i, w in enumerate(opt.weights):
        out[f"w{i}"] = w.view(torch.int16).numpy().copy()
    if cfg["level"] == "O3":
        out["w8_scale"] = opt.w8_scale.numpy().copy()
        for i, c in enumerate(opt.w8):
            out[f"w8_{i}"] = c.numpy().copy()
    lo, hi = opt.own
    for j in range(hi - lo):
        out[f"m{lo + j}"] = opt.m[j].numpy().copy()
        out[f"v{lo + j}"] = opt.v[j].view(torch.int16).numpy().copy()
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), **out)
    dist.destroy_process_group()


def reference(cfg, world=2):
    """The same pipeline whole, in one process, with the oracle."""
    wl = workload()
    n = len(wl.shapes)
    states = [oracle.StepState(np.zeros(wl.numels[i], np.uint8), 1.0,
                               np.zeros(wl.numels[i], np.uint8), 1.0,
                               np.zeros(wl.numels[i], np.uint16),
                               wl.weight(i).view(torch.int16).numpy().view(np.uint16),
                               o3=cfg["level"] == "O3", scaled_v=cfg["scaled_v"])
              for i in range(n)]
    found, norms, step = [], [], 0
    for t in range(1, cfg["steps"] + 1):
        casts = []
        for r in range(world):
            cs = []
            for g in local_grads(wl, t, r, cfg["inf_at"]):
                a, dt = host_src(g)
                c, _, s = oracle.cast_scaled(a, dt, oracle.E4M3)
                cs.append((c, s))
            casts.append(cs)
        for i in range(n):
            codes, _, sc = oracle.reduce_scaled(
                np.stack([casts[r][i][0] for r in range(world)]),
                np.array([casts[r][i][1] for r in range(world)], np.float32),
                oracle.E4M3, oracle.E4M3, 1.0 / world)
            states[i].g, states[i].g_scale = codes, float(sc)
        hp = (wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, step + 1, 1.0)
        if cfg["max_norm"] is not None:
            f, nv = oracle.adam_step_clipped(states, *hp, cfg["max_norm"], l2=cfg["l2"])
        else:
            f, nv = oracle.adamw_step(states, *hp, l2=cfg["l2"]), 0.0
        found.append(f)
        norms.append(nv)
        if f == 0:
            step += 1
    return states, found, norms


CASES = {
    "o2": dict(level="O2", l2=False, scaled_v=False, max_norm=None, steps=3,
               inf_at=None),
    "o3_clip": dict(level="O3", l2=False, scaled_v=False, max_norm=0.05, steps=3,
                    inf_at=None),
    "o2_l2_scaled_v_clip": dict(level="O2", l2=True, scaled_v=True, max_norm=0.02,
                                steps=2, inf_at=None),
    "inf_on_one_rank": dict(level="O3", l2=False, scaled_v=False, max_norm=None,
                            steps=3, inf_at=(2, 1, 3, 7)),
}


@pytest.mark.parametrize("case,world", [(c, 2) for c in sorted(CASES)] +
                         [("o3_clip", 3), ("o3_clip", 4)])
def test_cpu_ranks_match_the_whole_pipeline(case, world, tmp_path):
    import torch.multiprocessing as mp
    cfg = CASES[case]
    mp.spawn(worker, args=(world, free_port(), cfg, str(tmp_path)), nprocs=world,
             join=True)
    res = [dict(np.load(tmp_path / f"rank{r}.npz")) for r in range(world)]
    states, found, norms = reference(cfg, world)
    wl = workload()
    for r in range(world):
        assert list(res[r]["found"]) == found
        assert np.array_equal(res[r]["norms"], np.array(norms, np.float64))
        for i, st in enumerate(states):
            if cfg["level"] == "O2":
                assert np.array_equal(res[r][f"w{i}"].view(np.uint16), st.w), (r, i)
            else:
                assert np.array_equal(res[r][f"w8_{i}"], st.w8), (r, i)
                assert res[r]["w8_scale"][i] == st.w8_scale[0]
            if f"m{i}" in res[r]:
                assert np.array_equal(res[r][f"m{i}"], st.m), (r, i)
                assert np.array_equal(res[r][f"v{i}"].view(np.uint16), st.v), (r, i)
                if cfg["level"] == "O3":
                    assert np.array_equal(res[r][f"w{i}"].view(np.uint16), st.w)
    # each tensor owned by exactly one rank, and every rank owns some
    owned = [k for r in range(world) for k in res[r] if k.startswith("m")]
    assert sorted(owned) == sorted(f"m{i}" for i in range(len(wl.shapes)))
    assert all(any(k.startswith("m") for k in res[r]) for r in range(world))
    if cfg["inf_at"] is not None:
        assert found[cfg["inf_at"][0] - 1] == 1 and sum(found) == 1


def test_partition_is_balanced_and_contiguous():
    from bit_optimizer_gb300.sharded import partition
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(0, 40))
        numels = [int(x) for x in rng.integers(0, 10000, n)]
        world = int(rng.integers(1, 9))
        parts = partition(numels, world)
        assert len(parts) == world
        assert parts[0][0] == 0 and parts[-1][1] == n
        for (a, b), (c, d) in zip(parts, parts[1:]):
            assert b == c and a <= b
        w = [max(x, 1) for x in numels]
        best = max(sum(w[a:b]) for a, b in parts) if n else 0
        # no contiguous split does better: brute force on small lists
        if n <= 8:
            import itertools
            opt = None
            for cuts in itertools.combinations_with_replacement(range(n + 1), world - 1):
                bounds = [0, *cuts, n]
                if any(x > y for x, y in zip(bounds, bounds[1:])):
                    continue
                m = max(sum(w[x:y]) for x, y in zip(bounds, bounds[1:]))
                opt = m if opt is None else min(opt, m)
            assert best == opt


class FailingEngine:
    """Wraps an engine; its step's begin raises on one step (a rank that
    dies between the first pass and the exchange)."""

    def __init__(self, inner, fail_step):
        self.inner, self.fail_step, self.calls = inner, fail_step, 0

    def __getattr__(self, name):
        return getattr(self.inner, name)

    def make_step(self, *args):
        step = self.inner.make_step(*args)
        outer = self

        class Step:
            def __getattr__(self, name):
                return getattr(step, name)

            def begin(self, *a, **k):
                outer.calls += 1
                if outer.calls == outer.fail_step:
                    raise RuntimeError("injected rank failure")
                return step.begin(*a, **k)
        return Step()


def failing_worker(rank, world, port, out_dir):
    sys.path[:0] = [ROOT, HERE]
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import datetime
    import torch.distributed as dist
    from bit_optimizer_gb300.sharded import ShardedFp8AdamW, TorchDistComm
    from oracle_engine import OracleEngine
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=20))
    wl = workload()
    engine = FailingEngine(OracleEngine(), 2) if rank == 1 else OracleEngine()
    opt = ShardedFp8AdamW(wl.weights(), TorchDistComm(), engine=engine,
                          device="cpu")
    outcome = "ok"
    try:
        for t in (1, 2, 3):
            opt.step(local_grads(wl, t, rank))
    except Exception as e:   # noqa: BLE001  (recorded for the parent)
        outcome = f"{type(e).__name__}: {e}"[:200]
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{outcome}\n{opt.step_count}\n")


def test_a_failing_rank_stops_the_others_at_the_exchange(tmp_path):
    """Rank 1 raises in its second step before the exchange; rank 0 gets an
    error from that step's collective (it does not hang) and neither rank
    counts the step."""
    import time
    import torch.multiprocessing as mp
    ctx = mp.spawn(failing_worker, args=(2, free_port(), str(tmp_path)),
                   nprocs=2, join=False)
    t0 = time.time()
    while not ctx.join(timeout=5):
        assert time.time() - t0 < 120, "ranks still running after 120 s"
    out = [open(tmp_path / f"rank{r}.txt").read().split("\n") for r in range(2)]
    assert out[1][0].startswith("RuntimeError: injected rank failure")
    assert out[0][0] != "ok"          # the collective reported the lost peer
    assert out[0][1] == "1" and out[1][1] == "1"
