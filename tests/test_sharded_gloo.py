"""The sharded data-parallel step on CPU ranks over gloo, with the oracle as
its engine: the element-space layout (tensors cut into pieces across ranks),
the all-to-all of gradient codes, the all-gather of scales, the FP8 mean of the
ranks' shards with each tensor's amax combined over its pieces, found_inf
combined over ranks, the global clip norm from exact sums combined over
ranks, the first moment's and the master's maxima combined over pieces, and
the all-gather of the new weights give, on every rank, the result of the same
pipeline run whole in one process, bit for bit."""
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
    out = {"found": np.array(found), "norms": np.array(norms)}
    for i, w in enumerate(opt.weights):
        out[f"w{i}"] = w.view(torch.int16).numpy().copy()
    if cfg["level"] == "O3":
        out["w8_scale"] = opt.w8_scale.numpy().copy()
        for i, c in enumerate(opt.w8):
            out[f"w8_{i}"] = c.numpy().copy()
    out["pieces"] = np.array(opt.pieces, dtype=np.int64).reshape(-1, 3)
    for j in range(len(opt.pieces)):
        out[f"m_{j}"] = opt.m[j].numpy().copy()
        out[f"v_{j}"] = opt.v[j].view(torch.int16).numpy().copy()
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
            if world == 1:        # one rank: its cast feeds the step
                codes, sc = casts[0][i]
            else:
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
                         [("o3_clip", 1), ("o2", 1), ("o3_clip", 3),
                          ("o3_clip", 4), ("o2_l2_scaled_v_clip", 4)])
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
        for j, (t, a, b) in enumerate(res[r]["pieces"]):
            st = states[t]
            assert np.array_equal(res[r][f"m_{j}"], st.m[a:b]), (r, t)
            assert np.array_equal(res[r][f"v_{j}"].view(np.uint16), st.v[a:b]), (r, t)
            if cfg["level"] == "O3":       # the masters of the rank's pieces
                assert np.array_equal(res[r][f"w{t}"].view(np.uint16)[a:b], st.w[a:b])
    # every element owned by exactly one rank; some tensor cut across ranks
    owner = {}
    for r in range(world):
        for t, a, b in res[r]["pieces"]:
            owner.setdefault(int(t), []).append((int(a), int(b), r))
    assert sorted(owner) == list(range(len(wl.shapes)))
    for t, parts in owner.items():
        parts.sort()
        assert parts[0][0] == 0 and parts[-1][1] == wl.numels[t]
        assert all(x[1] == y[0] for x, y in zip(parts, parts[1:]))
    if world > 1:
        assert any(len({r for *_, r in p}) > 1 for p in owner.values())
    if cfg["inf_at"] is not None:
        assert found[cfg["inf_at"][0] - 1] == 1 and sum(found) == 1


def _dump(opt):
    """Every state byte of a sharded optimizer, as numpy arrays."""
    out = {"m_scale": opt.m_scale.numpy().copy(),
           "pieces": np.array(opt.pieces, dtype=np.int64).reshape(-1, 3)}
    for i, w in enumerate(opt.weights):
        out[f"w{i}"] = w.view(torch.int16).numpy().copy()
    for j in range(len(opt.pieces)):
        out[f"m_{j}"] = opt.m[j].numpy().copy()
        out[f"v_{j}"] = opt.v[j].view(torch.int16).numpy().copy()
    if opt.v_bound is not None:
        out["v_bound"] = opt.v_bound.numpy().copy()
    if opt.level == "O3":
        out["w8_scale"] = opt.w8_scale.numpy().copy()
        out["w8_amax"] = opt.w8_amax.numpy().copy()
        for i, c in enumerate(opt.w8):
            out[f"w8_{i}"] = c.numpy().copy()
    return out


def resume_worker(rank, world, port, cfg, out_dir):
    """Two steps, a checkpoint (through torch.save), a third step; then a
    fresh optimizer built from the weights a model checkpoint would hold,
    the checkpoint loaded, and the same third step."""
    sys.path[:0] = [ROOT, HERE]
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    from bit_optimizer_gb300.sharded import ShardedFp8AdamW, TorchDistComm
    from oracle_engine import OracleEngine
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = workload()
    kw = dict(lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
              weight_decay=wl.wd, level=cfg["level"], l2=cfg["l2"],
              scaled_v=cfg["scaled_v"], max_grad_norm=cfg["max_norm"],
              engine=OracleEngine(), device="cpu")
    opt = ShardedFp8AdamW(wl.weights(), TorchDistComm(), **kw)
    for t in (1, 2):
        opt.step(local_grads(wl, t, rank))
    path = os.path.join(out_dir, f"ckpt{rank}.pt")
    torch.save(opt.state_dict(), path)
    model = [w.clone() for w in opt.weights]     # O2: the model's weights
    opt.step(local_grads(wl, 3, rank))
    first = _dump(opt)
    again = ShardedFp8AdamW(model if cfg["level"] == "O2" else wl.weights(),
                            TorchDistComm(), **kw)
    again.load_state_dict(torch.load(path))
    assert again.step_count == 2
    again.step(local_grads(wl, 3, rank))
    second = _dump(again)
    np.savez(os.path.join(out_dir, f"first{rank}.npz"), **first)
    np.savez(os.path.join(out_dir, f"second{rank}.npz"), **second)
    # a checkpoint of another rank, or of another layout, is refused
    other = torch.load(os.path.join(out_dir, f"ckpt{rank}.pt"))
    other["rank"] = (rank + 1) % max(world, 2)
    try:
        again.load_state_dict(other)
        refused = 0
    except ValueError:
        refused = 1
    np.save(os.path.join(out_dir, f"refused{rank}.npy"), np.array([refused]))
    dist.destroy_process_group()


@pytest.mark.parametrize("case,world", [("o2", 2), ("o3_clip", 2),
                                        ("o2_l2_scaled_v_clip", 3), ("o3_clip", 1)])
def test_checkpoint_resume_is_bit_identical(case, world, tmp_path):
    """ShardedFp8AdamW.state_dict / load_state_dict: a run resumed from a
    checkpoint takes the same step, byte for byte, on every rank."""
    import torch.multiprocessing as mp
    cfg = CASES[case]
    mp.spawn(resume_worker, args=(world, free_port(), cfg, str(tmp_path)),
             nprocs=world, join=True)
    for r in range(world):
        a = dict(np.load(tmp_path / f"first{r}.npz"))
        b = dict(np.load(tmp_path / f"second{r}.npz"))
        assert sorted(a) == sorted(b)
        for k in a:
            if cfg["level"] == "O3" and k.startswith("w") and k[1:].isdigit():
                continue          # O3 keeps only its pieces' masters (below)
            assert np.array_equal(a[k], b[k]), (r, k)
        if cfg["level"] == "O3":
            for t, lo, hi in a["pieces"]:
                assert np.array_equal(a[f"w{t}"][lo:hi], b[f"w{t}"][lo:hi]), (r, t)
        assert int(np.load(tmp_path / f"refused{r}.npy")[0]) == 1


def test_layout_covers_every_element_once_and_balances():
    from bit_optimizer_gb300.sharded import layout
    rng = np.random.default_rng(0)
    for _ in range(300):
        n = int(rng.integers(0, 40))
        numels = [int(x) for x in rng.integers(0, 10000, n)]
        numels = [0 if rng.random() < 0.1 else x for x in numels]
        world = int(rng.integers(1, 9))
        off, seg, pieces = layout(numels, world)
        assert len(pieces) == world and seg % 256 == 0
        seen = {t: [] for t in range(n)}
        for r, ps in enumerate(pieces):
            for t, a, b in ps:
                assert 0 <= a <= b <= numels[t] and a % 256 == 0
                # inside the rank's range of the element space
                assert r * seg <= off[t] + a and (b == a or off[t] + b <= (r + 1) * seg)
                seen[t].append((a, b))
            assert sum(b - a for _, a, b in ps) <= seg
        for t in range(n):
            parts = sorted(seen[t])
            assert parts and parts[0][0] == 0 and parts[-1][1] == numels[t]
            assert all(x[1] == y[0] for x, y in zip(parts, parts[1:]))
            assert numels[t] > 0 or parts == [(0, 0)]
        # offsets: in order, 256-element aligned, no overlap
        for t in range(n - 1):
            assert off[t] % 256 == 0 and off[t] + numels[t] <= off[t + 1]


def test_layout_balance_on_the_350m_list_at_8_ranks():
    """Equal segments: the busiest of 8 ranks holds at most 1.02x its share
    of the 350M list's elements (whole tensors put wte's 51.5 M elements on
    one rank: 1.158x)."""
    from bit_optimizer_gb300.sharded import layout
    wl = synth.o2_350m()
    _, _, pieces = layout(wl.numels, 8)
    loads = [sum(b - a for _, a, b in p) for p in pieces]
    assert max(loads) <= 1.02 * sum(wl.numels) / 8


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
