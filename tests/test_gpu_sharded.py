"""The sharded data-parallel step through the CUDA library.  Ranks are
emulated as threads of one process on one GPU, each on its own CUDA stream;
their exchanges go through the host (every kernel of a rank runs to
completion before its data is exchanged, so no kernel waits on another
rank's).  Sharded over 1 to 4 ranks, with tensors cut into pieces across
ranks, the library's result equals the same pipeline run whole through the
library (cast per rank, FP8 mean of the ranks' codes, one step over every
tensor; on one rank the cast feeds the step) bit for bit, and that pipeline
is within the step's tolerances of the oracle's."""
import threading

import numpy as np
import pytest
import torch

import oracle
from parity import check_codes, check_f16, check_f32_exact, to_np_u16, to_np_u8
from test_sharded_gloo import CASES, local_grads, reference, workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


class ThreadComm:
    """Collectives between rank threads of one process, through the host."""

    def __init__(self, rank, world, shared):
        self.rank, self.world, self.sh = rank, world, shared

    def _swap(self, value):
        torch.cuda.current_stream().synchronize()
        self.sh["slots"][self.rank] = value
        self.sh["barrier"].wait()
        vals = list(self.sh["slots"])
        self.sh["barrier"].wait()
        return vals

    def all_to_all(self, out, inp, out_splits, in_splits):
        parts, o = [], 0
        for s in in_splits:
            parts.append(inp[o:o + s].clone())
            o += s
        vals = self._swap(parts)
        out.copy_(torch.cat([vals[src][self.rank] for src in range(self.world)]))

    def all_reduce_sum(self, t):
        vals = self._swap(t.clone())
        acc = vals[0].clone()
        for v in vals[1:]:
            acc += v
        t.copy_(acc)

    def all_reduce_max(self, t):
        vals = self._swap(t.clone())
        t.copy_(torch.stack(vals).amax(0))

    def all_gather(self, out, inp):
        vals = self._swap(inp.clone())
        out.copy_(torch.cat(vals))


def run_sharded(bo, cfg, world):
    from bit_optimizer_gb300.sharded import ShardedFp8AdamW
    wl = workload()
    shared = {"slots": [None] * world, "barrier": threading.Barrier(world)}
    results, errors = [None] * world, []

    def rank_main(rank):
        try:
            with torch.cuda.stream(torch.cuda.Stream()):
                opt = ShardedFp8AdamW(
                    [w.cuda() for w in wl.weights()], ThreadComm(rank, world, shared),
                    lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                    weight_decay=wl.wd, level=cfg["level"], l2=cfg["l2"],
                    scaled_v=cfg["scaled_v"], max_grad_norm=cfg["max_norm"])
                found, norms = [], []
                for t in range(1, cfg["steps"] + 1):
                    grads = [g.cuda() for g in local_grads(wl, t, rank, cfg["inf_at"])]
                    found.append(opt.step(grads))
                    norms.append(opt.last_grad_norm)
                torch.cuda.current_stream().synchronize()
                results[rank] = (opt, found, norms)
        except BaseException as e:   # surface a rank's failure in the test
            errors.append(e)
            shared["barrier"].abort()

    threads = [threading.Thread(target=rank_main, args=(r,)) for r in range(world)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if errors:
        raise errors[0]
    return results


def run_whole(bo, cfg, world):
    """The pipeline whole through the library: every rank's cast, the FP8
    mean of the ranks' codes, one step over every tensor."""
    wl = workload()
    n, numels = len(wl.shapes), wl.numels
    w = [x.cuda() for x in wl.weights()]
    g = [torch.empty(x, dtype=torch.uint8, device="cuda") for x in numels]
    g_amax, g_scale = torch.zeros(n, device="cuda"), torch.ones(n, device="cuda")
    m = [torch.zeros(x, dtype=torch.uint8, device="cuda") for x in numels]
    v = [torch.zeros(x, dtype=torch.float16, device="cuda") for x in numels]
    m_scale = torch.ones(n, device="cuda")
    o3 = cfg["level"] == "O3"
    w8 = [torch.zeros(x, dtype=torch.uint8, device="cuda") for x in numels] if o3 else None
    w8s = torch.ones(n, device="cuda") if o3 else None
    w8a = torch.zeros(n, device="cuda") if o3 else None
    vb = torch.zeros(n, device="cuda") if cfg["scaled_v"] else None
    plan = bo.AdamWPlan(g, g_scale, m, m_scale, v, w, w8, w8s, w8a, "e4m3", vb)
    found, norms, step = [], [], 0
    for t in range(1, cfg["steps"] + 1):
        shards = [torch.empty((world, x), dtype=torch.uint8, device="cuda") for x in numels]
        scales = torch.empty((n, world), device="cuda")
        for r in range(world):
            grads = [x.cuda() for x in local_grads(wl, t, r, cfg["inf_at"])]
            codes, _, sc = bo.fp8_cast_scaled(grads, "e4m3")
            for i in range(n):
                shards[i][r].copy_(codes[i])
            scales[:, r] = sc[:n]
        if world == 1:        # one rank: its cast feeds the step
            for i in range(n):
                g[i].copy_(shards[i][0])
            g_scale[:n].copy_(scales[:, 0])
        else:
            bo.fp8_reduce_scaled(shards, scales, "e4m3", "e4m3", 1.0 / world,
                                 codes=g, amax=g_amax, scale=g_scale)
        f = plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, step + 1, 1.0,
                 l2=cfg["l2"], max_grad_norm=cfg["max_norm"])
        found.append(f)
        norms.append(plan.last_grad_norm)
        if f == 0:
            step += 1
    return dict(w=w, m=m, v=v, w8=w8, w8s=w8s, found=found, norms=norms)


@pytest.mark.parametrize("case,world", [(c, w) for c in sorted(CASES) for w in (1, 2)]
                         + [("o3_clip", 3), ("o2_l2_scaled_v_clip", 3),
                            ("o3_clip", 4)])
def test_sharded_equals_whole_and_oracle(bo, case, world):
    cfg = CASES[case]
    whole = run_whole(bo, cfg, world)
    results = run_sharded(bo, cfg, world)
    for opt, found, norms in results:
        assert found == whole["found"]
        if cfg["max_norm"] is not None:
            assert norms == whole["norms"]
        for i in range(len(whole["w"])):
            if cfg["level"] == "O2":
                assert torch.equal(opt.weights[i], whole["w"][i]), i
            else:
                assert torch.equal(opt.w8[i], whole["w8"][i]), i
                assert opt.w8_scale[i].item() == whole["w8s"][i].item()
        for j, (t, a, b) in enumerate(opt.pieces):
            assert torch.equal(opt.m[j], whole["m"][t][a:b]), (t, a, b)
            assert torch.equal(opt.v[j], whole["v"][t][a:b]), (t, a, b)
            if cfg["level"] == "O3":         # the masters of the rank's pieces
                assert torch.equal(opt.weights[t][a:b], whole["w"][t][a:b])
    if world > 1:                      # some tensor is cut across ranks
        owners = {}
        for opt, _, _ in results:
            for t, _, _ in opt.pieces:
                owners[t] = owners.get(t, 0) + 1
        assert max(owners.values()) > 1
    # the whole pipeline against the oracle's
    states, found, norms = reference(cfg, world)
    assert whole["found"] == found
    if cfg["max_norm"] is not None:
        assert whole["norms"] == norms
    for i, st in enumerate(states):
        check_codes(to_np_u8(whole["m"][i]), st.m, name=f"m[{i}]")
        check_f16(to_np_u16(whole["v"][i]), st.v, name=f"v[{i}]")
        check_f16(to_np_u16(whole["w"][i]), st.w, name=f"w[{i}]")
        if cfg["level"] == "O3":
            check_codes(to_np_u8(whole["w8"][i]), st.w8, name=f"w8[{i}]")


def _state_bytes(opt):
    out = {"m_scale": opt.m_scale.clone()}
    for j, (t, a, b) in enumerate(opt.pieces):
        out[f"m{j}"] = opt.m[j].clone()
        out[f"v{j}"] = opt.v[j].clone()
        out[f"w{j}"] = opt.weights[t][a:b].clone()
    if opt.v_bound is not None:
        out["v_bound"] = opt.v_bound.clone()
    if opt.level == "O2":
        for i, w in enumerate(opt.weights):
            out[f"W{i}"] = w.clone()
    else:
        out["w8_scale"] = opt.w8_scale.clone()
        out["w8_amax"] = opt.w8_amax.clone()
        for i, c in enumerate(opt.w8):
            out[f"w8_{i}"] = c.clone()
    return out


@pytest.mark.parametrize("case,world", [("o2", 2), ("o3_clip", 3),
                                        ("o2_l2_scaled_v_clip", 2), ("o3_clip", 1)])
def test_sharded_checkpoint_resume_on_the_gpu(bo, case, world):
    """ShardedFp8AdamW.state_dict / load_state_dict through the library:
    two steps, a checkpoint (through torch.save), a third step; a fresh
    optimizer built from the model's weights and loaded from the checkpoint
    takes the same third step, byte for byte, on every rank."""
    import io
    from bit_optimizer_gb300.sharded import ShardedFp8AdamW
    cfg = CASES[case]
    wl = workload()
    shared = {"slots": [None] * world, "barrier": threading.Barrier(world)}
    results, errors = [None] * world, []

    def rank_main(rank):
        try:
            with torch.cuda.stream(torch.cuda.Stream()):
                kw = dict(lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                          weight_decay=wl.wd, level=cfg["level"], l2=cfg["l2"],
                          scaled_v=cfg["scaled_v"], max_grad_norm=cfg["max_norm"])
                comm = ThreadComm(rank, world, shared)
                opt = ShardedFp8AdamW([w.cuda() for w in wl.weights()], comm, **kw)
                for t in (1, 2):
                    opt.step([g.cuda() for g in local_grads(wl, t, rank)])
                buf = io.BytesIO()
                torch.save(opt.state_dict(), buf)
                model = [w.clone() for w in opt.weights]
                grads3 = [g.cuda() for g in local_grads(wl, 3, rank)]
                opt.step(grads3)
                first = _state_bytes(opt)
                again = ShardedFp8AdamW(
                    model if cfg["level"] == "O2" else [w.cuda() for w in wl.weights()],
                    comm, **kw)
                buf.seek(0)
                again.load_state_dict(torch.load(buf))
                again.step(grads3)
                torch.cuda.current_stream().synchronize()
                results[rank] = (first, _state_bytes(again), again.step_count)
        except BaseException as e:   # surface a rank's failure in the test
            errors.append(e)
            shared["barrier"].abort()

    threads = [threading.Thread(target=rank_main, args=(r,)) for r in range(world)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if errors:
        raise errors[0]
    for first, second, steps in results:
        assert steps == 3
        assert sorted(first) == sorted(second)
        for k in first:
            assert torch.equal(first[k], second[k]), k
