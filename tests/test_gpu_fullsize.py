"""Parity at the workloads' full sizes, in the launch configuration the
bench times.  Every tensor is resident and stepped by the library; the
oracle follows a sample of whole tensors (all the small ones and the
position embedding, and for the cast every tensor), and properties that hold
at any size are checked on every tensor."""
import concurrent.futures as cf
import dataclasses
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import DeviceList, host_src, oracle_step, oracle_step_threads
from parity import (check_codes, check_f16, check_f32_exact, check_master,
                    to_np_u16, to_np_u8)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


def sample_of(wl, limit):
    """The position embedding (a multi-chunk tensor with a ragged last tile)
    and whole tensors, smallest first, up to `limit` parameters."""
    order = sorted(range(len(wl.shapes)), key=lambda i: wl.numels[i])
    out, total = [1], wl.numels[1]
    for i in order:
        if i == 1:
            continue
        if total + wl.numels[i] <= limit:
            out.append(i)
            total += wl.numels[i]
    return sorted(out)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_cast_gpt2_124m_every_tensor(bo, fmt):
    wl = synth.gpt2_cast()
    assert wl.n_params == 124_439_808
    dev = [wl.grad(i, 1, "cuda") for i in range(len(wl.shapes))]
    codes, amax, scale = bo.fp8_cast_scaled(dev, fmt)
    torch.cuda.synchronize()
    amax, scale = amax.cpu().numpy(), scale.cpu().numpy()
    f = oracle.FMT[fmt]
    for i, g in enumerate(dev):
        a, dt = host_src(g)
        rc, ra, rs = oracle.cast_scaled(a, dt, f)
        check_f32_exact(amax[i:i + 1], [ra], f"amax[{i}]")
        check_f32_exact(scale[i:i + 1], [rs], f"scale[{i}]")
        check_codes(to_np_u8(codes[i]), rc, f, name=f"codes[{i}]")


def lockstep_full(wl, steps, sample, first=1, fused=False, scaled_v=False,
                  pool=None, workers=1):
    """Every tensor stepped by the library; the sampled ones start each step
    from the oracle's state.  fused: one fp8_cast_adamw_step call per step
    (the bench's configuration), else fp8_cast_scaled then fp8_adamw_step.
    pool: a thread pool for the oracle's casts, steps and the comparisons
    (workers threads), for samples of whole large lists."""
    dl = DeviceList(wl, scaled_v=scaled_v)
    states = {i: dl.fresh_oracle(i) for i in sample}
    each = (lambda f, xs: list(pool.map(f, xs))) if pool else \
        (lambda f, xs: [f(x) for x in xs])
    for t in range(first, first + steps):
        dl.gen_grads(t)
        if fused:
            for i in sample:
                dl.put(i, states[i])
            f = dl.cast_step(t)
            each(lambda i: dl.check_cast([i], states), sample)
        else:
            dl.cast()
            torch.cuda.synchronize()
            each(lambda i: dl.check_cast([i], states), sample)
            for i in sample:
                dl.put(i, states[i])
            f = dl.step(t)
        listed = [states[i] for i in sample]
        f_ref = (oracle_step_threads(listed, wl, t, pool, workers) if pool
                 else oracle_step(listed, wl, t))
        assert f == f_ref == 0
        each(lambda i: dl.compare(i, states[i]), sample)
    return dl, states


def test_o2_350m_full_inf_skip_and_step(bo):
    """The 350M list, every tensor against the oracle: the warm-up steps, a
    step whose gradients hold one +inf (nothing may change), and the same
    step with the inf cleared."""
    wl = synth.o2_350m()
    clean = dataclasses.replace(wl, inf_site=None)
    sample = list(range(len(wl.shapes)))
    workers = max(1, min(32, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as pool:
        dl, states = lockstep_full(clean, wl.warmup_steps, sample, pool=pool,
                                   workers=workers)
        t = wl.warmup_steps + 1
        listed = [states[i] for i in sample]
        # the measured step's gradients hold one +inf: nothing may change
        dl.gen_grads(t, wl)
        dl.cast()
        torch.cuda.synchronize()
        list(pool.map(lambda i: dl.check_cast([i], states), sample))
        for i in sample:
            dl.put(i, states[i])
        sums = [(x.sum(dtype=torch.int64).item(), x.numel()) for x in dl.m]
        vsum = [x.view(torch.int16).sum(dtype=torch.int64).item() for x in dl.v]
        wsum = [x.view(torch.int16).sum(dtype=torch.int64).item() for x in dl.w]
        mscale = dl.m_scale.clone()
        # found_inf is the maximum over the oracle's groups (the inf is in
        # one); the groups without it would step, so they run on copies
        probe = [st.copy() for st in listed]
        assert oracle_step_threads(probe, wl, t, pool, workers) == 1
        del probe
        assert dl.step(t) == 1 and dl.found_dev.item() == 1
        assert sums == [(x.sum(dtype=torch.int64).item(), x.numel()) for x in dl.m]
        assert vsum == [x.view(torch.int16).sum(dtype=torch.int64).item() for x in dl.v]
        assert wsum == [x.view(torch.int16).sum(dtype=torch.int64).item() for x in dl.w]
        assert torch.equal(mscale, dl.m_scale)
        # the same step with the inf cleared
        dl.gen_grads(t, clean)
        dl.cast()
        torch.cuda.synchronize()
        list(pool.map(lambda i: dl.check_cast([i], states), sample))
        for i in sample:
            dl.put(i, states[i])
        listed = [states[i] for i in sample]
        assert oracle_step_threads(listed, wl, t, pool, workers) == 0
        assert dl.step(t) == 0
        list(pool.map(lambda i: dl.compare(i, states[i]), sample))
    dl.invariants()


def test_o3_1p3b_full_two_calls(bo):
    """The 1.3B O3 list through fp8_cast_scaled then fp8_adamw_step, with the
    oracle on a sample of whole tensors."""
    wl = synth.o3_1p3b()
    sample = sample_of(wl, 6_000_000)
    dl, _ = lockstep_full(wl, wl.warmup_steps + 1, sample, fused=False)
    dl.invariants()


def test_o3_1p3b_every_tensor(bo):
    """The 1.3B O3 list through the fused call (the bench's configuration),
    with the oracle stepping every tensor from the same inputs: every
    gradient code, m, v, master and weight-copy element and every scale of
    all 292 tensors, including wte, qkv, fc and fc2, whose hundreds to
    thousands of chunks merge their amax through atomics from many CTAs.
    Three steps (two warm-up steps, then the measured one), so the moments
    carry history."""
    wl = synth.o3_1p3b()
    workers = max(1, min(32, os.cpu_count() or 1))
    sample = list(range(len(wl.shapes)))
    with cf.ThreadPoolExecutor(workers) as pool:
        dl, _ = lockstep_full(wl, wl.warmup_steps + 1, sample, fused=True,
                              pool=pool, workers=workers)
    dl.invariants()


def test_o2_6p7b_tail_full_10_steps(bo):
    wl = synth.o2_6p7b_tail()
    assert len(wl.shapes) == 589
    sample = sample_of(wl, 12_000_000)       # every tail tensor, norms, biases, wpe
    assert len(wl.shapes) - 1 in sample and 1 in sample
    dl, _ = lockstep_full(wl, wl.steps, sample, fused=True)
    dl.invariants()
    zero = len(wl.shapes) - 1
    assert dl.m_scale[zero].item() == 1.0 and not bool(dl.m[zero].any().item())


def test_o2_6p7b_tail_every_tensor(bo):
    """The 6.7B long-tail list through the fused call (the bench's workload
    and configuration), with the oracle stepping all 589 tensors from the
    same inputs: every gradient code, m, v and weight element and every scale
    of 6.66 G parameters, over two steps so the moments carry history.  About
    40 GB of host memory for the oracle's state and 3 to 4 minutes on a
    16-core host."""
    wl = synth.o2_6p7b_tail()
    workers = max(1, min(32, os.cpu_count() or 1))
    sample = list(range(len(wl.shapes)))
    with cf.ThreadPoolExecutor(workers) as pool:
        dl, _ = lockstep_full(wl, 2, sample, fused=True, pool=pool,
                              workers=workers)
    dl.invariants()


def test_o2_6p7b_tail_full_scaled_v(bo):
    """The long-tail list with the scaled second moment, through the fused
    call, 3 steps."""
    wl = synth.o2_6p7b_tail()
    sample = sample_of(wl, 12_000_000)
    dl, _ = lockstep_full(wl, 3, sample, fused=True, scaled_v=True)
    dl.invariants()
    assert float(dl.v_bound.max().item()) > 0


def test_reduce_gpt2_124m_8_shards_every_tensor(bo):
    """The 124M list with 8 shards per tensor (1 GB of codes), every output
    compared with the oracle.  Each shard is a rank's gradient put into E4M3
    codes by torch's float8 type at scale 448 / max |g| (torch's amax)."""
    wl = synth.fp8_reduce()
    assert wl.n_params == 124_439_808 and wl.ranks == 8
    k = wl.ranks
    shards, scales = [], torch.empty((len(wl.shapes), k))
    for i in range(len(wl.shapes)):
        rows = torch.empty((k, wl.numels[i]), dtype=torch.uint8, device="cuda")
        for r in range(k):
            g = wl.rank_grad(i, 1, r, "cuda").float()
            s = torch.tensor(448.0, device="cuda") / g.abs().max()
            rows[r] = (g * s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
            scales[i, r] = s.item()
        shards.append(rows)
    codes, amax, scale = bo.fp8_reduce_scaled(shards, scales.cuda(), "e4m3",
                                              "e4m3", 1.0 / k)
    torch.cuda.synchronize()
    amax, scale = amax.cpu().numpy(), scale.cpu().numpy()
    for i in range(len(wl.shapes)):
        rc, ra, rs = oracle.reduce_scaled(to_np_u8(shards[i]).reshape(k, -1),
                                          scales[i].numpy(), oracle.E4M3,
                                          oracle.E4M3, 1.0 / k)
        check_f32_exact(amax[i:i + 1], [ra], f"amax[{i}]")
        check_f32_exact(scale[i:i + 1], [rs], f"scale[{i}]")
        check_codes(to_np_u8(codes[i]), rc, oracle.E4M3, name=f"codes[{i}]")


def test_grad_norm_and_clipped_step_o3_1p3b(bo):
    """The 1.3B list (1.3 G gradient codes): the library's norm over every
    tensor equals the oracle's bit for bit, and one clipped O3 step of the
    whole list matches the oracle's step at the oracle's coefficient on
    every tensor (the oracle steps groups of tensors in host threads; with
    the coefficient given, each tensor's step is its own).  Gradient codes
    are put into E4M3 by torch's float8 type at scale 448 / max |g| (torch's
    amax)."""
    wl = synth.o3_1p3b()
    n = len(wl.shapes)
    numels = wl.numels
    g = bo.arena_views(numels, torch.uint8, "cuda")
    g_scale = torch.empty(n, device="cuda")
    for i in range(n):
        x = wl.grad(i, 1, "cuda").float()
        s = torch.tensor(448.0, device="cuda") / x.abs().max()
        g[i].copy_((x * s).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8))
        g_scale[i] = s
    del x
    w = bo.arena_views(numels, torch.float16, "cuda")
    for i in range(n):
        w[i].copy_(wl.weight(i, "cuda"))
    m = bo.arena_views(numels, torch.uint8, "cuda", fill=0)
    v = bo.arena_views(numels, torch.float16, "cuda", fill=0)
    m_scale = torch.ones(n, device="cuda")
    w8 = bo.arena_views(numels, torch.uint8, "cuda", fill=0)
    w8_scale = torch.ones(n, device="cuda")
    w8_amax = torch.zeros(n, device="cuda")
    plan = bo.AdamWPlan(g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax)
    host_g = [to_np_u8(t) for t in g]
    scales = g_scale.cpu().numpy()
    found, norm = oracle.grad_norm_codes(host_g, scales, oracle.E4M3, 1.0)
    assert found == 0
    assert plan.grad_norm(1.0) == (0, norm)
    max_norm = norm / 3.0
    sample = list(range(n))
    states = []
    for i in sample:
        ne = numels[i]
        states.append(oracle.StepState(host_g[i], scales[i], np.zeros(ne, np.uint8),
                                       1.0, np.zeros(ne, np.uint16),
                                       to_np_u16(w[i]), o3=True))
    assert plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, 1, 1.0,
                max_grad_norm=max_norm) == 0
    assert plan.last_grad_norm == norm
    coef = oracle.clip_coef(norm, max_norm)
    assert coef < 1.0
    workers = max(1, min(32, os.cpu_count() or 1))
    groups = [[] for _ in range(workers)]
    load = [0] * workers
    for j in sorted(range(len(states)), key=lambda j: -states[j].numel):
        k = load.index(min(load))
        groups[k].append(states[j])
        load[k] += states[j].numel
    ms, w8s = m_scale.cpu().numpy(), w8_scale.cpu().numpy()

    def compare(j):
        i, st = sample[j], states[j]
        check_f32_exact(ms[i:i + 1], st.m_scale, f"m_scale[{i}]")
        check_f32_exact(w8s[i:i + 1], st.w8_scale, f"w8_scale[{i}]")
        check_codes(to_np_u8(m[i]), st.m, name=f"m[{i}]")
        check_f16(to_np_u16(v[i]), st.v, name=f"v[{i}]")
        check_master(to_np_u16(w[i]), st.w, name=f"master[{i}]")
        check_codes(to_np_u8(w8[i]), st.w8, name=f"w8[{i}]")

    with cf.ThreadPoolExecutor(workers) as pool:
        found = list(pool.map(
            lambda grp: oracle.adam_step_coef(grp, wl.lr, wl.beta1, wl.beta2,
                                              wl.eps, wl.wd, 1, 1.0, coef)
            if grp else 0, groups))
        assert max(found) == 0
        list(pool.map(compare, range(len(states))))


def test_cast_tensor_above_two_giga_elements(bo):
    """One BF16 tensor of 2^31 + 12345 elements (past 32-bit indexing):
    amax and scale bit-exact against the oracle over the whole tensor, and
    the codes of a strided sample plus the last 40,000 elements."""
    n = (1 << 31) + 12345
    g = torch.Generator(device="cuda")
    g.manual_seed(synth.tensor_seed(7, 0, "grad"))
    x = (torch.randn(n, generator=g, device="cuda") * 1e-3).to(torch.bfloat16)
    x[n - 7] = 0.25                       # the largest element, in the tail
    codes, amax, scale = bo.fp8_cast_scaled([x], "e4m3")
    torch.cuda.synchronize()
    host = x.view(torch.int16).cpu().numpy().view(np.uint16)
    rc, ra, rs = oracle.cast_scaled(host, oracle.BF16, oracle.E4M3)
    check_f32_exact(amax.cpu().numpy()[:1], [ra], "amax")
    check_f32_exact(scale.cpu().numpy()[:1], [rs], "scale")
    got = codes[0]
    idx = np.concatenate([np.arange(0, n, 9973), np.arange(n - 40000, n)])
    assert np.array_equal(got[torch.from_numpy(idx).cuda()].cpu().numpy(), rc[idx])
    assert int(got[n - 7].item()) == 0x7E


def test_o3_step_tensor_above_two_giga_elements(bo):
    """An O3 step over one tensor of 2^31 + 12345 elements (past 32-bit
    indexing; 65537 chunks).  The oracle steps a sample of its elements (a
    strided sample and the last 40,000, which straddle element 2^31) as a
    tensor of its own.  First step from m = v = 0: this step's m is
    (1 - beta1) * g, so with the one largest gradient code (448) planted in
    the sample the tensor's m amax, and so its m scale, are the sample's;
    with the one largest weight (1.0, far above the others' |w| < 0.2)
    planted in the sample, the master's amax and the weight copy's scale are
    the sample's too.  Every other element's result depends only on its own
    inputs, so the sampled elements must match the oracle's sample: scales
    and found_inf bit-exact, codes, v and weights within the tolerances."""
    n = (1 << 31) + 12345
    gen = torch.Generator(device="cuda")
    gen.manual_seed(synth.tensor_seed(8, 0, "grad"))
    g = torch.randint(0, 0x7E, (n,), generator=gen, device="cuda", dtype=torch.uint8)
    g |= torch.randint(0, 2, (n,), generator=gen, device="cuda", dtype=torch.uint8) << 7
    w = (torch.randn(n, generator=gen, device="cuda") * 0.02).clamp_(-0.19, 0.19)
    w = w.to(torch.float16)
    idx = np.concatenate([np.arange(0, n - 40000, 9973), np.arange(n - 40000, n)])
    top_g, top_w = int(idx[len(idx) // 3]), int(idx[-3])
    g[top_g] = 0xFE                         # -448: the largest |g|
    w[top_w] = 1.0                          # the largest |master|
    m = torch.zeros(n, dtype=torch.uint8, device="cuda")
    v = torch.zeros(n, dtype=torch.float16, device="cuda")
    w8 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    g_scale = torch.full((1,), 2.0 ** -4, device="cuda")
    m_scale = torch.ones(1, device="cuda")
    w8_scale = torch.ones(1, device="cuda")
    w8_amax = torch.zeros(1, device="cuda")
    sel = torch.from_numpy(idx).cuda()
    st = oracle.StepState(to_np_u8(g[sel]), 2.0 ** -4, np.zeros(idx.size, np.uint8),
                          1.0, np.zeros(idx.size, np.uint16), to_np_u16(w[sel]),
                          o3=True)
    plan = bo.AdamWPlan([g], g_scale, [m], m_scale, [v], [w], [w8], w8_scale,
                        w8_amax)
    found_dev = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    args = (1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 0.5)
    assert plan(*args, found_inf_dev=found_dev) == 0 and found_dev.item() == 0
    assert oracle.adamw_step([st], *args) == 0
    check_f32_exact(m_scale.cpu().numpy(), st.m_scale, "m_scale")
    check_f32_exact(w8_scale.cpu().numpy(), st.w8_scale, "w8_scale")
    check_f32_exact(w8_amax.cpu().numpy(), st.w8_amax, "w8_amax")
    assert st.w8_amax[0] == np.float32(np.float16(w[top_w].item()))
    check_codes(to_np_u8(m[sel]), st.m, name="m")
    check_f16(to_np_u16(v[sel]), st.v, name="v")
    check_master(to_np_u16(w[sel]), st.w, name="master")
    check_f16(to_np_u16(w[sel]), st.w, name="w")
    check_codes(to_np_u8(w8[sel]), st.w8, name="w8")
    assert int(m[top_g].item()) == 0xFE      # the largest |m| on the maximum
