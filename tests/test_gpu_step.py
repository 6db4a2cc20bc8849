"""GPU parity of fp8_adamw_step against the oracle, through the C ABI, on
the five workloads at reduced sizes (several chunks and ragged tails each),
plus the found_inf skip, E5M2 gradients, unaligned buffers and empty lists."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import (GpuState, fresh_states, oracle_cast, oracle_step,
                     set_grads)
from parity import check_codes, check_f16, check_f32_exact, to_np_u16, to_np_u8

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


def cast_both(bo, grads, fmt=E4M3):
    """Oracle cast of the gradients, with the GPU cast of the same values
    checked against it; returns the oracle's codes and scales."""
    codes, amax, scale = oracle_cast(grads, fmt)
    gc, ga, gs = bo.fp8_cast_scaled([g.cuda() for g in grads], fmt)
    check_f32_exact(ga.cpu().numpy()[:len(grads)], amax, "grad amax")
    check_f32_exact(gs.cpu().numpy()[:len(grads)], scale, "grad scale")
    for i, (c, r) in enumerate(zip(gc, codes)):
        check_codes(to_np_u8(c), r, fmt, name=f"grad codes[{i}]")
    return codes, scale


def warm_up(wl, states, steps, fmt=E4M3):
    clean = dataclasses.replace(wl, inf_site=None)
    for t in range(1, steps + 1):
        codes, _, scale = oracle_cast(clean.grads(t), fmt)
        set_grads(states, codes, scale)
        assert oracle_step(states, wl, t) == 0


def lockstep(bo, wl, states, t0, t1, fmt=E4M3, misalign=(), l2=False):
    """Steps t0..t1: each step the GPU starts from the oracle's state."""
    gpu = None
    for t in range(t0, t1 + 1):
        codes, scale = cast_both(bo, wl.grads(t), fmt)
        set_grads(states, codes, scale)
        if gpu is None:
            gpu = GpuState([s.copy() for s in states], misalign=misalign)
        else:
            gpu.load_state(states)
        f_ref = oracle_step(states, wl, t, l2=l2)
        assert gpu.step(wl, t, l2=l2) == f_ref == 0
        rates = gpu.compare(states)
    return gpu, rates


def test_tiny_o2_lockstep_10_steps(bo):
    wl = synth.tiny()
    states = fresh_states(wl.weights(), o3=False)
    _, rates = lockstep(bo, wl, states, 1, wl.steps)
    assert rates["m"] >= 0.999 and rates["w"] >= 0.999


def test_tiny_o2_free_running_public_api(bo):
    """Fp8AdamW (cast + step) run for 10 steps on its own against the oracle
    run on its own: the two never exchange state."""
    wl = synth.tiny()
    weights = wl.weights()
    params = [w.cuda() for w in weights]
    opt = bo.Fp8AdamW(params, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                      weight_decay=wl.wd, level="O2")
    states = fresh_states(weights, o3=False)
    for t in range(1, wl.steps + 1):
        grads = wl.grads(t)
        assert opt.step([g.cuda() for g in grads]) == 0
        codes, _, scale = oracle_cast(grads, E4M3)
        set_grads(states, codes, scale)
        assert oracle_step(states, wl, t) == 0
    assert opt.step_count == wl.steps
    check_f32_exact(opt.m_scale.cpu().numpy()[:3], [s.m_scale[0] for s in states])
    for i, s in enumerate(states):
        check_codes(to_np_u8(opt.m[i]), s.m, name=f"m[{i}]")
        check_f16(to_np_u16(opt.v[i]), s.v, name=f"v[{i}]")
        check_f16(to_np_u16(params[i].view(-1)), s.w, name=f"w[{i}]")


def reduced_350m():
    return synth.o2_350m(n_layer=2, d=128, ffn=512, vocab=1000, ctx=64)


def test_o2_350m_reduced_inf_skip_then_step(bo):
    wl = reduced_350m()
    states = fresh_states(wl.weights(), o3=False)
    warm_up(wl, states, wl.warmup_steps)
    t = wl.warmup_steps + 1
    # the measured step's gradients carry one +inf: found_inf, nothing written
    codes, scale = cast_both(bo, wl.grads(t))
    set_grads(states, codes, scale)
    gpu = GpuState([s.copy() for s in states])
    before = [s.copy() for s in states]
    assert oracle_step(states, wl, t) == 1
    assert gpu.step(wl, t) == 1
    for i, s in enumerate(before):
        assert np.array_equal(to_np_u8(gpu.m[i]), s.m)
        assert np.array_equal(to_np_u16(gpu.v[i]), s.v)
        assert np.array_equal(to_np_u16(gpu.w[i]), s.w)
    check_f32_exact(gpu.m_scale.cpu().numpy(), [s.m_scale[0] for s in before])
    # the same step with the inf cleared
    clean = dataclasses.replace(wl, inf_site=None)
    codes, scale = cast_both(bo, clean.grads(t))
    set_grads(states, codes, scale)
    gpu.load_state(states)
    assert oracle_step(states, wl, t) == 0
    assert gpu.step(wl, t) == 0
    gpu.compare(states)


def test_o3_1p3b_reduced(bo):
    wl = synth.o3_1p3b(n_layer=2, d=128, ffn=512, vocab=1000, ctx=64)
    states = fresh_states(wl.weights(), o3=True)
    warm_up(wl, states, wl.warmup_steps)
    gpu, rates = lockstep(bo, wl, states, wl.warmup_steps + 1, wl.warmup_steps + 2)
    assert rates["w8"] >= 0.999


def test_o2_6p7b_tail_reduced_10_steps(bo):
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=1000, ctx=64)
    assert len(wl.shapes) == 2 + 12 + 2 + 200 + 1
    states = fresh_states(wl.weights(), o3=False)
    gpu, _ = lockstep(bo, wl, states, 1, wl.steps)
    zero = len(states) - 1
    assert gpu.m_scale[zero].item() == 1.0 and not gpu.m[zero].any().item()


def test_e5m2_gradients(bo):
    wl = dataclasses.replace(synth.tiny(), grad_fmt="e5m2")
    states = fresh_states(wl.weights(), o3=False, g_fmt=E5M2)
    lockstep(bo, wl, states, 1, 3, fmt=E5M2)


def test_unaligned_buffers(bo):
    wl = synth.o3_1p3b(n_layer=1, d=64, ffn=256, vocab=300, ctx=32)
    states = fresh_states(wl.weights(), o3=True)
    lockstep(bo, wl, states, 1, 2, misalign={0, 3, 5})


@pytest.mark.parametrize("case", ["nan_code", "overflow_after_unscale", "e5m2_inf"])
def test_found_inf_leaves_state_unchanged(bo, case):
    wl = synth.tiny()
    fmt = E5M2 if case == "e5m2_inf" else E4M3
    states = fresh_states(wl.weights(), o3=True, g_fmt=fmt)
    codes, _, scale = oracle_cast(wl.grads(1), fmt)
    set_grads(states, codes, scale)
    oracle_step(states, wl, 1)
    codes, _, scale = oracle_cast(wl.grads(2), fmt)
    set_grads(states, codes, scale)
    ils = 1.0
    if case == "nan_code":
        states[2].g[1234] = 0xFF
    elif case == "e5m2_inf":
        states[0].g[5] = 0x7C
    else:
        states[1].g_scale = float(np.float32(1e-30))
        ils = 1e12
    gpu = GpuState([s.copy() for s in states])
    before = [s.copy() for s in states]
    assert oracle_step(states, wl, 2, ils=ils) == 1
    assert gpu.step(wl, 2, ils=ils) == 1
    for i, s in enumerate(before):
        assert np.array_equal(to_np_u8(gpu.m[i]), s.m)
        assert np.array_equal(to_np_u16(gpu.v[i]), s.v)
        assert np.array_equal(to_np_u16(gpu.w[i]), s.w)
        assert np.array_equal(to_np_u8(gpu.w8[i]), s.w8)
    for name in ("m_scale", "w8_scale", "w8_amax"):
        check_f32_exact(getattr(gpu, name).cpu().numpy(),
                        [getattr(s, name)[0] for s in before], name)


def test_empty_single_and_odd_tensors(bo):
    wl = synth.tiny()
    sizes = [0, 1, 3, 0, 17, 4097]
    g = torch.Generator().manual_seed(9)
    weights = [(torch.randn(n, generator=g) * 0.02).half() for n in sizes]
    states = fresh_states(weights, o3=True)
    for t in (1, 2):
        grads = [torch.randn(n, generator=g) * 1e-3 for n in sizes]
        codes, scale = cast_both(bo, grads)
        set_grads(states, codes, scale)
        if t == 1:
            gpu = GpuState([s.copy() for s in states])
        else:
            gpu.load_state(states)
        assert oracle_step(states, wl, t) == 0
        assert gpu.step(wl, t) == 0
        gpu.compare(states)
    assert gpu.m_scale[0].item() == 1.0 and gpu.w8_scale[0].item() == 1.0


def test_empty_list_and_async_flag(bo):
    flag = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    plan = bo.AdamWPlan([], torch.ones(1, device="cuda"), [],
                        torch.ones(1, device="cuda"), [], [])
    assert plan(1e-3, 0.9, 0.999, 1e-8, 0.0, 1, found_inf_dev=flag) == 0
    assert flag.item() == 0
    # sync=False: no host wait, the flag still lands on the device
    wl = synth.tiny()
    states = fresh_states(wl.weights(), o3=False)
    codes, _, scale = oracle_cast(wl.grads(1), E4M3)
    set_grads(states, codes, scale)
    gpu = GpuState([s.copy() for s in states])
    gpu.found_dev.fill_(9)
    assert gpu.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, 1,
                    found_inf_dev=gpu.found_dev, sync=False) is None
    torch.cuda.synchronize()
    assert gpu.found_dev.item() == 0
    oracle_step(states, wl, 1)
    gpu.compare(states)


def test_checkpoint_resume_is_bit_identical(bo):
    wl = synth.tiny()
    weights = [w.cuda() for w in wl.weights()]
    mk = lambda ps: bo.Fp8AdamW(ps, lr=wl.lr, betas=(wl.beta1, wl.beta2),
                                eps=wl.eps, weight_decay=wl.wd, level="O3")
    a = mk(weights)
    for t in (1, 2, 3):
        a.step([g.cuda() for g in wl.grads(t)])
    sd = a.state_dict()
    w_saved = [w.clone() for w in weights]
    b_weights = [w.clone() for w in w_saved]
    b = mk(b_weights)
    b.load_state_dict(sd)
    g4 = [g.cuda() for g in wl.grads(4)]
    a.step(g4)
    b.step(g4)
    assert b.step_count == a.step_count == 4
    for x, y in zip(weights, b_weights):
        assert torch.equal(x, y)
    for name in ("m", "v", "w8"):
        for x, y in zip(getattr(a, name), getattr(b, name)):
            assert torch.equal(x, y)
    assert torch.equal(a.m_scale, b.m_scale) and torch.equal(a.w8_scale, b.w8_scale)


@pytest.mark.parametrize("fused", [True, False])
def test_timing_records_each_kernel(bo, fused):
    wl = synth.tiny()
    params = [w.cuda() for w in wl.weights()]
    opt = bo.Fp8AdamW(params, level="O3", fused=fused)
    bo.timing_enable(True)
    for t in (1, 2):
        opt.step([g.cuda() for g in wl.grads(t)])
    bo.timing_enable(False)
    ran = ({"cast_amax", "cast_step_amax", "step_update", "step_w8"} if fused else
           {"cast_amax", "cast_encode", "step_amax", "step_update", "step_w8"})
    for k in bo.KERNELS:
        n, ms = bo.timing_read(k)
        if k in ran:
            assert n == 2 and ms > 0.0, k
        else:
            assert n == 0, k


def test_workspace_reuse_across_list_lengths(bo):
    """A short step list, then a longer cast and step on the same stream: the
    longer calls' per-tensor slots must not see the shorter call's scratch."""
    small = synth.tiny()
    s_states = fresh_states(small.weights(), o3=False)
    codes, _, scale = oracle_cast(small.grads(1), E4M3)
    set_grads(s_states, codes, scale)
    GpuState([s.copy() for s in s_states]).step(small, 1)
    wl = synth.o2_6p7b_tail(n_layer=1, d=64, ffn=256, vocab=300, ctx=32, n_tail=20)
    states = fresh_states(wl.weights(), o3=False)
    lockstep(bo, wl, states, 1, 2)


# ----------------------------------------------------------- fused call

def lockstep_fused(bo, wl, states, t0, t1, fmt=E4M3, misalign=(), clean=None):
    """Steps t0..t1 through fp8_cast_adamw_step: each step the GPU starts
    from the oracle's state and casts the same gradients itself."""
    gpu = None
    found = []
    for t in range(t0, t1 + 1):
        grads = (clean or wl).grads(t)
        codes, amax, scale = oracle_cast(grads, fmt)
        set_grads(states, codes, scale)
        if gpu is None:
            gpu = GpuState([s.copy() for s in states], misalign=misalign)
        else:
            gpu.load_state(states)
        before = [s.copy() for s in states]
        src = [g.cuda() for g in grads]
        g_amax = torch.empty(max(len(src), 1), device="cuda")
        fused = bo.CastStepPlan(bo.CastPlan(src, gpu.g, g_amax, gpu.g_scale, fmt),
                                gpu.plan)
        f_ref = oracle_step(states, wl, t)
        f = fused(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t, wl.inv_loss_scale,
                  found_inf_dev=gpu.found_dev)
        assert f == f_ref == int(gpu.found_dev.item())
        n = len(grads)
        check_f32_exact(g_amax.cpu().numpy()[:n], amax, "grad amax")
        check_f32_exact(gpu.g_scale.cpu().numpy()[:n], scale, "grad scale")
        for i, (c, r) in enumerate(zip(gpu.g, codes)):
            check_codes(to_np_u8(c), r, fmt, name=f"grad codes[{i}]")
        if f == 0:
            gpu.compare(states)
        else:
            for i, s in enumerate(before):
                assert np.array_equal(to_np_u8(gpu.m[i]), s.m)
                assert np.array_equal(to_np_u16(gpu.v[i]), s.v)
                assert np.array_equal(to_np_u16(gpu.w[i]), s.w)
        found.append(f)
    return gpu, found


def test_fused_tiny_10_steps(bo):
    wl = synth.tiny()
    states = fresh_states(wl.weights(), o3=False)
    _, found = lockstep_fused(bo, wl, states, 1, wl.steps)
    assert found == [0] * wl.steps


def test_fused_350m_reduced_inf_skip_then_step(bo):
    wl = reduced_350m()
    states = fresh_states(wl.weights(), o3=False)
    warm_up(wl, states, wl.warmup_steps)
    t = wl.warmup_steps + 1
    _, found = lockstep_fused(bo, wl, states, t, t)          # +inf: skipped
    assert found == [1]
    clean = dataclasses.replace(wl, inf_site=None)
    _, found = lockstep_fused(bo, wl, states, t, t, clean=clean)
    assert found == [0]


def test_fused_o3_and_long_tail_reduced(bo):
    wl = synth.o3_1p3b(n_layer=2, d=128, ffn=512, vocab=1000, ctx=64)
    states = fresh_states(wl.weights(), o3=True)
    warm_up(wl, states, wl.warmup_steps)
    lockstep_fused(bo, wl, states, wl.warmup_steps + 1, wl.warmup_steps + 2)
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=1000, ctx=64)
    states = fresh_states(wl.weights(), o3=False)
    lockstep_fused(bo, wl, states, 1, 3)


def test_fused_e5m2_unaligned_and_odd(bo):
    wl = dataclasses.replace(synth.tiny(), grad_fmt="e5m2")
    states = fresh_states(wl.weights(), o3=False, g_fmt=E5M2)
    lockstep_fused(bo, wl, states, 1, 3, fmt=E5M2, misalign={0, 2})
    sizes = [0, 1, 3, 17, 4097]
    g = torch.Generator().manual_seed(21)
    weights = [(torch.randn(n, generator=g) * 0.02).half() for n in sizes]
    odd = dataclasses.replace(synth.tiny(), names=[f"t{i}" for i in range(5)],
                              shapes=[(n,) for n in sizes])
    states = fresh_states(weights, o3=True)
    lockstep_fused(bo, odd, states, 1, 2)


def test_fused_equals_the_two_calls(bo):
    """The fused entry and fp8_cast_scaled + fp8_adamw_step, from the same
    state and gradients, give byte-identical results."""
    wl = synth.o2_6p7b_tail(n_layer=1, d=256, ffn=1024, vocab=2000, ctx=64, n_tail=50)
    weights = [w.cuda() for w in wl.weights()]
    grads = [g.cuda() for g in wl.grads(1)]
    outs = []
    for fused in (True, False):
        params = [w.clone() for w in weights]
        opt = bo.Fp8AdamW(params, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                          weight_decay=wl.wd, level="O3", fused=fused)
        for t in (1, 2):
            assert opt.step([g * t for g in grads]) == 0
        outs.append((params, opt))
    (pa, a), (pb, b) = outs
    for x, y in zip(pa, pb):
        assert torch.equal(x, y)
    for name in ("g_codes", "m", "v", "w8"):
        for x, y in zip(getattr(a, name), getattr(b, name)):
            assert torch.equal(x, y), name
    for name in ("g_amax", "g_scale", "m_scale", "w8_scale", "w8_amax"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


# ------------------------------------- scaled second moment, Adam with L2

@pytest.mark.parametrize("l2", [False, True])
def test_scaled_v_long_tail_reduced(bo, l2):
    """The long-tail list at reduced size has gradients down to sigma ~ 1e-5,
    where a plain FP16 second moment underflows."""
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=1000, ctx=64, n_tail=60)
    states = fresh_states(wl.weights(), o3=False, scaled_v=True)
    gpu, _ = lockstep(bo, wl, states, 1, 4, l2=l2)
    assert (gpu.v_bound.cpu().numpy()[:len(states) - 1] > 0).all()


@pytest.mark.parametrize("l2", [False, True])
def test_plain_v_adam_l2_o3_reduced(bo, l2):
    wl = synth.o3_1p3b(n_layer=1, d=128, ffn=512, vocab=500, ctx=64)
    states = fresh_states(wl.weights(), o3=True)
    lockstep(bo, wl, states, 1, 3, l2=l2, misalign={2})


def test_scaled_v_o3_unaligned_and_fused(bo):
    wl = synth.o3_1p3b(n_layer=1, d=128, ffn=512, vocab=500, ctx=64)
    states = fresh_states(wl.weights(), o3=True, scaled_v=True)
    lockstep(bo, wl, states, 1, 2, misalign={0, 4})
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=1000, ctx=64, n_tail=40)
    states = fresh_states(wl.weights(), o3=False, scaled_v=True)
    lockstep_fused(bo, wl, states, 1, 3)


def test_found_inf_keeps_v_bound(bo):
    wl = synth.tiny()
    states = fresh_states(wl.weights(), o3=False, scaled_v=True)
    codes, _, scale = oracle_cast(wl.grads(1), E4M3)
    set_grads(states, codes, scale)
    oracle_step(states, wl, 1)
    codes, _, scale = oracle_cast(wl.grads(2), E4M3)
    set_grads(states, codes, scale)
    states[1].g[7] = 0x7F
    gpu = GpuState([s.copy() for s in states])
    before = gpu.v_bound.clone()
    assert oracle_step(states, wl, 2) == 1
    assert gpu.step(wl, 2) == 1
    assert torch.equal(gpu.v_bound, before)


def test_optimizer_options_checkpoint(bo):
    """Fp8AdamW with scaled_v and with l2: state_dict round trip, and the
    two configurations differ from plain AdamW where they should."""
    wl = synth.tiny()
    weights = [w.cuda() for w in wl.weights()]
    outs = {}
    for name, kw in (("plain", {}), ("scaled", {"scaled_v": True}),
                     ("l2", {"l2": True})):
        params = [w.clone() for w in weights]
        opt = bo.Fp8AdamW(params, lr=wl.lr, weight_decay=0.1, **kw)
        for t in (1, 2):
            opt.step([g.cuda() * 1e-3 for g in wl.grads(t)])
        sd = opt.state_dict()
        b_params = [p.clone() for p in params]
        b = bo.Fp8AdamW(b_params, lr=wl.lr, weight_decay=0.1, **kw)
        b.load_state_dict(sd)
        g3 = [g.cuda() * 1e-3 for g in wl.grads(3)]
        opt.step(g3)
        b.step(g3)
        for x, y in zip(params, b_params):
            assert torch.equal(x, y)
        outs[name] = params
    assert not torch.equal(outs["plain"][0], outs["scaled"][0])
    assert not torch.equal(outs["plain"][0], outs["l2"][0])
