"""GPU parity of the gradient norm (fp8_grad_norm) and of the clipped step
(fp8_adam_step_clipped) against the oracle, through the C ABI: the norm is
bit-exact as a double, and the clipped step's state meets the step's
tolerances."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import GpuState, fresh_states, oracle_cast, set_grads
from parity import check_f32_exact, to_np_u16, to_np_u8

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


def states_for(wl, step, fmt=E4M3, o3=False, scaled_v=False):
    states = fresh_states(wl.weights(), o3=o3, g_fmt=fmt, scaled_v=scaled_v)
    codes, _, scale = oracle_cast(wl.grads(step), fmt)
    set_grads(states, codes, scale)
    return states


def gpu_norm(gpu, ils):
    nd = torch.full((1,), -1.0, device="cuda")
    found, norm = gpu.plan.grad_norm(ils, norm_dev=nd)
    assert nd.item() == np.float32(norm) or (math.isinf(norm) and math.isinf(nd.item()))
    return found, norm


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("ils", [1.0, 2.0 ** -16, 0.37])
def test_grad_norm_bit_exact(bo, fmt, ils):
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64,
                            n_tail=40)
    wl = dataclasses.replace(wl, grad_mult=1.0 / ils)
    states = states_for(wl, 1, fmt)
    gpu = GpuState([s.copy() for s in states], misalign={1, 7})
    found, norm = gpu_norm(gpu, ils)
    rf, rn = oracle.grad_norm(states, ils)
    assert found == rf == 0
    assert norm == rn, (norm, rn)


def test_grad_norm_mixed_formats(bo):
    """A list whose tensors alternate E4M3 and E5M2 codes (runs of one
    tensor's chunks, whole chunks and ragged ends, in both formats within
    one CTA's range): the norm bit-exact against the oracle."""
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64,
                            n_tail=40)
    grads = wl.grads(1)
    fmts = [E4M3 if i % 2 == 0 else E5M2 for i in range(len(grads))]
    states = fresh_states(wl.weights(), o3=False)
    for i, (s, g) in enumerate(zip(states, grads)):
        codes, _, scale = oracle_cast([g], fmts[i])
        s.g_fmt = fmts[i]
        set_grads([s], codes, scale)
    gpu = GpuState([s.copy() for s in states])
    for ils in (1.0, 0.37):
        found, norm = gpu_norm(gpu, ils)
        assert (found, norm) == oracle.grad_norm(states, ils)


def test_grad_norm_exactness_case(bo):
    """One E5M2 maximum and 4096 minimum subnormals: only an exact sum keeps
    the small squares (the oracle's exactness pin, on the GPU)."""
    g = np.concatenate([[0x7B], np.full(4096, 0x01), np.full(40000, 0x81)]).astype(np.uint8)
    n = g.size
    st = oracle.StepState(g, 1.0, np.zeros(n, np.uint8), 1.0, np.zeros(n, np.uint16),
                          np.zeros(n, np.uint16), g_fmt=E5M2)
    gpu = GpuState([st.copy()])
    found, norm = gpu_norm(gpu, 1.0)
    assert (found, norm) == oracle.grad_norm([st], 1.0)
    assert norm == math.sqrt(57344.0 ** 2 + 44096 * 2.0 ** -32)


@pytest.mark.parametrize("case", ["nan_code", "e5m2_inf", "overflow"])
def test_grad_norm_found_inf(bo, case):
    wl = synth.tiny()
    fmt = E5M2 if case == "e5m2_inf" else E4M3
    states = states_for(wl, 1, fmt)
    ils = 1.0
    if case == "nan_code":
        states[2].g[1234] = 0xFF
    elif case == "e5m2_inf":
        states[0].g[5] = 0x7C
    else:
        states[1].g_scale = 1.0
        ils = 1e37
    gpu = GpuState([s.copy() for s in states])
    assert gpu_norm(gpu, ils) == (1, math.inf) == oracle.grad_norm(states, ils)


def clipped_lockstep(bo, wl, states, steps, max_norm, l2=False, fmt=E4M3,
                     misalign=()):
    gpu = None
    norms = []
    for t in range(1, steps + 1):
        codes, _, scale = oracle_cast(wl.grads(t), fmt)
        set_grads(states, codes, scale)
        if gpu is None:
            gpu = GpuState([s.copy() for s in states], misalign=misalign)
        else:
            gpu.load_state(states)
        f_ref, n_ref = oracle.adam_step_clipped(
            states, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
            wl.inv_loss_scale, max_norm, l2=l2)
        nd = torch.zeros(1, device="cuda")
        found = gpu.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
                         wl.inv_loss_scale, found_inf_dev=gpu.found_dev, l2=l2,
                         max_grad_norm=max_norm, grad_norm_dev=nd)
        assert found == f_ref == 0
        assert gpu.plan.last_grad_norm == n_ref
        assert nd.item() == np.float32(n_ref)
        gpu.compare(states)
        norms.append(n_ref)
    return norms


@pytest.mark.parametrize("l2", [False, True])
def test_clipped_steps_o2_long_tail(bo, l2):
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64,
                            n_tail=30)
    states = fresh_states(wl.weights(), o3=False)
    # the gradient norm of this list is far above 0.05: every step clips
    norms = clipped_lockstep(bo, wl, states, 3, 0.05, l2=l2)
    assert min(norms) > 0.05


def test_clipped_steps_o3_scaled_v_unaligned(bo):
    wl = synth.o3_1p3b(n_layer=1, d=64, ffn=256, vocab=300, ctx=32)
    states = fresh_states(wl.weights(), o3=True, scaled_v=True)
    clipped_lockstep(bo, wl, states, 2, 0.01, misalign={0, 3})


def test_clip_threshold_above_the_norm_equals_the_plain_step(bo):
    wl = synth.tiny()
    states = states_for(wl, 1)
    a = GpuState([s.copy() for s in states])
    b = GpuState([s.copy() for s in states])
    assert a.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, 1,
                  max_grad_norm=1e9) == 0
    assert b.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, 1) == 0
    for i in range(len(states)):
        assert torch.equal(a.m[i], b.m[i]) and torch.equal(a.v[i], b.v[i])
        assert torch.equal(a.w[i], b.w[i])
    assert torch.equal(a.m_scale, b.m_scale)


def test_clipped_step_with_found_inf_writes_nothing(bo):
    wl = synth.tiny()
    states = states_for(wl, 1)
    states[0].g[10] = 0x7F
    gpu = GpuState([s.copy() for s in states])
    found = gpu.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, 1,
                     found_inf_dev=gpu.found_dev, max_grad_norm=0.1)
    assert found == 1 and gpu.found_dev.item() == 1
    assert gpu.plan.last_grad_norm == math.inf
    for i, s in enumerate(states):
        assert np.array_equal(to_np_u8(gpu.m[i]), s.m)
        assert np.array_equal(to_np_u16(gpu.v[i]), s.v)
        assert np.array_equal(to_np_u16(gpu.w[i]), s.w)


def test_optimizer_with_clipping_against_the_oracle(bo):
    """Fp8AdamW(max_grad_norm): the library's cast, then the clipped step; the
    oracle follows from the same gradient values."""
    wl = synth.tiny()
    params = [w.cuda() for w in wl.weights()]
    opt = bo.Fp8AdamW(params, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                      weight_decay=wl.wd, max_grad_norm=0.02)
    assert opt.fused           # one fp8_cast_adam_step_clipped call per step
    states = fresh_states(wl.weights(), o3=False)
    for t in range(1, 4):
        grads = wl.grads(t)
        assert opt.step([g.cuda() for g in grads]) == 0
        codes, _, scale = oracle_cast(grads, E4M3)
        set_grads(states, codes, scale)
        f, n = oracle.adam_step_clipped(states, wl.lr, wl.beta1, wl.beta2,
                                        wl.eps, wl.wd, t, 1.0, 0.02)
        assert f == 0 and opt.last_grad_norm == n
        check_f32_exact(opt.m_scale.cpu().numpy()[:3], [s.m_scale[0] for s in states])
        for i, s in enumerate(states):
            assert np.array_equal(to_np_u16(params[i].view(-1)), s.w) or \
                np.abs(to_np_u16(params[i].view(-1)).astype(int) - s.w.astype(int)).max() <= 1


# ------------------------------------- the cast and the clipped step fused

def fused_clipped_lockstep(bo, wl, steps, max_norm, l2=False, o3=False,
                           scaled_v=False, fmt="e4m3", misalign=()):
    """fp8_cast_adam_step_clipped over the whole list against the oracle's
    cast, then its clipped step, from the same gradient values."""
    f = oracle.FMT[fmt]
    states = fresh_states(wl.weights(), o3=o3, g_fmt=f, scaled_v=scaled_v)
    gpu = GpuState([s.copy() for s in states], misalign=misalign)
    n = len(states)
    srcs = [torch.zeros(x, dtype=wl.grad_dtype, device="cuda") for x in wl.numels]
    amax = torch.zeros(n, device="cuda")
    cast = bo.CastPlan(srcs, gpu.g, amax, gpu.g_scale, fmt)
    fused = bo.CastStepPlan(cast, gpu.plan)
    norms = []
    for t in range(1, steps + 1):
        grads = wl.grads(t)
        for d, h in zip(srcs, grads):
            d.copy_(h)
        codes, _, scale = oracle_cast(grads, f)
        set_grads(states, codes, scale)
        gpu.load_state(states)
        f_ref, n_ref = oracle.adam_step_clipped(
            states, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
            wl.inv_loss_scale, max_norm, l2=l2)
        nd = torch.zeros(1, device="cuda")
        found = fused(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
                      wl.inv_loss_scale, found_inf_dev=gpu.found_dev, l2=l2,
                      max_grad_norm=max_norm, grad_norm_dev=nd)
        assert found == f_ref
        assert fused.last_grad_norm == n_ref
        if f_ref == 0:
            assert nd.item() == np.float32(n_ref)
            for i, c in enumerate(codes):
                assert np.array_equal(to_np_u8(gpu.g[i]), c)
            gpu.compare(states)
        norms.append(n_ref)
    return gpu, states, norms


@pytest.mark.parametrize("l2", [False, True])
def test_fused_clipped_long_tail(bo, l2):
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64,
                            n_tail=30)
    _, _, norms = fused_clipped_lockstep(bo, wl, 3, 0.05, l2=l2)
    assert min(norms) > 0.05


@pytest.mark.parametrize("o3,scaled_v,fmt", [(False, False, "e4m3"),
                                              (True, True, "e5m2")])
def test_fused_adam_l2_without_norm(bo, o3, scaled_v, fmt):
    """Adam with L2 decay through fp8_cast_adam_step_clipped with no norm
    asked for: the cast's encode pass fused with the step's first pass,
    which reads the weights for the decay term.  Every code, scale and
    state byte against the oracle's cast and then its step."""
    wl = synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64,
                            n_tail=30)
    f = oracle.FMT[fmt]
    states = fresh_states(wl.weights(), o3=o3, g_fmt=f, scaled_v=scaled_v)
    gpu = GpuState([s.copy() for s in states])
    srcs = [torch.zeros(x, dtype=wl.grad_dtype, device="cuda") for x in wl.numels]
    amax = torch.zeros(len(states), device="cuda")
    fused = bo.CastStepPlan(bo.CastPlan(srcs, gpu.g, amax, gpu.g_scale, fmt),
                            gpu.plan)
    for t in range(1, 4):
        grads = wl.grads(t)
        for d, h in zip(srcs, grads):
            d.copy_(h)
        codes, amax_ref, scale = oracle_cast(grads, f)
        set_grads(states, codes, scale)
        gpu.load_state(states)
        f_ref = oracle.adamw_step(states, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd,
                                  t, wl.inv_loss_scale, l2=True)
        found = fused(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
                      wl.inv_loss_scale, found_inf_dev=gpu.found_dev, l2=True)
        assert found == f_ref == 0
        assert fused.last_grad_norm is None
        assert np.array_equal(amax.cpu().numpy(), amax_ref)
        for i, c in enumerate(codes):
            assert np.array_equal(to_np_u8(gpu.g[i]), c)
        gpu.compare(states)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_fused_clipped_formats_and_sources(bo, fmt, dtype):
    """Whole 32768-element chunks of 16-bit sources take the encode pass's
    tile pipeline (E5M2 codes with their two-part sums), FP32 sources and
    ragged ends the per-chunk path: every code, the norm and the state
    against the oracle over three steps."""
    wl = dataclasses.replace(
        synth.o2_6p7b_tail(n_layer=1, d=128, ffn=512, vocab=3000, ctx=64,
                           n_tail=30), grad_dtype=dtype)
    _, _, norms = fused_clipped_lockstep(bo, wl, 3, 0.05, fmt=fmt)
    assert min(norms) > 0.05


def test_fused_clipped_o3_scaled_v_e5m2_unaligned(bo):
    wl = synth.o3_1p3b(n_layer=1, d=64, ffn=256, vocab=300, ctx=32)
    fused_clipped_lockstep(bo, wl, 2, 0.01, o3=True, scaled_v=True, fmt="e5m2",
                           misalign={0, 3})


def test_fused_clipped_threshold_above_norm_and_zero(bo):
    wl = synth.tiny()
    fused_clipped_lockstep(bo, wl, 2, 1e9)      # never clips
    fused_clipped_lockstep(bo, wl, 2, 0.0)      # measures only


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fused_clipped_inf_in_a_gradient_skips(bo, fmt):
    wl = dataclasses.replace(synth.o2_350m(n_layer=1, d=64, ffn=256, vocab=300,
                                           ctx=32), inf_site=(3, 17))
    gpu, states, norms = fused_clipped_lockstep(bo, wl, 1, 0.1, fmt=fmt)
    assert norms == [math.inf]
    for i, s in enumerate(states):
        assert np.array_equal(to_np_u8(gpu.m[i]), s.m)
        assert np.array_equal(to_np_u16(gpu.w[i]), s.w)


def test_fused_clipped_equals_the_two_calls(bo):
    """fp8_cast_adam_step_clipped against fp8_cast_scaled followed by
    fp8_adam_step_clipped on the same buffers: identical bytes."""
    wl = synth.o2_6p7b_tail(n_layer=1, d=64, ffn=256, vocab=1000, ctx=32,
                            n_tail=20)
    outs = []
    for fused in (True, False):
        params = [w.cuda() for w in wl.weights()]
        opt = bo.Fp8AdamW(params, lr=wl.lr, weight_decay=0.1, fused=fused,
                          max_grad_norm=0.03)
        norms = []
        for t in (1, 2, 3):
            assert opt.step([g.cuda() for g in wl.grads(t)]) == 0
            norms.append(opt.last_grad_norm)
        outs.append((params, opt, norms))
    (pa, oa, na), (pb, ob, nb) = outs
    assert na == nb
    for x, y in zip(pa, pb):
        assert torch.equal(x, y)
    for x, y in zip(oa.m + oa.v, ob.m + ob.v):
        assert torch.equal(x, y)
    assert torch.equal(oa.m_scale, ob.m_scale)


# ------------- found_inf of the split step's first pass under a clip factor
#
# GradScaler unscales the gradients, and finds any inf, before
# clip_grad_norm_ runs: a gradient that overflows fp32 when unscaled skips
# the step even where the clip coefficient would bring it back in range.
# With k0 = 2^121 an E4M3 code overflows exactly from magnitude 0x70 (128 *
# 2^121 = 2^128) up, while 0x6F (120) stays finite; the clip coefficient
# 2^-8 brings every code back in range.

K0_EXP, CLIP = 121, 2.0 ** -8


def boundary_states(top_code):
    """Two tensors; tensor 0's gradient holds top_code (and smaller codes),
    tensor 1 is ordinary; unscaled by k0 = 2^121 through g_scale."""
    rng = np.random.default_rng(31)
    out = []
    for i, n in enumerate((5000, 3000)):
        g = rng.integers(0, 0x40, n).astype(np.uint8) | \
            (rng.integers(0, 2, n).astype(np.uint8) << 7)
        if i == 0:
            g[1234] = top_code
            g[4321] = 0x6F
        w = oracle.f32_to_f16((rng.standard_normal(n) * 0.02).astype(np.float32))
        out.append(oracle.StepState(g, float(2.0 ** -K0_EXP) if i == 0 else 1.0,
                                    np.zeros(n, np.uint8), 1.0,
                                    np.zeros(n, np.uint16), w))
    return out


HP = (1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 1.0)


def assert_unchanged(gpu, states):
    for i, s in enumerate(states):
        assert np.array_equal(to_np_u8(gpu.m[i]), s.m)
        assert np.array_equal(to_np_u16(gpu.v[i]), s.v)
        assert np.array_equal(to_np_u16(gpu.w[i]), s.w)
    check_f32_exact(gpu.m_scale.cpu().numpy()[:len(states)],
                    [s.m_scale[0] for s in states], "m_scale")


@pytest.mark.parametrize("top", [0x6F, 0x70, 0xF0, 0x7E])
@pytest.mark.parametrize("finish", [False, True])
def test_split_step_found_inf_is_unclipped(bo, top, finish):
    states = boundary_states(top)
    expect = 0 if top == 0x6F else 1
    gpu = GpuState([s.copy() for s in states])
    ref = [s.copy() for s in states]
    assert oracle.adam_step_coef(ref, *HP, CLIP) == expect
    clip = torch.full((1,), CLIP, device="cuda")
    found = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    hp = HP + (False,)
    gpu.plan.begin(hp, clip=clip, found=found)
    torch.cuda.synchronize()
    assert found.item() == expect
    if finish:
        out = torch.full((1,), 7, dtype=torch.int32, device="cuda")
        gpu.plan.finish(hp, clip=clip, found=out)
        torch.cuda.synchronize()
        assert out.item() == expect
        if expect:
            assert_unchanged(gpu, states)
        else:
            gpu.compare(ref)


@pytest.mark.parametrize("top", [0x6F, 0x70])
def test_clipped_step_found_inf_is_unclipped(bo, top):
    """fp8_adam_step_clipped on the same gradients: the norm (+inf when
    found_inf) and the state against the oracle's clipped step."""
    states = boundary_states(top)
    gpu = GpuState([s.copy() for s in states])
    ref = [s.copy() for s in states]
    f_ref, n_ref = oracle.adam_step_clipped(ref, *HP, 1.0)
    assert f_ref == (0 if top == 0x6F else 1)
    found = gpu.plan(*HP, found_inf_dev=gpu.found_dev, max_grad_norm=1.0)
    assert found == f_ref == gpu.found_dev.item()
    assert gpu.plan.last_grad_norm == n_ref
    if f_ref:
        assert_unchanged(gpu, states)
    else:
        gpu.compare(ref)


def test_fused_clipped_found_inf_is_unclipped(bo):
    """fp8_cast_adam_step_clipped: a float32 gradient near the fp32 maximum
    casts to finite codes whose unscaled value (inv_loss_scale 4) overflows,
    while the clipped one would not: found_inf = 1 and nothing written, as in
    the oracle's cast followed by its clipped step."""
    rng = np.random.default_rng(33)
    grads = [torch.from_numpy((rng.standard_normal(n) * 1e-3).astype(np.float32))
             for n in (4000, 2500)]
    grads[1][77] = 2.0e38
    ils = 4.0
    states = fresh_states([torch.zeros(g.numel(), dtype=torch.float16) for g in grads],
                          o3=False)
    codes, _, scale = oracle_cast(grads, E4M3)
    set_grads(states, codes, scale)
    k1 = np.float32(np.float32(ils) / np.float32(scale[1]))
    with np.errstate(over="ignore"):
        assert codes[1][77] == 0x7E and not np.isfinite(np.float32(448.0) * k1)
    ref = [s.copy() for s in states]
    f_ref, n_ref = oracle.adam_step_clipped(ref, 1e-3, 0.9, 0.999, 1e-8, 0.01, 1,
                                            ils, 1.0)
    assert (f_ref, n_ref) == (1, math.inf)
    gpu = GpuState([s.copy() for s in states])
    srcs = [g.cuda() for g in grads]
    amax = torch.zeros(2, device="cuda")
    fused = bo.CastStepPlan(bo.CastPlan(srcs, gpu.g, amax, gpu.g_scale, "e4m3"),
                            gpu.plan)
    found = fused(1e-3, 0.9, 0.999, 1e-8, 0.01, 1, ils,
                  found_inf_dev=gpu.found_dev, max_grad_norm=1.0)
    assert found == 1 and gpu.found_dev.item() == 1
    assert fused.last_grad_norm == math.inf
    assert_unchanged(gpu, states)
