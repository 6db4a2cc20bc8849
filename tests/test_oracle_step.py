"""Pins of the oracle's FP8-state AdamW step.

* torch.optim.AdamW in float64 (a library routine) run from the dequantized
  state: the oracle's stored FP16 v / w are within one FP16 ulp of it and its
  E4M3 first moment within one code, across settings where eps, weight decay
  and the bias corrections each move the result.
* the closed form of the first bias-corrected step, and the beta1 = beta2 = 0
  special case (a sign-like normalised step at every step).
* the GradScaler check against torch's own non-finite-check-and-unscale.
* the O3 weight copy, the empty tensor, and the 62.5% state footprint.
"""
import os

import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
F32 = 0

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tdec(codes, fmt=E4M3):
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(codes)).view(dt).double()


def f16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).double()


def f16_bits(x64):
    return x64.numpy().astype(np.float16).view(np.uint16)


def make_states(orc, sizes, rng, g_sigma=1e-2, m_sigma=1e-3, v_mag=1e-6,
                o3=False, g_fmt=E4M3, fresh=False):
    states = []
    for n in sizes:
        g, _, gs = orc.cast_scaled(
            (rng.standard_normal(n) * g_sigma).astype(np.float32), F32, g_fmt)
        if fresh:
            m, ms = np.zeros(n, np.uint8), np.float32(1.0)
            v = np.zeros(n, np.uint16)
        else:
            m, _, ms = orc.cast_scaled(
                (rng.standard_normal(n) * m_sigma).astype(np.float32), F32, E4M3)
            v = (np.abs(rng.standard_normal(n)) * v_mag).astype(np.float16).view(np.uint16)
        w = (rng.standard_normal(n) * 0.02).astype(np.float16).view(np.uint16)
        states.append(orc.StepState(g, gs, m, ms, v, w, g_fmt=g_fmt, o3=o3))
    return states


def torch_adamw_f64(st, lr, b1, b2, eps, wd, step, ils):
    """One torch.optim.AdamW step in float64 from the dequantized state."""
    p = torch.nn.Parameter(f16(st.w).clone())
    p.grad = tdec(st.g, st.g_fmt) / float(st.g_scale) * ils
    opt = torch.optim.AdamW([p], lr=lr, betas=(b1, b2), eps=eps,
                            weight_decay=wd, foreach=False)
    opt.state[p] = {
        "step": torch.tensor(float(step - 1)),
        "exp_avg": tdec(st.m) / float(st.m_scale[0]),
        "exp_avg_sq": f16(st.v).clone(),
    }
    opt.step()
    s = opt.state[p]
    return p.detach(), s["exp_avg"], s["exp_avg_sq"]


def within_one_f16_ulp(bits, x64, min_exact):
    rne = f16_bits(x64).astype(np.int32)
    got = bits.astype(np.int32)
    d = np.abs(got - rne)
    # same-sign fp16 patterns are ordered, so a bit difference of 1 is one ulp
    same_sign = (got >> 15) == (rne >> 15)
    ok = (d <= 1) & (same_sign | (x64.abs().numpy() < 6e-8))
    assert ok.all(), (np.flatnonzero(~ok)[:5], got[~ok][:5], rne[~ok][:5])
    assert (d == 0).mean() >= min_exact


SETTINGS = [
    # lr, beta1, beta2, eps, wd, step, inv_loss_scale
    (1e-2, 0.9, 0.99, 1e-3, 0.1, 3, 1.0),       # eps comparable to sqrt(v)
    (1e-3, 0.9, 0.999, 1e-8, 0.01, 1, 0.5),     # first step
    (5e-3, 0.8, 0.95, 1e-6, 0.0, 10, 2.0 ** -10),
    (1e-2, 0.0, 0.5, 1e-4, 0.5, 2, 1.0),
]


@pytest.mark.parametrize("setting", SETTINGS)
@pytest.mark.parametrize("o3", [False, True])
def test_step_matches_torch_adamw_float64(orc, setting, o3):
    lr, b1, b2, eps, wd, step, ils = setting
    rng = np.random.default_rng(hash((setting, o3)) % 2**32)
    states = make_states(orc, [37, 64, 1000], rng, g_sigma=1e-2 / ils, o3=o3)
    before = [s.copy() for s in states]
    assert orc.adamw_step(states, lr, b1, b2, eps, wd, step, ils) == 0
    for s0, s1 in zip(before, states):
        w64, m64, v64 = torch_adamw_f64(s0, lr, b1, b2, eps, wd, step, ils)
        within_one_f16_ulp(s1.v, v64, 0.99)
        within_one_f16_ulp(s1.w, w64, 0.99)
        # E4M3 first moment: scale from this step's amax, code within 1
        amax64 = m64.abs().max().item()
        assert abs(float(s1.m_scale[0]) - 448.0 / amax64) <= 4e-7 * 448.0 / amax64
        ref = torch.from_numpy((m64.numpy() * float(s1.m_scale[0])).astype(np.float32))
        ref_codes = ref.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        dcode = np.abs(s1.m.astype(np.int32) - ref_codes.astype(np.int32))
        dcode = np.where((s1.m ^ ref_codes) & 0x80, 999, dcode)
        ok = (dcode <= 1) | (np.abs(m64.numpy()) * float(s1.m_scale[0]) < 2.0 ** -9)
        assert ok.all()
        if o3:
            master = s1.w.view(np.float16).astype(np.float32)
            assert s1.w8_amax[0] == np.abs(master).max()
            assert s1.w8_scale[0] == np.float32(448.0) / s1.w8_amax[0]
            ref8 = (torch.from_numpy(master) * torch.tensor(s1.w8_scale[0])).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(s1.w8, ref8)


def test_first_step_closed_form(orc):
    """m = v = 0, t = 1: m_hat = g and v_hat = g^2, so
    w1 = w0 (1 - lr wd) - lr g / (|g| + eps) ~= w0 (1 - lr wd) - lr sign(g)."""
    rng = np.random.default_rng(3)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    states = make_states(orc, [4096], rng, g_sigma=1e-3, fresh=True)
    s0 = states[0].copy()
    assert orc.adamw_step(states, lr, b1, b2, eps, wd, 1, 1.0) == 0
    g = (tdec(s0.g) / s0.g_scale).numpy()
    w0 = f16(s0.w).numpy()
    closed = w0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    within_one_f16_ulp(states[0].w, torch.from_numpy(closed), 0.99)
    big = np.abs(g) > 1e3 * eps                 # eps << |g|
    assert big.mean() > 0.9
    sign_step = w0 * (1 - lr * wd) - lr * np.sign(g)
    got = f16(states[0].w).numpy()
    ulp = np.spacing(np.abs(sign_step).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(got - sign_step)[big] <= (ulp + 2e-3 * lr)[big])
    # stored moments: v = (1 - beta2) g^2, m = (1 - beta1) g
    within_one_f16_ulp(states[0].v, torch.from_numpy((1 - b2) * g * g), 0.99)
    m_back = tdec(states[0].m).numpy() / states[0].m_scale[0]
    assert np.allclose(m_back, (1 - b1) * g, rtol=2 ** -4, atol=1e-12)


def test_zero_betas_give_normalised_step_every_step(orc):
    """beta1 = beta2 = 0, wd = 0: both bias corrections are 1, m = g and
    v = g^2, so each step moves w by lr g / (|g| + eps)."""
    rng = np.random.default_rng(4)
    lr, eps = 1e-2, 1e-6
    states = make_states(orc, [333], rng, g_sigma=1e-3)
    for t in range(1, 6):
        new = make_states(orc, [333], rng, g_sigma=1e-3)[0]
        states[0].g, states[0].g_scale = new.g, new.g_scale
        s0 = states[0].copy()
        assert orc.adamw_step(states, lr, 0.0, 0.0, eps, 0.0, t, 1.0) == 0
        g = (tdec(s0.g) / s0.g_scale).numpy()
        expect = f16(s0.w).numpy() - lr * g / (np.abs(g) + eps)
        within_one_f16_ulp(states[0].w, torch.from_numpy(expect), 0.99)
        within_one_f16_ulp(states[0].v, torch.from_numpy(g * g), 0.99)


@pytest.mark.parametrize("case", ["nan_code", "overflow_after_unscale",
                                  "e5m2_inf", "clean"])
def test_found_inf_matches_torch_gradscaler_check(orc, case):
    rng = np.random.default_rng(5)
    g_fmt = E5M2 if case == "e5m2_inf" else E4M3
    states = make_states(orc, [50, 70], rng, g_fmt=g_fmt)
    ils = 1.0
    if case == "nan_code":
        states[1].g[13] = 0xFF
    elif case == "e5m2_inf":
        states[0].g[7] = 0x7C
    elif case == "overflow_after_unscale":
        states[0].g_scale = float(np.float32(1e-36))
        ils = 1e10
    before = [s.copy() for s in states]
    found = orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.01, 2, ils)
    grads = [(tdec(s.g, s.g_fmt).float() * (np.float32(1.0) / np.float32(s.g_scale)))
             for s in before]
    flag = torch.zeros(1)
    torch._amp_foreach_non_finite_check_and_unscale_(
        grads, flag, torch.tensor(ils, dtype=torch.float32))
    assert found == int(flag.item())
    assert found == (0 if case == "clean" else 1)
    if found:
        for a, b in zip(before, states):
            for k in ("m", "m_scale", "v", "w"):
                assert np.array_equal(getattr(a, k), getattr(b, k))


@pytest.mark.parametrize("l2", [False, True])
def test_found_inf_looks_at_the_gradients_only(orc, l2):
    """GradScaler's check runs over the unscaled gradients alone, before the
    optimizer adds any decay term: an infinite weight with finite gradients
    is no found_inf, in AdamW or in Adam-L2 mode, and the step runs."""
    rng = np.random.default_rng(13)
    states = make_states(orc, [40, 60], rng)
    states[1].w[3] = 0x7C00                       # +inf FP16 weight
    before = [s.copy() for s in states]
    grads = [(tdec(s.g, s.g_fmt).float() * (np.float32(1.0) / np.float32(s.g_scale)))
             for s in states]
    flag = torch.zeros(1)
    torch._amp_foreach_non_finite_check_and_unscale_(
        grads, flag, torch.tensor(1.0, dtype=torch.float32))
    assert flag.item() == 0
    assert orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.01, 2, 1.0, l2=l2) == 0
    assert not np.isfinite(f16(states[1].w[3:4]).numpy()[0])
    assert not np.array_equal(states[0].w, before[0].w)


def test_empty_and_zero_tensors(orc):
    rng = np.random.default_rng(6)
    states = make_states(orc, [0, 16, 5], rng, fresh=True)
    states[2].g[:] = 0
    states[2].g_scale = 1.0
    w_before = states[2].w.copy()
    assert orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0) == 0
    assert states[0].m_scale[0] == 1.0          # empty: amax 0 -> scale 1
    assert states[2].m_scale[0] == 1.0          # zero moment -> scale 1
    assert not states[2].m.any() and not states[2].v.any()
    assert np.array_equal(states[2].w, w_before)   # wd 0, zero update


def test_bad_arguments(orc):
    rng = np.random.default_rng(8)
    states = make_states(orc, [4], rng)
    with pytest.raises(ValueError):
        orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.0, 0, 1.0)


def read_levels():
    rows, saving = {}, None
    for line in open(os.path.join(GOLDEN, "optimization_levels.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "saving_O2_percent":
            saving = float(f[1])
        else:
            rows[f[0]] = f[1:]
    return rows, saving


def test_state_footprint_is_the_published_saving(orc):
    rows, saving = read_levels()
    width = {"FP8": 1, "FP16": 2, "FP32": 4}
    for lvl, name in ((0, "FP16_AMP"), (1, "MSAMP_O1"), (2, "MSAMP_O2"),
                      (3, "MSAMP_O3")):
        a, b = rows[name][5].split("+")
        assert orc.state_bytes(lvl) == width[a] + width[b]
    # the oracle's own state arrays: uint8 first moment, uint16 second moment
    st = make_states(orc, [10], np.random.default_rng(0))[0]
    assert st.m.itemsize + st.v.itemsize == orc.state_bytes(2) == 3
    assert 100.0 * (1 - orc.state_bytes(2) / orc.state_bytes(0)) == saving


# ------------------------------------------- scaled second moment, Adam L2

def make_states_v(orc, sizes, rng, g_sigma, scaled_v, o3=False):
    """Fresh state (m = v = 0), gradients N(0, g_sigma) cast to E4M3."""
    out = []
    for n in sizes:
        g, _, gs = orc.cast_scaled(
            (rng.standard_normal(n) * g_sigma).astype(np.float32), F32, E4M3)
        w = (rng.standard_normal(n) * 0.02).astype(np.float16).view(np.uint16)
        out.append(orc.StepState(g, gs, np.zeros(n, np.uint8), 1.0,
                                 np.zeros(n, np.uint16), w, o3=o3,
                                 scaled_v=scaled_v))
    return out


def stored_v(st):
    """The second moment a state holds, as float64."""
    v = f16(st.v)
    if st.v_bound is not None:
        v = v * (float(st.v_bound[0]) * 2.0 ** -14)
    return v


def torch_step_f64(st, lr, b1, b2, eps, wd, step, ils, l2):
    """One torch.optim.AdamW (or torch.optim.Adam with L2 weight decay) step
    in float64 from the state's dequantized values."""
    p = torch.nn.Parameter(f16(st.w).clone())
    p.grad = tdec(st.g, st.g_fmt) / float(st.g_scale) * ils
    cls = torch.optim.Adam if l2 else torch.optim.AdamW
    opt = cls([p], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd,
              foreach=False)
    opt.state[p] = {"step": torch.tensor(float(step - 1)),
                    "exp_avg": tdec(st.m) / float(st.m_scale[0]),
                    "exp_avg_sq": stored_v(st).clone()}
    opt.step()
    return p.detach(), opt.state[p]["exp_avg_sq"]


def run_against_torch(orc, states, steps, lr, b1, b2, eps, wd, l2, rng,
                      g_sigma):
    """Steps 1..steps; each step compares the oracle with torch in float64
    from the same dequantized state; returns the worst relative v error and
    the fraction of weights within one FP16 ulp."""
    worst_v, w_ok = 0.0, []
    for t in range(1, steps + 1):
        for s in states:
            g, _, gs = orc.cast_scaled(
                (rng.standard_normal(s.numel) * g_sigma).astype(np.float32), F32, E4M3)
            s.g, s.g_scale = g, float(gs)
        before = [s.copy() for s in states]
        assert orc.adamw_step(states, lr, b1, b2, eps, wd, t, 1.0, l2=l2) == 0
        for s0, s1 in zip(before, states):
            w64, v64 = torch_step_f64(s0, lr, b1, b2, eps, wd, t, 1.0, l2)
            got = stored_v(s1).numpy()
            ref = v64.numpy()
            big = ref > ref.max() * 2.0 ** -20
            worst_v = max(worst_v, float(np.max(np.abs(got - ref)[big] / ref[big])))
            rne = f16_bits(w64).astype(np.int32)
            w_ok.append(np.abs(s1.w.astype(np.int32) - rne) <= 1)
    return worst_v, float(np.mean(np.concatenate(w_ok)))


def free_run_weight_change(orc, scaled_v, g_sigma, steps=3):
    """The oracle and torch.optim.AdamW (float64 state throughout) run side by
    side on the same dequantized gradients; returns the median relative
    difference of their total weight change."""
    lr, betas, eps, wd = 1e-3, (0.9, 0.999), 1e-8, 0.0
    states = make_states_v(orc, [3000], np.random.default_rng(1), g_sigma, scaled_v)
    st = states[0]
    w0 = f16(st.w).clone()
    p = torch.nn.Parameter(w0.clone())
    opt = torch.optim.AdamW([p], lr=lr, betas=betas, eps=eps, weight_decay=wd,
                            foreach=False)
    rng = np.random.default_rng(2)
    for t in range(1, steps + 1):
        g, _, gs = orc.cast_scaled((rng.standard_normal(3000) * g_sigma)
                                   .astype(np.float32), F32, E4M3)
        st.g, st.g_scale = g, float(gs)
        p.grad = tdec(g) / float(gs)
        opt.step()
        assert orc.adamw_step(states, lr, *betas, eps, wd, t, 1.0) == 0
    dw_torch = (p.detach() - w0).numpy()
    dw_oracle = (f16(st.w) - w0).numpy()
    keep = np.abs(dw_torch) > 1e-4
    return float(np.median(np.abs(dw_oracle - dw_torch)[keep] / np.abs(dw_torch)[keep]))


def test_scaled_v_follows_torch_where_plain_fp16_underflows(orc):
    """Gradients near 1e-5: (1 - beta2) g^2 ~ 1e-13 is below FP16's smallest
    subnormal, so a plain FP16 second moment stores 0 and every later step
    sees only its own (1 - beta2) g^2, off by the whole history; the scaled
    second moment keeps the trajectory torch's AdamW takes (to the precision
    of the E4M3 first moment and the FP16 weights)."""
    assert free_run_weight_change(orc, False, 1e-5) > 0.3      # the hazard
    assert free_run_weight_change(orc, True, 1e-5) < 0.02
    # with gradients FP16 can hold, both follow torch
    assert free_run_weight_change(orc, False, 1e-1) < 0.02
    assert free_run_weight_change(orc, True, 1e-1) < 0.02


@pytest.mark.parametrize("l2", [False, True])
@pytest.mark.parametrize("o3", [False, True])
def test_scaled_v_and_l2_match_torch_over_steps(orc, l2, o3):
    states = make_states_v(orc, [37, 1000, 2048], np.random.default_rng(3), 1e-2,
                           True, o3=o3)
    worst, ok = run_against_torch(orc, states, 5, lr=3e-3, b1=0.9, b2=0.99,
                                  eps=1e-6, wd=0.1, l2=l2,
                                  rng=np.random.default_rng(4), g_sigma=1e-2)
    assert worst <= 2.0 ** -10
    assert ok >= 0.99


def test_l2_mode_plain_v_matches_torch_adam(orc):
    """Adam with L2 decay on the plain FP16 second moment (gradients large
    enough for FP16): torch.optim.Adam with weight_decay."""
    states = make_states_v(orc, [500, 64], np.random.default_rng(5), 1e-2, False)
    worst, ok = run_against_torch(orc, states, 4, lr=1e-2, b1=0.8, b2=0.95,
                                  eps=1e-4, wd=0.3, l2=True,
                                  rng=np.random.default_rng(6), g_sigma=1e-2)
    assert ok >= 0.99


@pytest.mark.parametrize("l2", [False, True])
def test_v_bound_holds_and_stays_below_fp16_overflow(orc, l2):
    """The bound covers every element of v.  With L2 decay v accumulates the
    decayed gradient g + wd * w, which here often outweighs g itself."""
    rng = np.random.default_rng(7)
    states = make_states_v(orc, [4096], rng, 1e-3, True)
    st = states[0]
    wd = 0.1 if l2 else 0.0
    for t in range(1, 11):
        sigma = 10.0 ** rng.uniform(-6, -1)           # gradients jump around
        g, _, gs = orc.cast_scaled((rng.standard_normal(4096) * sigma)
                                   .astype(np.float32), F32, E4M3)
        st.g, st.g_scale = g, float(gs)
        assert orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, wd, t, 1.0,
                              l2=l2) == 0
        codes = f16(st.v).numpy()
        assert codes.max() <= 16384 * (1 + 2.0 ** -9)   # far below 65504
        assert stored_v(st).max().item() <= st.v_bound[0] * (1 + 2.0 ** -9)
        assert codes.max() >= 16384 / 4096           # the bound is not loose


def test_scaled_v_with_a_tiny_bound_stores_only_finite_values(orc):
    """Gradients near 1e-17 give a bound B so small that 2^14 / B overflows
    fp32.  Finite gradients must still leave finite state: torch's second
    moment here is finite (and tiny), so no stored v or w may be inf or
    NaN."""
    rng = np.random.default_rng(16)
    states = make_states_v(orc, [300], rng, 1e-3, True)
    st = states[0]
    st.g_scale = float(np.float32(2.0 ** 64))       # |g| <= 448 * 2^-64
    assert orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0) == 0
    b = float(st.v_bound[0])
    assert 0.0 < b < 16384.0 / float(np.finfo(np.float32).max)
    assert np.isfinite(f16(st.v).numpy()).all()
    assert np.isfinite(f16(st.w).numpy()).all()


def test_found_inf_leaves_v_bound_unchanged(orc):
    states = make_states_v(orc, [100], np.random.default_rng(8), 1e-3, True)
    assert orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0) == 0
    b = states[0].v_bound.copy()
    states[0].g[3] = 0x7F
    before = states[0].copy()
    assert orc.adamw_step(states, 1e-3, 0.9, 0.999, 1e-8, 0.0, 2, 1.0) == 1
    assert np.array_equal(states[0].v_bound, b)
    assert np.array_equal(states[0].v, before.v)


def test_bias_power_is_beta_to_the_t(orc):
    """beta^t by binary exponentiation: exact where every product is exact
    (powers of two), otherwise within t * 2^-52 relative of the exact power
    (a rational computed with Python integers)."""
    from fractions import Fraction
    for b in (0.5, 0.25, 2.0 ** -10):
        for t in (1, 2, 3, 10, 77, 1000):
            assert orc.bias_power(b, t) == b ** t
    for b in (0.9, 0.999, 0.95, 0.8):
        for t in (1, 2, 5, 100, 1000, 12345):
            exact = Fraction(b) ** t
            if exact < Fraction(1, 2 ** 1000):       # past double's normal range
                continue
            got = Fraction(orc.bias_power(b, t))
            assert abs(got - exact) <= exact * Fraction(t, 2 ** 52)
    assert orc.bias_power(0.9, 0) == 1.0


# ------------------------------------------------ the step of a tensor's pieces

def piece_of(orc, st, a, b):
    """Elements [a, b) of a state as a state of its own with the tensor's
    scales and bound (copies)."""
    p = orc.StepState(st.g[a:b], st.g_scale, st.m[a:b], st.m_scale[0], st.v[a:b],
                      st.w[a:b], g_fmt=st.g_fmt, o3=st.w8 is not None,
                      scaled_v=st.v_bound is not None,
                      v_bound=st.v_bound[0] if st.v_bound is not None else 0.0)
    return p


def max_bits(values):
    """The largest of float32 maxima in the amax order (NaN above +inf above
    every finite value): as bit patterns of non-negative floats."""
    b = np.asarray(values, np.float32).view(np.int32)
    return np.int32(b.max()).view(np.float32)


@pytest.mark.parametrize("o3,scaled_v,l2,clip", [
    (False, False, False, 1.0), (True, False, False, 0.37),
    (False, True, True, 1.0), (True, True, False, 0.5)])
def test_pieces_with_the_whole_maxima_give_the_whole_step(orc, o3, scaled_v, l2,
                                                          clip):
    """A step's per-tensor quantities are maxima over the tensor's elements
    (this step's first-moment amax, max |g| for the bound, the new master's
    amax); everything else is elementwise.  So cutting every tensor into
    pieces, taking phase 1 on the pieces, combining each tensor's maxima by
    max, and running phases 2 and 3 on the pieces with the combined maxima
    must reproduce the whole step on every element and every scale."""
    rng = np.random.default_rng(41)
    sizes = [1, 700, 4099, 300]
    whole = make_states(orc, sizes, rng, o3=o3)
    if scaled_v:
        for st in whole:
            st.v_bound = np.array([1e-6], np.float32)
            st.v = (np.abs(rng.standard_normal(st.numel)) * 1000).astype(
                np.float16).view(np.uint16)
    hp = (1e-3, 0.9, 0.999, 1e-8, 0.01, 3, 0.5)
    pieces, owner = [], []
    for t, st in enumerate(whole):
        cuts = sorted(set([0, st.numel] + list(rng.integers(0, st.numel + 1, 3))))
        for a, b in zip(cuts, cuts[1:]):
            pieces.append((t, a, b, piece_of(orc, st, a, b)))
    ref = [s.copy() for s in whole]
    assert orc.adam_step_coef(ref, *hp, clip, l2=l2) == 0
    lr, b1, b2, eps, wd, step, ils = hp
    ps = [p for _, _, _, p in pieces]
    f, am, gm = orc.step_maxima(ps, lr, b1, b2, wd, step, ils, clip=clip, l2=l2)
    assert f == 0
    tam = [max_bits([am[i] for i, (t2, *_) in enumerate(pieces) if t2 == t])
           for t in range(len(whole))]
    tgm = [max_bits([gm[i] for i, (t2, *_) in enumerate(pieces) if t2 == t])
           for t in range(len(whole))]
    wm = orc.step_update(ps, lr, b1, b2, eps, wd, step, ils,
                         [tam[t] for t, *_ in pieces], [tgm[t] for t, *_ in pieces],
                         clip=clip, l2=l2)
    twm = [max_bits([wm[i] for i, (t2, *_) in enumerate(pieces) if t2 == t])
           for t in range(len(whole))]
    orc.weight_copy(ps, [twm[t] for t, *_ in pieces])
    for t, a, b, p in pieces:
        r = ref[t]
        assert np.array_equal(p.m, r.m[a:b]) and np.array_equal(p.v, r.v[a:b])
        assert np.array_equal(p.w, r.w[a:b])
        assert p.m_scale[0] == r.m_scale[0]
        if o3:
            assert np.array_equal(p.w8, r.w8[a:b])
            assert p.w8_scale[0] == r.w8_scale[0] and p.w8_amax[0] == r.w8_amax[0]
        if scaled_v:
            assert p.v_bound[0] == r.v_bound[0]


def test_phase_one_reports_found_inf_and_writes_nothing(orc):
    rng = np.random.default_rng(42)
    states = make_states(orc, [50, 60], rng)
    states[1].g[7] = 0x7F
    before = [s.copy() for s in states]
    assert orc.step_maxima(states, 1e-3, 0.9, 0.999, 0.01, 1, 1.0)[0] == 1
    for a, b in zip(states, before):
        assert np.array_equal(a.m, b.m) and a.m_scale[0] == b.m_scale[0]
