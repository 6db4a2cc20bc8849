"""Pins of the oracle's global gradient norm and the clipped step.

* the norm against torch.linalg.vector_norm in float64 of the dequantized,
  unscaled gradients (a library routine);
* exactness of each tensor's sum of squares where a plain double accumulation
  loses terms (one E5M2 maximum followed by 4096 minimum subnormals);
* invariants: a permutation within a tensor leaves the norm bit-identical,
  doubling every gradient scale halves it exactly;
* found_inf cases give +inf;
* the clipped step against torch.nn.utils.clip_grad_norm_ followed by
  torch.optim.AdamW / torch.optim.Adam, both in float64; a norm below the
  threshold leaves the step bit-identical to the unclipped one.
"""
import math

import numpy as np
import pytest
import torch

from test_oracle_step import f16, f16_bits, make_states, tdec, within_one_f16_ulp

E4M3, E5M2 = 0, 1


def torch_norm(states, ils):
    g = [tdec(s.g, s.g_fmt) * (float(np.float32(ils) / np.float32(s.g_scale)))
         for s in states]
    return torch.linalg.vector_norm(torch.cat(g), dtype=torch.float64).item()


@pytest.mark.parametrize("g_fmt", [E4M3, E5M2])
@pytest.mark.parametrize("ils", [1.0, 2.0 ** -16, 0.37])
def test_norm_matches_torch_float64(orc, g_fmt, ils):
    rng = np.random.default_rng(int(ils * 1000) + g_fmt)
    states = make_states(orc, [1, 37, 4096, 30000], rng, g_sigma=3e-3 / ils,
                         g_fmt=g_fmt)
    found, norm = orc.grad_norm(states, ils)
    assert found == 0
    ref = torch_norm(states, ils)
    assert abs(norm - ref) <= 1e-13 * ref


def test_each_tensor_sum_is_exact(orc):
    """57344^2 + 4096 * (2^-16)^2 = 57344^2 + 2^-20 is a double; adding the
    tiny squares one by one after the big one would lose all of them."""
    g = np.concatenate([[0x7B], np.full(4096, 0x01)]).astype(np.uint8)
    n = g.size
    st = orc.StepState(g, 1.0, np.zeros(n, np.uint8), 1.0, np.zeros(n, np.uint16),
                       np.zeros(n, np.uint16), g_fmt=E5M2)
    found, norm = orc.grad_norm([st], 1.0)
    exact_sq = 57344.0 ** 2 + 2.0 ** -20
    assert exact_sq != 57344.0 ** 2
    assert found == 0 and norm == math.sqrt(exact_sq)
    naive = 0.0
    for x in tdec(g, E5M2).numpy():
        naive += x * x
    assert math.sqrt(naive) != norm


def test_invariants(orc):
    rng = np.random.default_rng(5)
    states = make_states(orc, [100, 5000, 777], rng)
    _, n0 = orc.grad_norm(states, 1.0)
    perm = [s.copy() for s in states]
    for s in perm:
        s.g = s.g[rng.permutation(s.numel)].copy()
    assert orc.grad_norm(perm, 1.0)[1] == n0
    half = [s.copy() for s in states]
    for s in half:
        s.g_scale = float(np.float32(s.g_scale) * 2)
    assert orc.grad_norm(half, 1.0)[1] == n0 / 2
    assert orc.grad_norm(states, 4.0)[1] == n0 * 4


@pytest.mark.parametrize("case", ["nan_code", "inf_code", "overflow"])
def test_found_inf_gives_infinite_norm(orc, case):
    rng = np.random.default_rng(1)
    fmt = E4M3 if case != "inf_code" else E5M2
    states = make_states(orc, [300, 200], rng, g_fmt=fmt)
    ils = 1.0
    if case == "nan_code":
        states[1].g[17] = 0x7F
    elif case == "inf_code":
        states[0].g[3] = 0xFC
    else:                               # 448 * 1e37 overflows fp32
        states[0].g_scale, ils = 1.0, 1e37
    assert orc.grad_norm(states, ils) == (1, math.inf)


def test_clip_coefficient(orc):
    assert orc.clip_coef(0.5, 1.0) == 1.0
    assert orc.clip_coef(1.0 - 1e-6, 1.0) == 1.0
    assert orc.clip_coef(4.0, 1.0) == np.float32(1.0 / (4.0 + 1e-6))
    assert orc.clip_coef(4.0, 0.0) == 1.0 and orc.clip_coef(4.0, -1.0) == 1.0
    c = orc.clip_coef(123.0, 2.5)
    assert c * (123.0 + 1e-6) == pytest.approx(2.5, rel=1e-7)


def test_clip_coefficient_is_torchs_rounded_once(orc):
    """torch.nn.utils.clip_grad_norm_ in float64 scales every gradient by
    min(1, max_norm / (norm + 1e-6)); a unit gradient element then holds that
    coefficient exactly.  The oracle's coefficient is it rounded to float
    once, for the norm torch returns."""
    rng = np.random.default_rng(15)
    clipped = 0
    for _ in range(300):
        g = torch.tensor(rng.standard_normal(37) * 10.0 ** rng.uniform(-3, 3),
                         dtype=torch.float64)
        max_norm = float(np.float32(10.0 ** rng.uniform(-3, 1)))
        p1 = torch.zeros(37, dtype=torch.float64, requires_grad=True)
        p2 = torch.zeros(1, dtype=torch.float64, requires_grad=True)
        p1.grad, p2.grad = g.clone(), torch.ones(1, dtype=torch.float64)
        norm = torch.nn.utils.clip_grad_norm_([p1, p2], max_norm).item()
        coef = p2.grad.item()
        assert orc.clip_coef(norm, max_norm) == np.float32(coef)
        clipped += coef < 1.0
    assert 50 < clipped < 300


def torch_clipped_f64(st_list, lr, b1, b2, eps, wd, step, ils, max_norm, l2):
    """torch: dequantize, clip_grad_norm_ in float64, then one Adam / AdamW
    step per tensor from the dequantized state."""
    ps = []
    for st in st_list:
        p = torch.nn.Parameter(f16(st.w).clone())
        p.grad = tdec(st.g, st.g_fmt) * float(np.float32(ils) / np.float32(st.g_scale))
        ps.append(p)
    total = torch.nn.utils.clip_grad_norm_(ps, max_norm, foreach=False).item()
    cls = torch.optim.Adam if l2 else torch.optim.AdamW
    opt = cls(ps, lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    for p, st in zip(ps, st_list):
        opt.state[p] = {"step": torch.tensor(float(step - 1)),
                        "exp_avg": tdec(st.m) / float(st.m_scale[0]),
                        "exp_avg_sq": f16(st.v).clone()}
    opt.step()
    return total, [(p.detach(), opt.state[p]["exp_avg"], opt.state[p]["exp_avg_sq"])
                   for p in ps]


@pytest.mark.parametrize("l2", [False, True])
@pytest.mark.parametrize("max_norm", [0.05, 0.5])
def test_clipped_step_matches_torch(orc, l2, max_norm):
    rng = np.random.default_rng(int(max_norm * 100) + l2)
    lr, b1, b2, eps, wd, step, ils = 1e-3, 0.9, 0.999, 1e-8, 0.1, 3, 2.0 ** -8
    states = make_states(orc, [64, 1000, 5000], rng, g_sigma=1e-2 / ils)
    before = [s.copy() for s in states]
    found, norm = orc.adam_step_clipped(states, lr, b1, b2, eps, wd, step, ils,
                                        max_norm, l2=l2)
    assert found == 0
    total, ref = torch_clipped_f64(before, lr, b1, b2, eps, wd, step, ils,
                                   max_norm, l2)
    assert abs(norm - total) <= 1e-13 * total
    assert norm > max_norm          # the coefficient is below 1 here
    for s1, (w64, m64, v64) in zip(states, ref):
        within_one_f16_ulp(s1.v, v64, 0.99)
        within_one_f16_ulp(s1.w, w64, 0.99)
        amax64 = m64.abs().max().item()
        assert abs(float(s1.m_scale[0]) - 448.0 / amax64) <= 4e-7 * 448.0 / amax64


def test_norm_below_threshold_leaves_the_step_unchanged(orc):
    rng = np.random.default_rng(8)
    args = (1e-3, 0.9, 0.999, 1e-8, 0.01, 2, 1.0)
    states = make_states(orc, [100, 3000], rng)
    plain = [s.copy() for s in states]
    found, norm = orc.adam_step_clipped(states, *args, 1e9)
    assert found == 0 and orc.adamw_step(plain, *args) == 0
    for a, b in zip(states, plain):
        for f in ("m", "v", "w", "m_scale"):
            assert np.array_equal(getattr(a, f), getattr(b, f)), f
    # max_norm <= 0: the norm is reported, nothing is clipped
    states2 = [s.copy() for s in plain]
    assert orc.adam_step_clipped(states2, *args, 0.0)[0] == 0


def test_clipped_step_with_found_inf_writes_nothing(orc):
    rng = np.random.default_rng(9)
    states = make_states(orc, [100, 3000], rng)
    states[1].g[5] = 0x7F
    before = [s.copy() for s in states]
    assert orc.adam_step_clipped(states, 1e-3, 0.9, 0.999, 1e-8, 0.01, 2, 1.0,
                                 0.1) == (1, math.inf)
    for a, b in zip(states, before):
        for f in ("m", "v", "w", "m_scale"):
            assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_found_inf_is_decided_before_clipping(orc):
    """torch's recipe unscales the gradients (finding any inf) before
    clip_grad_norm_ runs: a gradient that overflows fp32 when unscaled skips
    the step even where the clip coefficient would bring it back in range."""
    rng = np.random.default_rng(14)
    states = make_states(orc, [50, 70], rng)
    s = states[0]
    s.g[:] = 0
    s.g[9] = 0x7E                                 # 448
    s.g_scale = float(np.float32(2.0 ** -120))    # 448 * 2^120 > fp32 max
    clip = 2.0 ** -8                              # 448 * 2^112 is finite
    grads = [(tdec(x.g, x.g_fmt).float() * (np.float32(1.0) / np.float32(x.g_scale)))
             for x in states]
    flag = torch.zeros(1)
    torch._amp_foreach_non_finite_check_and_unscale_(
        grads, flag, torch.tensor(1.0, dtype=torch.float32))
    assert flag.item() == 1
    assert np.isfinite(np.float32(448.0) * (np.float32(2.0 ** 120) * np.float32(clip)))
    before = [x.copy() for x in states]
    assert orc.adam_step_coef(states, 1e-3, 0.9, 0.999, 1e-8, 0.01, 2, 1.0, clip) == 1
    for a, b in zip(states, before):
        for f in ("m", "v", "w", "m_scale"):
            assert np.array_equal(getattr(a, f), getattr(b, f)), f


def test_step_with_a_given_coefficient_is_the_clipped_step(orc):
    rng = np.random.default_rng(11)
    args = (1e-3, 0.9, 0.999, 1e-8, 0.01, 2, 1.0)
    states = make_states(orc, [100, 3000], rng)
    a = [s.copy() for s in states]
    b = [s.copy() for s in states]
    c = [s.copy() for s in states]
    found, norm = orc.adam_step_clipped(a, *args, 0.01)
    assert found == 0
    assert orc.adam_step_coef(b, *args, orc.clip_coef(norm, 0.01)) == 0
    assert orc.grad_norm_codes([s.g for s in states], [s.g_scale for s in states],
                               E4M3, 1.0) == (0, norm)
    assert orc.adam_step_coef(c, *args, 1.0) == 0
    plain = [s.copy() for s in states]
    orc.adamw_step(plain, *args)
    for x, y, z, p in zip(a, b, c, plain):
        for f in ("m", "v", "w", "m_scale"):
            assert np.array_equal(getattr(x, f), getattr(y, f)), f
            assert np.array_equal(getattr(z, f), getattr(p, f)), f


def test_per_tensor_terms(orc):
    """Each term is the tensor's squared norm (torch float64), and the norm
    is the root of the terms summed in tensor order."""
    rng = np.random.default_rng(12)
    states = make_states(orc, [1, 500, 7000], rng)
    found, terms = orc.grad_norm_terms(states, 0.5)
    assert found == 0
    for s, t in zip(states, terms):
        ref = torch_norm([s], 0.5) ** 2
        assert abs(t - ref) <= 1e-13 * ref
    total = 0.0
    for t in terms:
        total += t
    assert orc.grad_norm(states, 0.5) == (0, math.sqrt(total))
    states[1].g[3] = 0x7F
    assert orc.grad_norm_terms(states, 0.5)[0] == 1


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_exact_square_sum(orc, fmt):
    """oracle_fp8_sq_sum against the sum of the decoded values' squares in
    Python integers (each decoded value is a multiple of 2^-16), with the
    non-finite codes left out; over pieces the sums add up to the whole's,
    and k^2 * S * 2^-32, rounded once, is the oracle's norm term."""
    rng = np.random.default_rng(44)
    codes = rng.integers(0, 256, 20000).astype(np.uint8)
    vals = orc.fp8_decode(codes, fmt)
    expect = sum(int(abs(float(x)) * 65536) ** 2 for x in vals if np.isfinite(x))
    s = orc.fp8_sq_sum(codes, fmt)
    assert s == expect
    cuts = [0, 5, 9999, 20000]
    assert sum(orc.fp8_sq_sum(codes[a:b], fmt) for a, b in zip(cuts, cuts[1:])) == s
    fin = codes.copy()
    fin[~np.isfinite(vals)] = 0
    st = orc.StepState(fin, 0.25, np.zeros(fin.size, np.uint8), 1.0,
                       np.zeros(fin.size, np.uint16), np.zeros(fin.size, np.uint16),
                       g_fmt=fmt)
    found, terms = orc.grad_norm_terms([st], 0.5)
    assert found == 0
    k = float(np.float32(np.float32(0.5) / np.float32(0.25)))
    assert terms[0] == (k * k) * (float(s) * 2.0 ** -32)
