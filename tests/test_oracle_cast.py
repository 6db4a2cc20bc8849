"""Pins of the oracle's scaled FP8 cast: invariants that any correct
just-in-time fp8_max/amax cast satisfies, a library comparison of the
encoding step, and the degenerate cases."""
import numpy as np
import pytest
import torch

import synth

E4M3, E5M2 = 0, 1
F32, BF16, F16 = 0, 1, 2
MAXV = {E4M3: 448.0, E5M2: 57344.0}
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def bits16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def as_input(x, dtype):
    t = torch.from_numpy(np.asarray(x, np.float32))
    if dtype == F32:
        return t.numpy(), t.numpy()
    td = t.to(torch.bfloat16 if dtype == BF16 else torch.float16)
    return bits16(td), td.float().numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_all_zero_tensor_keeps_scale_finite(orc, fmt):
    codes, amax, scale = orc.cast_scaled(np.zeros(1000, np.float32), F32, fmt)
    assert amax == 0.0 and scale == 1.0
    assert not codes.any()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_cast_matches_torch_float8(orc, fmt, dtype):
    rng = np.random.default_rng(fmt * 3 + dtype)
    x = (rng.standard_normal(5001) * 3e-3).astype(np.float32)
    src, xf = as_input(x, dtype)
    codes, amax, scale = orc.cast_scaled(src, dtype, fmt)
    # amax by torch, the scale as one fp32 division, encoding by torch's type
    t_amax = torch.from_numpy(xf).abs().max()
    assert amax == t_amax.item()
    t_scale = (torch.tensor(MAXV[fmt], dtype=torch.float32) / t_amax)
    assert scale == t_scale.item()
    t_codes = (torch.from_numpy(xf) * t_scale).to(TORCH_FP8[fmt]).view(torch.uint8)
    assert np.array_equal(codes, t_codes.numpy())


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_power_of_two_rescale_leaves_codes_unchanged(orc, fmt):
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(4096) * 0.1).astype(np.float32)
    c0, a0, s0 = orc.cast_scaled(x, F32, fmt)
    for k in (-20, -3, 5, 30):
        ck, ak, sk = orc.cast_scaled(np.ldexp(x, k).astype(np.float32), F32, fmt)
        assert np.array_equal(ck, c0)
        assert ak == np.float32(np.ldexp(a0, k))
        assert sk == np.float32(np.ldexp(s0, -k))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_largest_element_maps_to_max_code(orc, fmt):
    rng = np.random.default_rng(9)
    for n in (1, 2, 17, 1000):
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        codes, amax, scale = orc.cast_scaled(x, F32, fmt)
        i = int(np.argmax(np.abs(x)))
        assert amax == np.abs(x)[i]
        assert (codes[i] & 0x7F) == MAXCODE[fmt]
        assert (codes & 0x7F).max() == MAXCODE[fmt]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quantisation_error_within_half_spacing(orc, fmt):
    """Decoded / scale is within half a code spacing of x (relative 2^-(m+1)
    for normal codes, absolute half the subnormal step below)."""
    rng = np.random.default_rng(13)
    x = (rng.standard_normal(20000) * 1e-2).astype(np.float32)
    codes, amax, scale = orc.cast_scaled(x, F32, fmt)
    t = x.astype(np.float64) * np.float64(scale)
    back = orc.fp8_decode(codes, fmt).astype(np.float64)
    mbits = {E4M3: 3, E5M2: 2}[fmt]
    sub_step = {E4M3: 2.0 ** -9, E5M2: 2.0 ** -16}[fmt]
    bound = np.maximum(np.abs(t) * 2.0 ** -(mbits + 1), sub_step / 2)
    assert np.all(np.abs(back - t) <= bound * (1 + 1e-6))


def test_non_finite_inputs(orc):
    x = np.array([1.0, -2.0, np.inf, 0.5], np.float32)
    c4, a4, s4 = orc.cast_scaled(x, F32, E4M3)
    assert a4 == np.inf and s4 == 1.0
    assert list(c4) == [orc.fp8_encode(np.float32([1.0]), E4M3)[0],
                        orc.fp8_encode(np.float32([-2.0]), E4M3)[0], 0x7F,
                        orc.fp8_encode(np.float32([0.5]), E4M3)[0]]
    c5, a5, s5 = orc.cast_scaled(-x, F32, E5M2)
    assert a5 == np.inf and s5 == 1.0 and c5[2] == 0xFC
    y = np.array([1.0, np.nan, np.inf], np.float32)
    c, a, s = orc.cast_scaled(y, F32, E4M3)
    assert np.isnan(a) and s == 1.0
    assert np.float32(a).view(np.uint32) == 0x7FC00000
    assert list(c[1:]) == [0x7F, 0x7F]


def test_empty_tensor(orc):
    codes, amax, scale = orc.cast_scaled(np.zeros(0, np.float32), F32, E4M3)
    assert codes.size == 0 and amax == 0.0 and scale == 1.0


def test_tiny_amax_keeps_scale_finite(orc):
    x = np.array([1e-45, -1e-45], np.float32)   # 448 / 1e-45 overflows fp32
    codes, amax, scale = orc.cast_scaled(x, F32, E4M3)
    assert amax == np.float32(1e-45) and scale == 1.0


def test_synthetic_cast_list_small(orc):
    """The GPT-shaped cast workload at a reduced size: every tensor's largest
    element reaches the max code and the per-tensor scale is finite."""
    wl = synth.gpt2_cast(n_layer=1, d=64, ffn=256, vocab=300, ctx=32)
    for i, g in enumerate(wl.grads(step=1)):
        codes, amax, scale = orc.cast_scaled(bits16(g), BF16, E4M3)
        assert np.isfinite(scale) and scale > 0
        assert (codes & 0x7F).max() == 0x7E
