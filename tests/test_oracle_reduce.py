"""Pins of the oracle's local FP8 reduction (k shards, per-shard scales,
fp32 sum in shard order, then the just-in-time scaled cast): exact round trips,
a two-shard case computed with numpy's float32 arithmetic and torch's float8
types, the float64 error bound for longer sums, the summation order, and the
degenerate cases."""
import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
MAXV = {E4M3: 448.0, E5M2: 57344.0}
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def finite_codes(rng, shape, fmt):
    """Random finite codes of either sign."""
    c = rng.integers(0, 256, shape, dtype=np.uint8)
    if fmt == E4M3:
        bad = (c & 0x7F) == 0x7F
    else:
        bad = (c & 0x7C) == 0x7C
    c[bad] &= 0xF3 if fmt == E5M2 else 0xF7
    return c


def torch_decode(codes, fmt):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(TORCH_FP8[fmt]).float().numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_identical_shards_average_back_to_the_input(orc, fmt, k):
    """k copies of one tensor at one power-of-two scale, averaged with post =
    1/k: every partial sum is exact, so the mean is the input itself and the
    re-encode (a max code is present) gives back the same codes and scale."""
    rng = np.random.default_rng(100 + k)
    c = finite_codes(rng, 3001, fmt)
    c[17] = MAXCODE[fmt]
    s = np.float32(2.0 ** -7)
    shards = np.tile(c, (k, 1))
    codes, amax, scale = orc.reduce_scaled(shards, [s] * k, fmt, fmt, 1.0 / k)
    assert np.array_equal(codes, c)
    assert scale == s
    assert amax == np.float32(MAXV[fmt] / s)


@pytest.mark.parametrize("in_fmt,out_fmt", [(E4M3, E4M3), (E5M2, E4M3),
                                            (E4M3, E5M2), (E5M2, E5M2)])
def test_two_shards_match_numpy_and_torch(orc, in_fmt, out_fmt):
    """Two shards with arbitrary scales: one fp32 product per shard and one
    fp32 sum (numpy float32 arithmetic), then torch's amax, one fp32 division
    and torch's float8 encode."""
    rng = np.random.default_rng(7 + in_fmt * 2 + out_fmt)
    n = 20000
    c = finite_codes(rng, (2, n), in_fmt)
    scales = np.float32(rng.uniform(0.5, 3.0, 2) * 2.0 ** rng.integers(-8, 8, 2))
    post = np.float32(0.5)
    codes, amax, scale = orc.reduce_scaled(c, scales, in_fmt, out_fmt, post)
    r = np.float32(1) / scales
    x0 = torch_decode(c[0], in_fmt) * r[0]
    x1 = torch_decode(c[1], in_fmt) * r[1]
    y = (x0 + x1) * post
    assert y.dtype == np.float32
    t_amax = np.float32(np.abs(y).max())
    assert amax == t_amax
    t_scale = np.float32(MAXV[out_fmt]) / t_amax
    assert scale == t_scale
    ref = torch.from_numpy(y * t_scale).to(TORCH_FP8[out_fmt]).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


@pytest.mark.parametrize("k", [3, 5, 16])
def test_long_sums_within_the_float64_bound(orc, k):
    """Power-of-two shard scales make every term exact, so float64 gives the
    exact sum; the fp32 shard-order sum is within (k - 1) * 2^-24 of the sum
    of magnitudes of it, and each decoded output within half a code spacing
    (plus that bound) of the exact value."""
    rng = np.random.default_rng(40 + k)
    n = 5000
    c = finite_codes(rng, (k, n), E4M3)
    scales = np.float32(2.0 ** rng.integers(-4, 5, k))
    codes, amax, scale = orc.reduce_scaled(c, scales, E4M3, E4M3)
    terms = torch_decode(c, E4M3).astype(np.float64) / scales[:, None].astype(np.float64)
    exact = terms.sum(axis=0)
    err = (k - 1) * 2.0 ** -24 * np.abs(terms).sum(axis=0)
    assert abs(float(amax) - np.abs(exact).max()) <= err.max()
    back = torch_decode(codes, E4M3).astype(np.float64) / np.float64(scale)
    half = np.maximum(np.abs(exact) * 2.0 ** -4, 2.0 ** -10 / np.float64(scale))
    assert np.all(np.abs(back - exact) <= half + err * (1 + 2.0 ** -3) + 1e-30)


def test_sum_is_taken_in_shard_order(orc):
    """E5M2 spans more than fp32's 24 bits, so 57344 + 2^-16 rounds back to
    57344: shard order [L, -L, s] gives s, while [L, s, -L] and [s, L, -L]
    give 0 (adding -L first, or in reverse order, would differ)."""
    L, NL, S, Z = 0x7B, 0xFB, 0x01, 0x00
    shards = np.array([[L, L, S, Z],
                       [NL, S, L, Z],
                       [S, NL, NL, S]], dtype=np.uint8)
    codes, amax, scale = orc.reduce_scaled(shards, [1.0, 1.0, 1.0], E5M2, E4M3)
    assert amax == np.float32(2.0 ** -16)
    assert scale == np.float32(448.0 * 65536.0)
    assert list(codes) == [0x7E, 0x00, 0x00, 0x7E]


def test_opposite_shards_cancel(orc):
    rng = np.random.default_rng(3)
    c = finite_codes(rng, 4096, E4M3)
    shards = np.stack([c, c ^ 0x80])
    codes, amax, scale = orc.reduce_scaled(shards, [3.0, 3.0], E4M3, E4M3)
    assert amax == 0.0 and scale == 1.0
    assert not codes.any()


@pytest.mark.parametrize("p", [2.0 ** -3, 2.0 ** 5])
def test_power_of_two_post_factor_moves_only_amax_and_scale(orc, p):
    rng = np.random.default_rng(5)
    c = finite_codes(rng, (4, 3000), E4M3)
    s = [1.5, 0.75, 2.0, 1.25]
    c0, a0, s0 = orc.reduce_scaled(c, s, E4M3, E4M3, 1.0)
    c1, a1, s1 = orc.reduce_scaled(c, s, E4M3, E4M3, p)
    assert np.array_equal(c0, c1)
    assert a1 == np.float32(a0 * p) and s1 == np.float32(s0 / p)


def test_non_finite_elements(orc):
    # E4M3 NaN code in one shard: that element's sum is NaN
    c = np.array([[0x38, 0x40, 0x30], [0x38, 0x7F, 0x30]], dtype=np.uint8)
    codes, amax, scale = orc.reduce_scaled(c, [1.0, 1.0], E4M3, E4M3)
    assert np.float32(amax).view(np.uint32) == 0x7FC00000 and scale == 1.0
    assert codes[1] == 0x7F
    # E5M2 infinity survives into an E5M2 output; +inf + -inf is NaN
    c = np.array([[0x7C, 0xFC, 0x3C, 0x7C], [0x3C, 0x3C, 0x3C, 0xFC]], dtype=np.uint8)
    codes, amax, scale = orc.reduce_scaled(c, [1.0, 1.0], E5M2, E5M2)
    assert np.isnan(amax) and scale == 1.0
    assert list(codes[:3]) == [0x7C, 0xFC, 0x40] and codes[3] == 0x7F
    c = np.array([[0x7C, 0x3C], [0x3C, 0x3C]], dtype=np.uint8)
    codes, amax, scale = orc.reduce_scaled(c, [1.0, 1.0], E5M2, E4M3)
    assert amax == np.inf and scale == 1.0 and list(codes) == [0x7F, 0x40]


def test_stride_padding_is_not_read(orc):
    rng = np.random.default_rng(8)
    c = finite_codes(rng, (3, 1000), E4M3)
    padded = np.full((3, 1024), 0x7F, dtype=np.uint8)   # NaN codes past numel
    padded[:, :1000] = c
    a = orc.reduce_scaled(c, [1.0, 2.0, 4.0], E4M3, E4M3)
    b = orc.reduce_scaled(padded, [1.0, 2.0, 4.0], E4M3, E4M3, numel=1000)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1] and a[2] == b[2]


def test_empty_tensor(orc):
    codes, amax, scale = orc.reduce_scaled(np.zeros((4, 0), np.uint8), [1.0] * 4,
                                           E4M3, E4M3)
    assert codes.size == 0 and amax == 0.0 and scale == 1.0


def test_bad_arguments_are_refused(orc):
    """Each C entry point refuses a malformed call with -1 before reading
    anything (buffers here are large enough that a call which did read would
    stay in bounds)."""
    import ctypes as C
    L = orc.lib()
    buf = np.zeros(4096, np.uint8)
    scales = np.ones(65, np.float32)
    codes = np.zeros(4096, np.uint8)
    amax = np.zeros(1, np.float32)
    scale = np.zeros(1, np.float32)

    def reduce(numel, stride, k, in_fmt=0, out_fmt=0):
        return L.oracle_reduce_scaled(buf.ctypes.data, numel, stride,
                                      scales.ctypes.data, k, in_fmt, out_fmt,
                                      C.c_float(1.0), codes.ctypes.data,
                                      amax.ctypes.data, scale.ctypes.data)

    assert reduce(64, 64, 2) == 0
    assert reduce(64, 63, 2) == -1           # shards overlap
    assert reduce(64, 64, 0) == -1           # no shard
    assert reduce(32, 32, 65) == -1          # more shards than the limit
    assert reduce(-1, 64, 2) == -1
    assert reduce(64, 64, 2, in_fmt=2) == -1
    assert reduce(64, 64, 2, out_fmt=-1) == -1

    def cast(numel, dtype, fmt=0):
        return L.oracle_cast_scaled(buf.ctypes.data, dtype, numel, fmt,
                                    codes.ctypes.data, amax.ctypes.data,
                                    scale.ctypes.data)

    assert cast(64, 0) == 0 and cast(64, 2) == 0
    assert cast(64, 3) == -1 and cast(64, -1) == -1
    assert cast(64, 0, fmt=2) == -1 and cast(-1, 0) == -1


def test_pieces_with_the_whole_amax_give_the_whole_reduction(orc):
    """The reduction's only per-tensor quantity is the amax of the reduced
    values: pieces (column ranges of every shard) reduced with the largest
    of the pieces' own amax give the whole tensor's codes and scale."""
    rng = np.random.default_rng(43)
    k, n = 4, 5000
    shards = rng.integers(0, 256, (k, n)).astype(np.uint8)
    shards[(shards & 0x7F) == 0x7F] = 0x11            # finite codes only
    scales = (2.0 ** rng.integers(-6, 7, k)).astype(np.float32)
    for out_fmt in (orc.E4M3, orc.E5M2):
        whole, amax, scale = orc.reduce_scaled(shards, scales, orc.E4M3, out_fmt,
                                               1.0 / k)
        cuts = [0, 1, 700, 701, 4096, n]
        own = [orc.reduce_scaled(np.ascontiguousarray(shards[:, a:b]), scales,
                                 orc.E4M3, out_fmt, 1.0 / k)[1]
               for a, b in zip(cuts, cuts[1:])]
        big = np.float32(max(own))
        assert big == amax
        for a, b in zip(cuts, cuts[1:]):
            c, sc = orc.reduce_scaled_given(np.ascontiguousarray(shards[:, a:b]),
                                            scales, orc.E4M3, out_fmt, 1.0 / k, big)
            assert sc == scale
            assert np.array_equal(c, whole[a:b])
