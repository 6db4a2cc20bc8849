"""Pins of the oracle's FP8 / FP16 / BF16 codecs against definitions and
library routines that share nothing with it (torch's float8 and bfloat16
types, numpy's float16, a brute-force nearest-value search)."""
import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
MAXV = {E4M3: 448.0, E5M2: 57344.0}
MBITS = {E4M3: 3, E5M2: 2}


def torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.uint8)
    return codes.view(TORCH_FP8[fmt]).float().numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_all_codes_matches_torch(orc, fmt):
    ours = orc.fp8_decode(np.arange(256, dtype=np.uint8), fmt)
    ref = torch_decode(fmt)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    # sign of zero is kept
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0])


def test_format_maxima_and_special_codes(orc):
    d4 = orc.fp8_decode(np.arange(256, dtype=np.uint8), E4M3)
    d5 = orc.fp8_decode(np.arange(256, dtype=np.uint8), E5M2)
    assert np.nanmax(d4) == 448.0 and d4[0x7E] == 448.0 and d4[0xFE] == -448.0
    assert np.isnan(d4[0x7F]) and np.isnan(d4[0xFF])
    assert np.isnan(d4).sum() == 2               # E4M3 has no infinity
    assert np.nanmax(d5[np.isfinite(d5)]) == 57344.0 and d5[0x7B] == 57344.0
    assert d5[0x7C] == np.inf and d5[0xFC] == -np.inf
    assert np.isnan(d5).sum() == 6
    assert orc.fp8_max(E4M3) == 448.0 and orc.fp8_max(E5M2) == 57344.0
    # smallest subnormals
    assert d4[1] == 2.0 ** -9 and d5[1] == 2.0 ** -16


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_round_trip_every_code(orc, fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.fp8_decode(codes, fmt)
    keep = ~np.isnan(vals)
    back = orc.fp8_encode(vals[keep], fmt)
    assert np.array_equal(back, codes[keep])


def brute_force_encode(x, fmt):
    """Nearest finite code by exhaustive search over the 256 codes; ties go
    to the even code; magnitudes beyond the maximum saturate."""
    vals = torch_decode(fmt).astype(np.float64)
    codes = np.arange(256)
    pos = (codes < 0x80) & np.isfinite(vals)
    pv, pc = vals[pos], codes[pos]
    order = np.argsort(pv)
    pv, pc = pv[order], pc[order]
    a = np.abs(x.astype(np.float64))
    idx = np.clip(np.searchsorted(pv, a), 1, len(pv) - 1)
    lo, hi = pv[idx - 1], pv[idx]
    dlo, dhi = a - lo, hi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (pc[idx] % 2 == 0))
    c = np.where(pick_hi, pc[idx], pc[idx - 1])
    c = np.where(a >= pv[-1], pc[-1], c)
    c = np.where(a <= pv[0], pc[0], c)
    return (c | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def probe_values(fmt, rng):
    """Random values across the whole range plus every midpoint between
    adjacent codes and its two fp32 neighbours."""
    vals = np.sort(torch_decode(fmt)[:0x80])
    vals = vals[np.isfinite(vals)].astype(np.float64)
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(0))])
    expo = rng.uniform(-24, 20, 200000)
    rnd = (2.0 ** expo * rng.uniform(1, 2, expo.size)).astype(np.float32)
    big = np.array([MAXV[fmt], MAXV[fmt] * 1.03, MAXV[fmt] * 1.2, 1e30,
                    3.4e38], dtype=np.float32)
    tiny = np.array([0.0, 1e-45, 1e-38, 2.0 ** -20], dtype=np.float32)
    x = np.concatenate([near, rnd, big, tiny, vals.astype(np.float32)])
    return np.concatenate([x, -x]).astype(np.float32)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_is_nearest_even_saturating(orc, fmt):
    rng = np.random.default_rng(11 + fmt)
    x = probe_values(fmt, rng)
    assert np.array_equal(orc.fp8_encode(x, fmt), brute_force_encode(x, fmt))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_in_range(orc, fmt):
    rng = np.random.default_rng(21 + fmt)
    x = probe_values(fmt, rng)
    x = x[np.abs(x) <= MAXV[fmt]]
    ref = torch.from_numpy(x).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(orc.fp8_encode(x, fmt), ref)


def test_encode_non_finite(orc):
    x = np.array([np.nan, np.inf, -np.inf], dtype=np.float32)
    assert list(orc.fp8_encode(x, E4M3)) == [0x7F, 0x7F, 0x7F]
    assert list(orc.fp8_encode(x, E5M2)) == [0x7F, 0x7C, 0xFC]


def test_f16_to_f32_exhaustive(orc):
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_matches_numpy(orc):
    rng = np.random.default_rng(5)
    # every fp32 pattern whose low 9 mantissa bits are one of a few values,
    # across all exponents (2^23 * 6 patterns), plus random patterns
    hi = np.arange(1 << 23, dtype=np.uint32) << 9
    parts = [hi | np.uint32(k) for k in (0, 1, 0xFF, 0x100, 0x101, 0x1FF)]
    parts.append(rng.integers(0, 1 << 32, 4_000_000, dtype=np.uint64)
                 .astype(np.uint32))
    bits = np.concatenate(parts)
    x = bits.view(np.float32)
    ours = orc.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all((ours[nan] & 0x7C00) == 0x7C00) and np.all(ours[nan] & 0x3FF)


def test_bf16_widen_matches_torch(orc):
    import ctypes
    L = orc.lib()
    h = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    ours = np.array([L.oracle_bf16_to_f32(int(v)) for v in h], np.float32)
    ref = torch.from_numpy(h.astype(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
