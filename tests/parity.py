"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (fixed by the library's specification):
* amax, scales and found_inf: bit-exact;
* FP8 codes: at most 1 code apart, at least 99.9% identical;
* FP16 second moment and weights: at most 1 ulp apart;
* FP16 master weights (O3): within 2e-3 relative.
NaN codes / NaN halves must sit at the same positions, and E5M2 infinity
codes must be identical.
"""
import numpy as np
import torch

E4M3, E5M2 = 0, 1
CODE_MIN_EXACT = 0.999
MASTER_REL = 2e-3


def to_np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.uint8, copy=False)


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_np_u16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(
        torch.float16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def nan_code(c: np.ndarray, fmt: int) -> np.ndarray:
    c = c.astype(np.int32)
    if fmt == E4M3:
        return (c & 0x7F) == 0x7F
    return ((c & 0x7C) == 0x7C) & ((c & 0x03) != 0)


def inf_code(c: np.ndarray, fmt: int) -> np.ndarray:
    """Infinity codes (E5M2 only; E4M3 has none)."""
    c = c.astype(np.int32)
    if fmt == E4M3:
        return np.zeros(c.shape, bool)
    return (c & 0x7F) == 0x7C


def _ord(x: np.ndarray, sign_bit: int) -> np.ndarray:
    x = x.astype(np.int64)
    mag = x & (sign_bit - 1)
    return np.where(x & sign_bit, -mag, mag)


def check_codes(got, ref, fmt=E4M3, name="codes", min_exact=CODE_MIN_EXACT):
    got = np.asarray(got, np.uint8).ravel()
    ref = np.asarray(ref, np.uint8).ravel()
    assert got.shape == ref.shape, name
    if ref.size == 0:
        return 1.0
    nan = nan_code(ref, fmt)
    assert np.array_equal(nan, nan_code(got, fmt)), f"{name}: NaN codes differ"
    # E5M2 infinities come only from infinite values (finite ones saturate),
    # so they are no rounding neighbour of the largest finite code
    inf = inf_code(ref, fmt)
    assert np.array_equal(inf, inf_code(got, fmt)) and np.array_equal(
        got[inf], ref[inf]), f"{name}: infinity codes differ"
    d = np.abs(_ord(got, 0x80) - _ord(ref, 0x80))[~(nan | inf)]
    assert d.size == 0 or d.max() <= 1, (
        f"{name}: codes {int(d.max())} apart at {np.flatnonzero(d > 1)[:5]}")
    exact = float(np.mean(got == ref))
    assert exact >= min_exact, f"{name}: only {exact:.5f} identical"
    return exact


def check_f16(got, ref, name="f16", max_ulp=1):
    got = np.asarray(got, np.uint16).ravel()
    ref = np.asarray(ref, np.uint16).ravel()
    assert got.shape == ref.shape, name
    if ref.size == 0:
        return 1.0
    isnan = lambda h: ((h & 0x7C00) == 0x7C00) & ((h & 0x03FF) != 0)
    nan = isnan(ref)
    assert np.array_equal(nan, isnan(got)), f"{name}: NaN positions differ"
    d = np.abs(_ord(got, 0x8000) - _ord(ref, 0x8000))[~nan]
    assert d.size == 0 or d.max() <= max_ulp, (
        f"{name}: {int(d.max())} ulp apart at {np.flatnonzero(d > max_ulp)[:5]}")
    return float(np.mean(got == ref))


def check_master(got, ref, name="master", rel=MASTER_REL):
    g = np.asarray(got, np.uint16).view(np.float16).astype(np.float64).ravel()
    r = np.asarray(ref, np.uint16).view(np.float16).astype(np.float64).ravel()
    both_nan = np.isnan(g) & np.isnan(r)
    ok = both_nan | (np.abs(g - r) <= rel * np.abs(r)) | (g == r)
    assert ok.all(), f"{name}: relative error above {rel} at {np.flatnonzero(~ok)[:5]}"
    return float(np.mean(np.asarray(got).ravel() == np.asarray(ref).ravel()))


def check_f32_exact(got, ref, name="scalar"):
    g = np.asarray(got, np.float32).ravel()
    r = np.asarray(ref, np.float32).ravel()
    assert g.shape == r.shape, name
    nan = np.isnan(r)
    assert np.array_equal(nan, np.isnan(g)), f"{name}: NaN differs"
    gb, rb = g.view(np.uint32)[~nan], r.view(np.uint32)[~nan]
    bad = np.flatnonzero(gb != rb)
    assert bad.size == 0, f"{name}: not bit-exact at {bad[:5]}: {g[~nan][bad[:5]]} vs {r[~nan][bad[:5]]}"
