"""The device FP8 encoders against the oracle's encoder on every input, bit
for bit (no tolerance).

Formats: E4M3 and E5M2 as the TransformerEngine issue #131 ("FP8 questions")
names them, with the OCP bit layouts; the encode rounds to nearest, ties to
even, and saturates finite overflow.  A cast multiplies by its per-tensor
scale before it encodes, so the tests pin the scale to exactly 1.0 (x * 1.0
is x for every float, subnormals included) and the codes are then the pure
encode of each input:
  * every one of the 2^32 fp32 bit patterns through fp8_cast_scaled's checked
    path: the tensor also holds a NaN, so its amax is not finite, the scale
    falls back to 1.0, and every element takes the encoder that selects the
    non-finite codes explicitly (infinities, NaNs, saturation above max);
  * every fp32 pattern with |x| <= fp8_max through the plain vector path: the
    tensor also holds fp8_max itself, so amax = fp8_max and the scale is
    fp8_max / fp8_max = 1.0;
  * every BF16 and FP16 pattern, the same two ways, through the cast's
    16-bit loads;
  * every FP16 master with |x| <= 448 through the O3 weight copy (a step with
    lr = 0 and zero gradients keeps the master, and one master at 448 makes
    its scale 1.0).
The oracle's codes come from oracle_fp8_encode_array, run on the host's
cores in threads (ctypes releases the GIL)."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from harness import GpuState

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2
FMT_NAME = {E4M3: "e4m3", E5M2: "e5m2"}
MAX_BITS = {E4M3: 0x43E00000, E5M2: 0x47600000}   # 448.0, 57344.0
SLICE = 1 << 28
THREADS = max(1, min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def bo():
    import bit_optimizer_gb300 as bo
    return bo


@pytest.fixture(scope="module")
def pool():
    with cf.ThreadPoolExecutor(THREADS) as ex:
        yield ex


def oracle_codes(pool, x: np.ndarray, fmt: int) -> np.ndarray:
    out = np.empty(x.size, np.uint8)
    lib = oracle.lib()
    step = (x.size + THREADS - 1) // THREADS

    def part(i):
        a, o = x[i * step:(i + 1) * step], out[i * step:(i + 1) * step]
        if a.size:
            lib.oracle_fp8_encode_array(a.ctypes.data, a.size, fmt, o.ctypes.data)

    list(pool.map(part, range(THREADS)))
    return out


def device_cast(bo, host: np.ndarray, sentinel, dtype, fmt):
    """Casts host's values followed by one sentinel element; returns the
    codes of host's values, amax and scale."""
    n = host.size
    raw = torch.from_numpy(host.view({torch.float32: np.int32,
                                      torch.bfloat16: np.int16,
                                      torch.float16: np.int16}[dtype]))
    src = torch.empty(n + 1, dtype=dtype, device="cuda")
    src[:n].view(raw.dtype).copy_(raw)
    src[n] = sentinel
    codes, amax, scale = bo.fp8_cast_scaled([src], FMT_NAME[fmt])
    return codes[0][:n].cpu().numpy(), amax[0].item(), scale[0].item()


def assert_same(got, ref, what, x):
    bad = np.flatnonzero(got != ref)
    if bad.size:
        i = bad[:8]
        raise AssertionError(
            f"{what}: {bad.size} codes differ; first inputs "
            f"{[hex(v) for v in x.view(np.uint32 if x.itemsize == 4 else np.uint16)[i]]} "
            f"device {[hex(v) for v in got[i]]} oracle {[hex(v) for v in ref[i]]}")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_every_fp32_pattern(bo, pool, fmt):
    top = MAX_BITS[fmt]
    checked = plain = 0
    for lo in range(0, 1 << 32, SLICE):
        bits = np.arange(SLICE, dtype=np.uint32) + np.uint32(lo)
        x = bits.view(np.float32)
        ref = oracle_codes(pool, x, fmt)
        got, amax, scale = device_cast(bo, x, float("nan"), torch.float32, fmt)
        assert np.isnan(amax) and scale == 1.0
        assert_same(got, ref, f"checked path, slice {lo:#x}", x)
        checked += x.size
        # the part of the slice with |x| <= fp8_max: a contiguous range
        mag_lo = lo & 0x7FFFFFFF
        if mag_lo <= top:
            hi = min(SLICE, top - mag_lo + 1)
            got, amax, scale = device_cast(bo, x[:hi], float(np.float32(
                np.uint32(top).view(np.float32))), torch.float32, fmt)
            assert scale == 1.0
            assert_same(got, ref[:hi], f"vector path, slice {lo:#x}", x[:hi])
            plain += hi
    assert checked == 1 << 32
    assert plain == 2 * (top + 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_every_16_bit_pattern(bo, pool, dtype, fmt):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(dtype)
    x = t.float().numpy()                    # exact widening
    ref = oracle_codes(pool, x, fmt)
    got, amax, scale = device_cast(bo, bits, float("nan"), dtype, fmt)
    assert np.isnan(amax) and scale == 1.0
    assert_same(got, ref, "checked path", x)
    fmax = float(np.uint32(MAX_BITS[fmt]).view(np.float32))
    keep = np.abs(x) <= fmax                 # NaNs drop out
    got, amax, scale = device_cast(bo, bits[keep], fmax, dtype, fmt)
    assert scale == 1.0
    assert_same(got, ref[keep], "vector path", x[keep])


def test_every_fp16_master_in_the_o3_copy(bo, pool):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = oracle.f16_to_f32(h)
    h = h[np.abs(x) <= 448.0]
    h = np.concatenate([h, np.array([0x5F00], np.uint16)])   # 448.0
    x = oracle.f16_to_f32(h)
    n = h.size
    st = oracle.StepState(np.zeros(n, np.uint8), 1.0, np.zeros(n, np.uint8), 1.0,
                          np.zeros(n, np.uint16), h, o3=True)
    gpu = GpuState([st])
    assert gpu.plan(0.0, 0.9, 0.999, 1e-8, 0.0, 1, 1.0) == 0
    assert np.array_equal(gpu.w[0].view(torch.int16).cpu().numpy().view(np.uint16), h)
    assert gpu.w8_scale.item() == 1.0 and gpu.w8_amax.item() == 448.0
    got = gpu.w8[0].cpu().numpy()
    assert_same(got, oracle_codes(pool, x, E4M3), "O3 weight copy", x)
