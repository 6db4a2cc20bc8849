"""Bounds of every write the library makes, checked without compute-sanitizer.

Each call gets one device allocation (an arena) filled with seeded random
bytes.  Every caller buffer of the call (sources, codes, moments, weights,
weight copies, shards, and every per-tensor scalar on its own) is carved out
of it between 256-byte bands, at aligned and unaligned starts.  After the
call, every byte outside the call's output buffers must read as before: the
bands (a store past a buffer's end or before its start), the gaps, and the
input buffers themselves (a store into an input).  Tensor sizes 0, 1, 7, 8,
9, 2047, 2049 and 32769 (vector groups, ragged tails, a tile past the tiny
lists' 2048-element chunks), alone and with a 100003-element tensor that moves
the list onto 32768-element chunks.  The outputs are compared with the
oracle as well, at the step's tolerances."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from harness import host_src
from parity import (check_codes, check_f16, check_f32_exact, check_master,
                    to_np_u16, to_np_u8)

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2
PAD = 256
SIZES = [1, 7, 8, 9, 2047, 2049, 32769, 0]
U8_SKEW = [0, 1, 3, 5, 0, 7, 2, 1]       # bytes past a 256-byte boundary
H_SKEW = [0, 2, 6, 0, 4, 0, 2, 2]        # 16-bit buffers
F_SKEW = [0, 4, 8, 12, 0, 4, 0, 4]       # fp32 buffers and scalars
LISTS = {"tiny": (SIZES, 0), "chunked": (SIZES + [100003], 3)}
HP = (1e-3, 0.9, 0.999, 1e-8, 0.01, 3, 0.5)   # lr, b1, b2, eps, wd, step, ils


@pytest.fixture(scope="module")
def lib():
    import bit_optimizer_gb300 as bo
    from bit_optimizer_gb300 import _lib
    return bo.load(), _lib


def sizes_of(name):
    sizes, extra_skew = LISTS[name]
    u8 = U8_SKEW + [extra_skew]
    h = H_SKEW + [2 * (extra_skew % 4)]
    f = F_SKEW + [4 * (extra_skew % 4)]
    return sizes, u8, h, f


class Arena:
    """Device buffers carved from one allocation between canary bands."""

    def __init__(self, seed, cap=4 << 20):
        self.init = np.random.default_rng(seed).integers(0, 256, cap, dtype=np.uint8)
        self.buf = torch.from_numpy(self.init.copy()).cuda()
        self.cap, self.used = cap, 0
        self.out = np.zeros(cap, bool)        # bytes the call may write
        self.expect = None

    def take(self, nbytes, skew=0, dtype=torch.uint8, out=False):
        start = -(-(self.used + PAD) // 256) * 256 + skew
        end = start + nbytes
        assert end + PAD <= self.cap, "arena too small"
        self.used = end + PAD
        if out:
            self.out[start:end] = True
        return self.buf[start:end].view(dtype)

    def scalar(self, value, skew=0, out=True, dtype=torch.float32):
        t = self.take(4, skew, dtype, out)
        t.fill_(value)
        return t

    def seal(self):
        """Inputs are in place: record what every byte must keep."""
        torch.cuda.synchronize()
        self.expect = self.buf.cpu().numpy().copy()

    def check(self, what):
        torch.cuda.synchronize()
        host = self.buf.cpu().numpy()
        bad = np.flatnonzero((host != self.expect) & ~self.out)
        assert bad.size == 0, (
            f"{what}: {bad.size} bytes outside the output buffers changed, "
            f"first at arena offsets {bad[:8].tolist()}")


def ptr(t):
    return t.data_ptr()


# ------------------------------------------------------------------ cast

DTYPES = [torch.float32, torch.bfloat16, torch.float16]
DT_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


def cast_case(arena, lib_, name, rng, dtype_of=None):
    """Sources (inputs) and codes, amax, scale (outputs) of one cast list."""
    _, L = lib_
    sizes, u8, h, f = sizes_of(name)
    host, codes, amax, scale = [], [], [], []
    items = (L.CastItem * len(sizes))()
    for i, n in enumerate(sizes):
        dt = DTYPES[i % 3] if dtype_of is None else dtype_of
        x = torch.from_numpy((rng.standard_normal(n) *
                              10.0 ** rng.uniform(-4, 1)).astype(np.float32)).to(dt)
        esz = 4 if dt == torch.float32 else 2
        src = arena.take(n * esz, f[i] if esz == 4 else h[i], dt)
        src.copy_(x)
        host.append(x)
        codes.append(arena.take(n, u8[i], out=True))
        amax.append(arena.scalar(-7.0, f[i]))
        scale.append(arena.scalar(-7.0, f[i]))
        it = items[i]
        it.src, it.numel, it.dtype = ptr(src), n, DT_CODE[dt]
        it.codes, it.amax, it.scale = ptr(codes[i]), ptr(amax[i]), ptr(scale[i])
    return items, host, codes, amax, scale


def check_cast(host, codes, amax, scale, fmt):
    ref_codes, ref_amax, ref_scale = [], [], []
    for x in host:
        a, dt = host_src(x)
        c, am, sc = oracle.cast_scaled(a, dt, fmt)
        ref_codes.append(c)
        ref_amax.append(am)
        ref_scale.append(sc)
    check_f32_exact([a.item() for a in amax], ref_amax, "amax")
    check_f32_exact([s.item() for s in scale], ref_scale, "scale")
    for i, (c, r) in enumerate(zip(codes, ref_codes)):
        check_codes(to_np_u8(c), r, fmt, name=f"codes[{i}]")
    return ref_codes, ref_scale


@pytest.mark.parametrize("name", list(LISTS))
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("entry", ["fp8_cast_scaled", "fp8_cast_scaled_noalloc"])
def test_cast_stays_in_bounds(lib, name, fmt, entry):
    Lib, L = lib
    arena = Arena(1)
    rng = np.random.default_rng(2)
    items, host, codes, amax, scale = cast_case(arena, lib, name, rng)
    arena.seal()
    assert getattr(Lib, entry)(items, len(host), fmt, None) == 0
    arena.check(entry)
    check_cast(host, codes, amax, scale, fmt)


# ------------------------------------------------------------------ step

def oracle_states(name, rng, fmt=E4M3, o3=False, scaled_v=False):
    sizes, _, _, _ = sizes_of(name)
    out = []
    for n in sizes:
        top = 0x7F if fmt == E4M3 else 0x7C
        g = (rng.integers(0, top, n) | (rng.integers(0, 2, n) << 7)).astype(np.uint8)
        m = (rng.integers(0, 0x7F, n) | (rng.integers(0, 2, n) << 7)).astype(np.uint8)
        vv = np.abs(rng.standard_normal(n)).astype(np.float32)
        v = oracle.f32_to_f16(vv * (1000.0 if scaled_v else 1e-4))
        w = oracle.f32_to_f16((rng.standard_normal(n) * 0.02).astype(np.float32))
        out.append(oracle.StepState(g, 2.0 ** -int(rng.integers(0, 12)), m,
                                    2.0 ** int(rng.integers(6, 14)), v, w,
                                    g_fmt=fmt, o3=o3, scaled_v=scaled_v,
                                    v_bound=1e-6))
    return out


class DeviceStep:
    """Step records over arena buffers holding the oracle states' values."""

    def __init__(self, arena, lib_, name, states, grads_from=None):
        _, L = lib_
        sizes, u8, h, f = sizes_of(name)
        self.states = states
        self.params = (L.Param * len(sizes))()
        self.bufs = []
        for i, (n, st) in enumerate(zip(sizes, states)):
            b = {}
            if grads_from is None:
                b["g"] = arena.take(n, u8[i])
                b["g"].copy_(torch.from_numpy(st.g))
                b["g_scale"] = arena.scalar(st.g_scale, f[i], out=False)
            else:                                   # the cast's outputs
                b["g"], b["g_scale"] = grads_from[0][i], grads_from[1][i]
            b["m"] = arena.take(n, u8[(i + 1) % len(u8)], out=True)
            b["m"].copy_(torch.from_numpy(st.m))
            b["m_scale"] = arena.scalar(float(st.m_scale[0]), f[i])
            for k, skew in (("v", h[i]), ("w", h[(i + 3) % len(h)])):
                b[k] = arena.take(2 * n, skew, torch.int16, out=True)
                b[k].copy_(torch.from_numpy(getattr(st, k).view(np.int16)))
            p = self.params[i]
            p.numel, p.g_fmt = n, st.g_fmt
            p.g, p.g_scale = ptr(b["g"]), ptr(b["g_scale"])
            p.m, p.m_scale, p.v, p.w = (ptr(b["m"]), ptr(b["m_scale"]), ptr(b["v"]),
                                        ptr(b["w"]))
            if st.w8 is not None:
                b["w8"] = arena.take(n, u8[(i + 2) % len(u8)], out=True)
                b["w8_scale"] = arena.scalar(-7.0, f[i])
                b["w8_amax"] = arena.scalar(-7.0, f[i])
                p.w8, p.w8_scale, p.w8_amax = (ptr(b["w8"]), ptr(b["w8_scale"]),
                                               ptr(b["w8_amax"]))
            if st.v_bound is not None:
                b["v_bound"] = arena.scalar(float(st.v_bound[0]), f[i])
                p.v_bound = ptr(b["v_bound"])
            self.bufs.append(b)

    def compare(self, ref):
        for i, (b, s) in enumerate(zip(self.bufs, ref)):
            check_f32_exact([b["m_scale"].item()], s.m_scale, f"m_scale[{i}]")
            check_codes(to_np_u8(b["m"]), s.m, name=f"m[{i}]")
            check_f16(to_np_u16(b["v"].view(torch.float16)), s.v, name=f"v[{i}]")
            w = to_np_u16(b["w"].view(torch.float16))
            if s.w8 is not None:
                check_master(w, s.w, name=f"master[{i}]")
                check_codes(to_np_u8(b["w8"]), s.w8, name=f"w8[{i}]")
                check_f32_exact([b["w8_scale"].item()], s.w8_scale, f"w8_scale[{i}]")
                check_f32_exact([b["w8_amax"].item()], s.w8_amax, f"w8_amax[{i}]")
            check_f16(w, s.w, name=f"w[{i}]")
            if s.v_bound is not None:
                check_f32_exact([b["v_bound"].item()], s.v_bound, f"v_bound[{i}]")


STEP_CASES = [  # (level O3, scaled second moment, Adam with L2 decay, format)
    (False, False, False, E4M3), (True, False, False, E5M2),
    (False, True, True, E4M3), (True, True, False, E4M3)]


@pytest.mark.parametrize("name", list(LISTS))
@pytest.mark.parametrize("o3,scaled_v,l2,fmt", STEP_CASES)
def test_step_stays_in_bounds(lib, name, o3, scaled_v, l2, fmt):
    Lib, _ = lib
    arena = Arena(3)
    states = oracle_states(name, np.random.default_rng(4), fmt, o3, scaled_v)
    dev = DeviceStep(arena, lib, name, states)
    found_dev = arena.scalar(7, 0, dtype=torch.int32)
    arena.seal()
    found = C.c_int(-1)
    fn = Lib.fp8_adam_step if l2 else Lib.fp8_adamw_step
    assert fn(dev.params, len(states), *HP, C.byref(found), ptr(found_dev), None) == 0
    arena.check("step")
    ref = [s.copy() for s in states]
    assert oracle.adamw_step(ref, *HP, l2=l2) == 0 == found.value == found_dev.item()
    dev.compare(ref)


@pytest.mark.parametrize("name", list(LISTS))
@pytest.mark.parametrize("o3,l2", [(False, False), (True, True)])
def test_clipped_step_stays_in_bounds(lib, name, o3, l2):
    Lib, _ = lib
    arena = Arena(5)
    states = oracle_states(name, np.random.default_rng(6), E4M3, o3)
    dev = DeviceStep(arena, lib, name, states)
    norm_dev = arena.scalar(-7.0, 4)
    found_dev = arena.scalar(7, 8, dtype=torch.int32)
    arena.seal()
    norm, found = C.c_double(0.0), C.c_int(-1)
    assert Lib.fp8_adam_step_clipped(dev.params, len(states), *HP, int(l2), 1.0,
                                     C.byref(norm), ptr(norm_dev), C.byref(found),
                                     ptr(found_dev), None) == 0
    arena.check("clipped step")
    ref = [s.copy() for s in states]
    f_ref, n_ref = oracle.adam_step_clipped(ref, *HP, 1.0, l2=l2)
    assert f_ref == found.value == found_dev.item() == 0 and norm.value == n_ref
    dev.compare(ref)


@pytest.mark.parametrize("name", list(LISTS))
@pytest.mark.parametrize("clip", [None, 0.5, "l2"])
def test_fused_cast_step_stays_in_bounds(lib, name, clip):
    """fp8_cast_adamw_step (clip None), fp8_cast_adam_step_clipped, and the
    latter for Adam with L2 decay with no norm asked for ("l2": the fused
    passes, the first one reading the weights): the cast's codes and scales
    are outputs the step then reads."""
    Lib, _ = lib
    arena = Arena(7)
    rng = np.random.default_rng(8)
    items, host, codes, amax, scale = cast_case(arena, lib, name, rng,
                                                dtype_of=torch.bfloat16)
    states = oracle_states(name, np.random.default_rng(9), E4M3, o3=True)
    dev = DeviceStep(arena, lib, name, states, grads_from=(codes, scale))
    found_dev = arena.scalar(7, 0, dtype=torch.int32)
    norm_dev = arena.scalar(-7.0, 4)
    arena.seal()
    found, norm = C.c_int(-1), C.c_double(0.0)
    n = len(states)
    if clip is None:
        rc = Lib.fp8_cast_adamw_step(items, dev.params, n, E4M3, *HP, C.byref(found),
                                     ptr(found_dev), None)
    elif clip == "l2":
        rc = Lib.fp8_cast_adam_step_clipped(items, dev.params, n, E4M3, *HP, 1, 0.0,
                                            None, None, C.byref(found),
                                            ptr(found_dev), None)
    else:
        rc = Lib.fp8_cast_adam_step_clipped(items, dev.params, n, E4M3, *HP, 0, clip,
                                            C.byref(norm), ptr(norm_dev),
                                            C.byref(found), ptr(found_dev), None)
    assert rc == 0
    arena.check("fused cast + step")
    ref_codes, ref_scale = check_cast(host, codes, amax, scale, E4M3)
    ref = [s.copy() for s in states]
    for s, c, sc in zip(ref, ref_codes, ref_scale):
        s.g, s.g_scale = np.ascontiguousarray(c), float(sc)
    if clip is None:
        assert oracle.adamw_step(ref, *HP) == 0
    elif clip == "l2":
        assert oracle.adamw_step(ref, *HP, l2=True) == 0
        assert norm_dev.item() == -7.0   # no norm asked for: left as it was
    else:
        f_ref, n_ref = oracle.adam_step_clipped(ref, *HP, clip)
        assert f_ref == 0 and norm.value == n_ref
    assert found.value == found_dev.item() == 0
    dev.compare(ref)


# ------------------------------------------------------------- reduction

@pytest.mark.parametrize("name", list(LISTS))
@pytest.mark.parametrize("k,norm", [(1, False), (2, True), (3, False), (8, False)])
def test_reduce_stays_in_bounds(lib, name, k, norm):
    Lib, L = lib
    arena = Arena(11, cap=8 << 20)
    rng = np.random.default_rng(12)
    sizes, u8, _, f = sizes_of(name)
    items = (L.ReduceItem * len(sizes))()
    shards, scales, codes, amax, scale = [], [], [], [], []
    for i, n in enumerate(sizes):
        stride = n + (i % 3) * 5 + (16 if i == 4 else 0)   # padded, unaligned
        sh = (rng.integers(0, 0x7F, (k, stride)) |
              (rng.integers(0, 2, (k, stride)) << 7)).astype(np.uint8)
        src = arena.take(k * stride, u8[i])
        src.copy_(torch.from_numpy(sh.ravel()))
        sc = (2.0 ** rng.integers(-4, 5, k)).astype(np.float32)
        scv = arena.take(4 * k, f[i], torch.float32)
        scv.copy_(torch.from_numpy(sc))
        shards.append(sh)
        scales.append(sc)
        codes.append(arena.take(n, u8[(i + 1) % len(u8)], out=True))
        amax.append(arena.scalar(-7.0, f[i]))
        scale.append(arena.scalar(-7.0, f[i]))
        it = items[i]
        it.src, it.numel, it.stride, it.src_scale = ptr(src), n, stride, ptr(scv)
        it.codes, it.amax, it.scale = ptr(codes[i]), ptr(amax[i]), ptr(scale[i])
    n = len(sizes)
    if norm:
        terms = arena.take(8 * n, 8, torch.float64, out=True)
        found_dev = arena.scalar(7, 0, dtype=torch.int32)
    arena.seal()
    post = 1.0 / k
    if norm:
        rc = Lib.fp8_reduce_scaled_norm(items, n, k, E4M3, E4M3, post, 1.0,
                                        ptr(terms), ptr(found_dev), None)
    else:
        rc = Lib.fp8_reduce_scaled(items, n, k, E4M3, E4M3, post, None)
    assert rc == 0
    arena.check("reduction")
    for i, (sh, sc) in enumerate(zip(shards, scales)):
        rc_, ra, rs = oracle.reduce_scaled(sh, sc, E4M3, E4M3, post, numel=sizes[i])
        check_f32_exact([amax[i].item()], [ra], f"amax[{i}]")
        check_f32_exact([scale[i].item()], [rs], f"scale[{i}]")
        check_codes(to_np_u8(codes[i]), rc_, name=f"codes[{i}]")
    if norm:
        assert found_dev.item() == 0
