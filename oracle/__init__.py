"""Python access to the scalar C oracle (fp8opt_oracle.c).

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it, and it never calls the CUDA library.

Arrays are numpy: FP8 codes ``uint8``; FP16 and BF16 as their ``uint16`` bit
patterns; FP32 as ``float32``.  ``build()`` compiles the C file with gcc
(``-ffp-contract=off``, no fast-math) into ``oracle/_build``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import List, Sequence

import numpy as np

E4M3, E5M2 = 0, 1
F32, BF16, F16 = 0, 1, 2
FMT = {"e4m3": E4M3, "e5m2": E5M2}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8opt_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_fp8opt.so")
_lib = None


def compile_library(src: str, out: str) -> str:
    """Compile a C source with the oracle's flags into the shared library
    ``out`` (written atomically); return ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
        "-fno-fast-math", "-fno-finite-math-only", "-Wall", "-o", tmp, src,
        "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc); return its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_library(_SRC, _LIB_PATH)


class Param(C.Structure):
    _fields_ = [
        ("numel", C.c_int64), ("g", C.c_void_p), ("g_scale", C.c_float),
        ("g_fmt", C.c_int), ("m", C.c_void_p), ("m_scale", C.c_void_p),
        ("v", C.c_void_p), ("w", C.c_void_p), ("w8", C.c_void_p),
        ("w8_scale", C.c_void_p), ("w8_amax", C.c_void_p),
        ("v_bound", C.c_void_p),
    ]


def lib():
    """The loaded oracle.  ``FP8OPT_ORACLE_LIB`` may name another build of
    the same C source (the mutation test plants one mistake in a copy and
    checks that the pins fail on it); otherwise the library ``build()``
    makes."""
    global _lib
    if _lib is None:
        L = C.CDLL(os.environ.get("FP8OPT_ORACLE_LIB") or build())
        L.oracle_fp8_decode.restype = C.c_float
        L.oracle_fp8_decode.argtypes = [C.c_uint8, C.c_int]
        L.oracle_fp8_encode.restype = C.c_uint8
        L.oracle_fp8_encode.argtypes = [C.c_float, C.c_int]
        L.oracle_f32_to_f16.restype = C.c_uint16
        L.oracle_f32_to_f16.argtypes = [C.c_float]
        L.oracle_f16_to_f32.restype = C.c_float
        L.oracle_f16_to_f32.argtypes = [C.c_uint16]
        L.oracle_bf16_to_f32.restype = C.c_float
        L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
        L.oracle_scale_from_amax.restype = C.c_float
        L.oracle_scale_from_amax.argtypes = [C.c_float, C.c_int]
        L.oracle_fp8_max.restype = C.c_double
        L.oracle_fp8_max.argtypes = [C.c_int]
        L.oracle_cast_scaled.restype = C.c_int
        L.oracle_cast_scaled.argtypes = [C.c_void_p, C.c_int, C.c_int64, C.c_int,
                                         C.c_void_p, C.c_void_p, C.c_void_p]
        L.oracle_reduce_scaled.restype = C.c_int
        L.oracle_reduce_scaled.argtypes = [C.c_void_p, C.c_int64, C.c_int64,
                                           C.c_void_p, C.c_int, C.c_int, C.c_int,
                                           C.c_float, C.c_void_p, C.c_void_p,
                                           C.c_void_p]
        L.oracle_adamw_step.restype = C.c_int
        L.oracle_adamw_step.argtypes = [C.POINTER(Param), C.c_int, C.c_float,
                                        C.c_float, C.c_float, C.c_float,
                                        C.c_float, C.c_int64, C.c_float]
        L.oracle_adam_step.restype = C.c_int
        L.oracle_adam_step.argtypes = [C.POINTER(Param), C.c_int, C.c_int,
                                       C.c_float, C.c_float, C.c_float,
                                       C.c_float, C.c_float, C.c_int64, C.c_float]
        L.oracle_grad_norm.restype = C.c_int
        L.oracle_grad_norm.argtypes = [C.POINTER(Param), C.c_int, C.c_float,
                                       C.POINTER(C.c_double)]
        L.oracle_grad_norm_terms.restype = C.c_int
        L.oracle_grad_norm_terms.argtypes = [C.POINTER(Param), C.c_int, C.c_float,
                                             C.c_void_p]
        L.oracle_clip_coef.restype = C.c_float
        L.oracle_clip_coef.argtypes = [C.c_double, C.c_float]
        L.oracle_adam_step_clipped.restype = C.c_int
        L.oracle_adam_step_clipped.argtypes = [
            C.POINTER(Param), C.c_int, C.c_int, C.c_float, C.c_float, C.c_float,
            C.c_float, C.c_float, C.c_int64, C.c_float, C.c_float,
            C.POINTER(C.c_double)]
        L.oracle_adam_step_coef.restype = C.c_int
        L.oracle_adam_step_coef.argtypes = [
            C.POINTER(Param), C.c_int, C.c_int, C.c_float, C.c_float, C.c_float,
            C.c_float, C.c_float, C.c_int64, C.c_float, C.c_float]
        step_head = [C.POINTER(Param), C.c_int, C.c_int, C.c_float, C.c_float,
                     C.c_float]
        L.oracle_step_maxima.restype = C.c_int
        L.oracle_step_maxima.argtypes = step_head + [
            C.c_float, C.c_int64, C.c_float, C.c_float, C.c_void_p, C.c_void_p]
        L.oracle_step_update.restype = C.c_int
        L.oracle_step_update.argtypes = step_head + [
            C.c_float, C.c_float, C.c_int64, C.c_float, C.c_float, C.c_void_p,
            C.c_void_p, C.c_void_p]
        L.oracle_weight_copy.restype = C.c_int
        L.oracle_weight_copy.argtypes = [C.POINTER(Param), C.c_int, C.c_void_p]
        L.oracle_reduce_scaled_given.restype = C.c_int
        L.oracle_reduce_scaled_given.argtypes = [
            C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int, C.c_int,
            C.c_int, C.c_float, C.c_float, C.c_void_p, C.c_void_p]
        L.oracle_fp8_sq_sum.restype = None
        L.oracle_fp8_sq_sum.argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_void_p]
        L.oracle_bias_power.restype = C.c_double
        L.oracle_bias_power.argtypes = [C.c_double, C.c_int64]
        L.oracle_v_scale_from_bound.restype = C.c_float
        L.oracle_v_scale_from_bound.argtypes = [C.c_float]
        L.oracle_state_bytes.restype = C.c_int
        L.oracle_state_bytes.argtypes = [C.c_int]
        for nm in ("oracle_fp8_encode_array", "oracle_fp8_decode_array"):
            getattr(L, nm).restype = None
            getattr(L, nm).argtypes = [C.c_void_p, C.c_int64, C.c_int, C.c_void_p]
        for nm in ("oracle_f32_to_f16_array", "oracle_f16_to_f32_array"):
            getattr(L, nm).restype = None
            getattr(L, nm).argtypes = [C.c_void_p, C.c_int64, C.c_void_p]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ------------------------------------------------------------------ codecs

def fp8_decode(codes: np.ndarray, fmt: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float32)
    lib().oracle_fp8_decode_array(_ptr(c), c.size, fmt, _ptr(out))
    return out


def fp8_encode(x: np.ndarray, fmt: int) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    lib().oracle_fp8_encode_array(_ptr(a), a.size, fmt, _ptr(out))
    return out


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_ptr(a), a.size, _ptr(out))
    return out


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(a.shape, dtype=np.float32)
    lib().oracle_f16_to_f32_array(_ptr(a), a.size, _ptr(out))
    return out


def scale_from_amax(amax: float, fmt: int) -> float:
    return lib().oracle_scale_from_amax(amax, fmt)


def fp8_max(fmt: int) -> float:
    return lib().oracle_fp8_max(fmt)


def state_bytes(level: int) -> int:
    return lib().oracle_state_bytes(level)


# -------------------------------------------------------------------- cast

def cast_scaled(src: np.ndarray, dtype: int, fmt: int):
    """Returns (codes uint8, amax float32 scalar, scale float32 scalar)."""
    want = np.float32 if dtype == F32 else np.uint16
    s = np.ascontiguousarray(src, dtype=want).ravel()
    codes = np.empty(s.size, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    scale = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_cast_scaled(_ptr(s), dtype, s.size, fmt, _ptr(codes),
                                  _ptr(amax), _ptr(scale))
    if rc != 0:
        raise ValueError(f"oracle_cast_scaled rejected its arguments ({rc})")
    return codes, amax[0], scale[0]


# ---------------------------------------------------------- FP8 reduction

def reduce_scaled_given(shards: np.ndarray, scales, in_fmt: int, out_fmt: int,
                        post: float, amax: float, numel: int = None):
    """reduce_scaled with the output scale taken from a given amax (a tensor
    reduced in pieces takes the whole tensor's amax): returns (codes uint8,
    scale float32 scalar)."""
    sh = np.ascontiguousarray(shards, dtype=np.uint8)
    assert sh.ndim == 2
    k, stride = sh.shape
    n = stride if numel is None else int(numel)
    sc = np.ascontiguousarray(scales, dtype=np.float32).ravel()
    assert sc.size == k
    codes = np.empty(n, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_reduce_scaled_given(_ptr(sh), n, stride, _ptr(sc), k, in_fmt,
                                          out_fmt, post, amax, _ptr(codes),
                                          _ptr(scale))
    if rc != 0:
        raise ValueError(f"oracle_reduce_scaled_given rejected its arguments ({rc})")
    return codes, scale[0]


def fp8_sq_sum(codes: np.ndarray, fmt: int) -> int:
    """The exact sum of the codes' squared values in units of 2^-32, as a
    Python int (non-finite codes count 0)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.zeros(2, dtype=np.uint64)
    lib().oracle_fp8_sq_sum(_ptr(c), c.size, fmt, _ptr(out))
    return int(out[0]) | (int(out[1]) << 64)


def reduce_scaled(shards: np.ndarray, scales, in_fmt: int, out_fmt: int,
                  post: float = 1.0, numel: int = None):
    """Local reduction of k FP8 shards: ``shards`` is a [k, stride] uint8
    array (each row one shard's codes; the first ``numel`` columns are used,
    all of them by default), ``scales`` the k encode scales.  Returns (codes
    uint8[numel], amax float32 scalar, scale float32 scalar)."""
    sh = np.ascontiguousarray(shards, dtype=np.uint8)
    assert sh.ndim == 2
    k, stride = sh.shape
    n = stride if numel is None else int(numel)
    sc = np.ascontiguousarray(scales, dtype=np.float32).ravel()
    assert sc.size == k
    codes = np.empty(n, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    scale = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_reduce_scaled(_ptr(sh), n, stride, _ptr(sc), k, in_fmt,
                                    out_fmt, post, _ptr(codes), _ptr(amax),
                                    _ptr(scale))
    if rc != 0:
        raise ValueError(f"oracle_reduce_scaled rejected its arguments ({rc})")
    return codes, amax[0], scale[0]


# -------------------------------------------------------------------- step

class StepState:
    """One tensor's optimizer state, as numpy arrays the oracle updates in place.

    g: uint8 gradient codes; g_scale: float; g_fmt: E4M3/E5M2;
    m: uint8 E4M3 codes; m_scale: float32[1]; v, w: uint16 FP16 bits;
    O3 only: w8 uint8, w8_scale float32[1], w8_amax float32[1].
    Scaled second moment only: v_bound float32[1] (v then holds FP16 of
    v * 2^14 / v_bound).
    """

    def __init__(self, g, g_scale, m, m_scale, v, w, g_fmt=E4M3, o3=False,
                 scaled_v=False, v_bound=0.0):
        self.g = np.ascontiguousarray(g, dtype=np.uint8).ravel()
        self.g_scale = float(np.float32(g_scale))
        self.g_fmt = g_fmt
        self.m = np.ascontiguousarray(m, dtype=np.uint8).ravel().copy()
        self.m_scale = np.array([m_scale], dtype=np.float32)
        self.v = np.ascontiguousarray(v, dtype=np.uint16).ravel().copy()
        self.w = np.ascontiguousarray(w, dtype=np.uint16).ravel().copy()
        n = self.g.size
        assert self.m.size == n and self.v.size == n and self.w.size == n
        if o3:
            self.w8 = np.zeros(n, dtype=np.uint8)
            self.w8_scale = np.ones(1, dtype=np.float32)
            self.w8_amax = np.zeros(1, dtype=np.float32)
        else:
            self.w8 = self.w8_scale = self.w8_amax = None
        self.v_bound = (np.array([v_bound], dtype=np.float32) if scaled_v
                        else None)

    @property
    def numel(self):
        return self.g.size

    def copy(self):
        c = StepState.__new__(StepState)
        for k, v in self.__dict__.items():
            setattr(c, k, v.copy() if isinstance(v, np.ndarray) else v)
        return c

    def _param(self) -> Param:
        p = Param()
        p.numel = self.g.size
        p.g = _ptr(self.g)
        p.g_scale = self.g_scale
        p.g_fmt = self.g_fmt
        p.m = _ptr(self.m)
        p.m_scale = _ptr(self.m_scale)
        p.v = _ptr(self.v)
        p.w = _ptr(self.w)
        if self.w8 is not None:
            p.w8 = _ptr(self.w8)
            p.w8_scale = _ptr(self.w8_scale)
            p.w8_amax = _ptr(self.w8_amax)
        if self.v_bound is not None:
            p.v_bound = _ptr(self.v_bound)
        return p


def bias_power(b: float, t: int) -> float:
    """beta^t as the step's bias corrections take it (binary exponentiation
    in double)."""
    return lib().oracle_bias_power(b, t)


def v_scale_from_bound(b: float) -> float:
    return lib().oracle_v_scale_from_bound(b)


def adamw_step(states: Sequence[StepState], lr, beta1, beta2, eps, wd, step,
               inv_loss_scale, l2=False) -> int:
    """One oracle step over the list (AdamW, or Adam with L2 decay when l2);
    returns found_inf (0 or 1)."""
    arr = (Param * max(1, len(states)))()
    for i, s in enumerate(states):
        arr[i] = s._param()
    rc = lib().oracle_adam_step(arr, len(states), 1 if l2 else 0, lr, beta1,
                                beta2, eps, wd, step, inv_loss_scale)
    if rc < 0:
        raise ValueError(f"oracle_adamw_step rejected its arguments ({rc})")
    return rc


def _params(states):
    arr = (Param * max(1, len(states)))()
    for i, s in enumerate(states):
        arr[i] = s._param()
    return arr


def grad_norm_codes(codes: Sequence[np.ndarray], g_scales, g_fmts,
                    inv_loss_scale):
    """grad_norm over gradient codes alone (no optimizer state):
    (found_inf, norm)."""
    n = len(codes)
    arr = (Param * max(1, n))()
    keep = []
    for i, c in enumerate(codes):
        c = np.ascontiguousarray(c, dtype=np.uint8).ravel()
        keep.append(c)
        arr[i].numel = c.size
        arr[i].g = _ptr(c)
        arr[i].g_scale = float(np.float32(g_scales[i]))
        arr[i].g_fmt = g_fmts[i] if isinstance(g_fmts, (list, tuple)) else g_fmts
    norm = C.c_double(0.0)
    rc = lib().oracle_grad_norm(arr, n, inv_loss_scale, C.byref(norm))
    if rc < 0:
        raise ValueError(f"oracle_grad_norm rejected its arguments ({rc})")
    return rc, norm.value


def adam_step_coef(states: Sequence[StepState], lr, beta1, beta2, eps, wd, step,
                   inv_loss_scale, clip, l2=False) -> int:
    """One oracle step with a given clip coefficient; returns found_inf."""
    rc = lib().oracle_adam_step_coef(_params(states), len(states),
                                     1 if l2 else 0, lr, beta1, beta2, eps, wd,
                                     step, inv_loss_scale, clip)
    if rc < 0:
        raise ValueError(f"oracle_adam_step_coef rejected its arguments ({rc})")
    return rc


def step_maxima(states: Sequence[StepState], lr, beta1, beta2, wd, step,
                inv_loss_scale, clip=1.0, l2=False):
    """The step's first phase: (found_inf, amax_m, gmax), the per-record
    amax of this step's first moment and max |g| (float32 arrays; not
    written when found_inf).  Writes no state."""
    n = len(states)
    am = np.zeros(max(1, n), np.float32)
    gm = np.zeros(max(1, n), np.float32)
    rc = lib().oracle_step_maxima(_params(states), n, 1 if l2 else 0, lr, beta1,
                                  beta2, wd, step, inv_loss_scale, clip,
                                  _ptr(am), _ptr(gm))
    if rc < 0:
        raise ValueError(f"oracle_step_maxima rejected its arguments ({rc})")
    return rc, am[:n], gm[:n]


def step_update(states: Sequence[StepState], lr, beta1, beta2, eps, wd, step,
                inv_loss_scale, amax_m, gmax, clip=1.0, l2=False):
    """The step's second phase from the given per-record maxima (updates the
    states in place); returns each record's new FP16 master amax."""
    n = len(states)
    am = np.ascontiguousarray(amax_m, np.float32)
    gm = np.ascontiguousarray(gmax, np.float32)
    assert am.size >= n and gm.size >= n
    wm = np.zeros(max(1, n), np.float32)
    rc = lib().oracle_step_update(_params(states), n, 1 if l2 else 0, lr, beta1,
                                  beta2, eps, wd, step, inv_loss_scale, clip,
                                  _ptr(am), _ptr(gm), _ptr(wm))
    if rc < 0:
        raise ValueError(f"oracle_step_update rejected its arguments ({rc})")
    return wm[:n]


def weight_copy(states: Sequence[StepState], master_amax) -> None:
    """The step's third phase: each O3 record's FP8 weight copy from the
    given master amax."""
    n = len(states)
    wm = np.ascontiguousarray(master_amax, np.float32)
    assert wm.size >= n
    rc = lib().oracle_weight_copy(_params(states), n, _ptr(wm))
    if rc < 0:
        raise ValueError(f"oracle_weight_copy rejected its arguments ({rc})")


def grad_norm(states: Sequence[StepState], inv_loss_scale):
    """(found_inf, norm): the global L2 norm of the unscaled gradient codes of
    the list (+inf when found_inf)."""
    norm = C.c_double(0.0)
    rc = lib().oracle_grad_norm(_params(states), len(states), inv_loss_scale,
                                C.byref(norm))
    if rc < 0:
        raise ValueError(f"oracle_grad_norm rejected its arguments ({rc})")
    return rc, norm.value


def grad_norm_terms(states: Sequence[StepState], inv_loss_scale):
    """(found_inf, terms): the per-tensor terms k_t^2 * S_t of the norm."""
    terms = np.zeros(max(1, len(states)), dtype=np.float64)
    rc = lib().oracle_grad_norm_terms(_params(states), len(states),
                                      inv_loss_scale, _ptr(terms))
    if rc < 0:
        raise ValueError(f"oracle_grad_norm_terms rejected its arguments ({rc})")
    return rc, terms[:len(states)]


def clip_coef(norm: float, max_norm: float) -> float:
    return lib().oracle_clip_coef(norm, max_norm)


def adam_step_clipped(states: Sequence[StepState], lr, beta1, beta2, eps, wd,
                      step, inv_loss_scale, max_norm, l2=False):
    """One oracle step with global gradient-norm clipping; returns
    (found_inf, norm)."""
    norm = C.c_double(0.0)
    rc = lib().oracle_adam_step_clipped(_params(states), len(states),
                                        1 if l2 else 0, lr, beta1, beta2, eps,
                                        wd, step, inv_loss_scale, max_norm,
                                        C.byref(norm))
    if rc < 0:
        raise ValueError(f"oracle_adam_step_clipped rejected its arguments ({rc})")
    return rc, norm.value
