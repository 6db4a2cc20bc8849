"""ctypes binding of libfp8opt (include/fp8opt.h): argument marshalling only.

Every computation runs in the library's CUDA kernels.  The binding loads the
in-tree ``_build/libfp8opt.so`` and raises if it is missing; there is no other
code path.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfp8opt.so")

E4M3, E5M2 = 0, 1
F32, BF16, F16 = 0, 1, 2
OK, ERR_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_LIMIT = 0, -1, -2, -4, -5

# Every entry point the header declares.
EXPORTS = ("fp8_cast_scaled", "fp8_adamw_step", "fp8_adam_step",
           "fp8_cast_adamw_step", "fp8_reduce_scaled", "fp8_grad_norm",
           "fp8_adam_step_clipped", "fp8_grad_norm_terms", "fp8_clip_coef",
           "fp8_adam_step_begin", "fp8_adam_step_finish",
           "fp8_cast_adam_step_clipped", "fp8_reduce_scaled_norm",
           "fp8_cast_scaled_noalloc", "fp8_adam_step_dev",
           "fp8_cast_adamw_step_dev", "fp8_cast_adam_step_clipped_dev",
           "fp8_adam_step_copy", "fp8_reduce_scaled_begin",
           "fp8_reduce_scaled_finish", "fp8_norm_terms_from_limbs",
           "fp8opt_strerror",
           "fp8opt_last_error", "fp8opt_timing_enable", "fp8opt_timing_read",
           "fp8opt_release", "fp8opt_release_stream")
KERNELS = ("cast_amax", "cast_encode", "step_amax", "step_update", "step_w8",
           "cast_step_amax", "reduce_amax", "reduce_encode", "grad_norm",
           "grad_norm_terms", "clip_coef", "found")
MAX_SHARDS = 64


class CastItem(C.Structure):
    """fp8opt_cast_item."""
    _fields_ = [
        ("src", C.c_void_p), ("numel", C.c_int64), ("dtype", C.c_int32),
        ("reserved", C.c_int32), ("codes", C.c_void_p), ("amax", C.c_void_p),
        ("scale", C.c_void_p),
    ]


class Param(C.Structure):
    """fp8opt_param."""
    _fields_ = [
        ("numel", C.c_int64), ("g", C.c_void_p), ("g_scale", C.c_void_p),
        ("g_fmt", C.c_int32), ("reserved", C.c_int32), ("m", C.c_void_p),
        ("m_scale", C.c_void_p), ("v", C.c_void_p), ("w", C.c_void_p),
        ("w8", C.c_void_p), ("w8_scale", C.c_void_p), ("w8_amax", C.c_void_p),
        ("v_bound", C.c_void_p),
    ]


class ReduceItem(C.Structure):
    """fp8opt_reduce_item."""
    _fields_ = [
        ("src", C.c_void_p), ("numel", C.c_int64), ("stride", C.c_int64),
        ("src_scale", C.c_void_p), ("codes", C.c_void_p), ("amax", C.c_void_p),
        ("scale", C.c_void_p),
    ]


class Fp8OptError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"libfp8opt status {status}: {detail}")
        self.status = status


_lib: Optional[C.CDLL] = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libfp8opt is not built ({path} is missing); run "
            "`python bit_optimizer_gb300/build.py` or __graft_entry__.build()")
    L = C.CDLL(path)
    L.fp8_cast_scaled.restype = C.c_int
    L.fp8_cast_scaled.argtypes = [C.POINTER(CastItem), C.c_int, C.c_int,
                                  C.c_void_p]
    L.fp8_adam_step.restype = C.c_int
    L.fp8_adam_step.argtypes = [
        C.POINTER(Param), C.c_int, C.c_float, C.c_float, C.c_float, C.c_float,
        C.c_float, C.c_int64, C.c_float, C.POINTER(C.c_int), C.c_void_p,
        C.c_void_p]
    L.fp8_cast_adamw_step.restype = C.c_int
    L.fp8_cast_adamw_step.argtypes = [
        C.POINTER(CastItem), C.POINTER(Param), C.c_int, C.c_int, C.c_float,
        C.c_float, C.c_float, C.c_float, C.c_float, C.c_int64, C.c_float,
        C.POINTER(C.c_int), C.c_void_p, C.c_void_p]
    L.fp8_reduce_scaled.restype = C.c_int
    L.fp8_reduce_scaled.argtypes = [C.POINTER(ReduceItem), C.c_int, C.c_int,
                                    C.c_int, C.c_int, C.c_float, C.c_void_p]
    L.fp8_grad_norm.restype = C.c_int
    L.fp8_grad_norm.argtypes = [C.POINTER(Param), C.c_int, C.c_float,
                                C.POINTER(C.c_double), C.c_void_p,
                                C.POINTER(C.c_int), C.c_void_p]
    L.fp8_adam_step_clipped.restype = C.c_int
    L.fp8_adam_step_clipped.argtypes = [
        C.POINTER(Param), C.c_int, C.c_float, C.c_float, C.c_float, C.c_float,
        C.c_float, C.c_int64, C.c_float, C.c_int, C.c_float,
        C.POINTER(C.c_double), C.c_void_p, C.POINTER(C.c_int), C.c_void_p,
        C.c_void_p]
    L.fp8_grad_norm_terms.restype = C.c_int
    L.fp8_grad_norm_terms.argtypes = [C.POINTER(Param), C.c_int, C.c_float,
                                      C.c_void_p, C.c_void_p, C.c_void_p]
    L.fp8_clip_coef.restype = C.c_int
    L.fp8_clip_coef.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_float,
                                C.c_void_p, C.c_void_p, C.c_void_p]
    step_head = [C.POINTER(Param), C.c_int, C.c_float, C.c_float, C.c_float,
                 C.c_float, C.c_float, C.c_int64, C.c_float, C.c_int]
    L.fp8_adam_step_begin.restype = C.c_int
    L.fp8_adam_step_begin.argtypes = step_head + [C.c_void_p, C.c_void_p,
                                                  C.c_void_p, C.c_void_p]
    L.fp8_adam_step_finish.restype = C.c_int
    L.fp8_adam_step_finish.argtypes = step_head + [C.c_void_p, C.c_void_p,
                                                   C.c_void_p, C.c_void_p,
                                                   C.c_void_p, C.c_void_p]
    L.fp8_adam_step_copy.restype = C.c_int
    L.fp8_adam_step_copy.argtypes = [C.POINTER(Param), C.c_int, C.c_void_p,
                                     C.c_void_p]
    L.fp8_reduce_scaled_begin.restype = C.c_int
    L.fp8_reduce_scaled_begin.argtypes = [C.POINTER(ReduceItem), C.c_int, C.c_int,
                                          C.c_int, C.c_float, C.c_void_p,
                                          C.c_void_p]
    L.fp8_reduce_scaled_finish.restype = C.c_int
    L.fp8_reduce_scaled_finish.argtypes = [
        C.POINTER(ReduceItem), C.c_int, C.c_int, C.c_int, C.c_int, C.c_float,
        C.c_void_p, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p]
    L.fp8_norm_terms_from_limbs.restype = C.c_int
    L.fp8_norm_terms_from_limbs.argtypes = [C.c_void_p, C.c_void_p, C.c_int,
                                            C.c_int, C.c_float, C.c_void_p,
                                            C.c_void_p]
    L.fp8_cast_adam_step_clipped.restype = C.c_int
    L.fp8_cast_adam_step_clipped.argtypes = [
        C.POINTER(CastItem), C.POINTER(Param), C.c_int, C.c_int, C.c_float,
        C.c_float, C.c_float, C.c_float, C.c_float, C.c_int64, C.c_float, C.c_int,
        C.c_float, C.POINTER(C.c_double), C.c_void_p, C.POINTER(C.c_int),
        C.c_void_p, C.c_void_p]
    L.fp8_reduce_scaled_norm.restype = C.c_int
    L.fp8_reduce_scaled_norm.argtypes = [C.POINTER(ReduceItem), C.c_int, C.c_int,
                                         C.c_int, C.c_int, C.c_float, C.c_float,
                                         C.c_void_p, C.c_void_p, C.c_void_p]
    L.fp8_cast_scaled_noalloc.restype = C.c_int
    L.fp8_cast_scaled_noalloc.argtypes = [C.POINTER(CastItem), C.c_int, C.c_int,
                                          C.c_void_p]
    L.fp8_adamw_step.restype = C.c_int
    L.fp8_adamw_step.argtypes = [
        C.POINTER(Param), C.c_int, C.c_float, C.c_float, C.c_float, C.c_float,
        C.c_float, C.c_int64, C.c_float, C.POINTER(C.c_int), C.c_void_p,
        C.c_void_p]
    L.fp8_adam_step_dev.restype = C.c_int
    L.fp8_adam_step_dev.argtypes = [
        C.POINTER(Param), C.c_int, C.c_float, C.c_float, C.c_float, C.c_float,
        C.c_int, C.c_void_p, C.c_void_p, C.c_void_p]
    L.fp8_cast_adamw_step_dev.restype = C.c_int
    L.fp8_cast_adamw_step_dev.argtypes = [
        C.POINTER(CastItem), C.POINTER(Param), C.c_int, C.c_int, C.c_float,
        C.c_float, C.c_float, C.c_float, C.c_void_p, C.c_void_p, C.c_void_p]
    L.fp8_cast_adam_step_clipped_dev.restype = C.c_int
    L.fp8_cast_adam_step_clipped_dev.argtypes = [
        C.POINTER(CastItem), C.POINTER(Param), C.c_int, C.c_int, C.c_float,
        C.c_float, C.c_float, C.c_float, C.c_int, C.c_float, C.c_void_p,
        C.c_void_p, C.c_void_p, C.c_void_p]
    L.fp8opt_strerror.restype = C.c_char_p
    L.fp8opt_strerror.argtypes = [C.c_int]
    L.fp8opt_last_error.restype = C.c_char_p
    L.fp8opt_last_error.argtypes = []
    L.fp8opt_timing_enable.restype = C.c_int
    L.fp8opt_timing_enable.argtypes = [C.c_int]
    L.fp8opt_timing_read.restype = C.c_int
    L.fp8opt_timing_read.argtypes = [C.c_char_p, C.POINTER(C.c_int),
                                     C.POINTER(C.c_double)]
    L.fp8opt_release.restype = None
    L.fp8opt_release.argtypes = []
    L.fp8opt_release_stream.restype = None
    L.fp8opt_release_stream.argtypes = [C.c_void_p]
    _lib = L
    return L


def check(status: int) -> int:
    if status != OK:
        L = load()
        raise Fp8OptError(status, (L.fp8opt_last_error() or b"").decode()
                          or L.fp8opt_strerror(status).decode())
    return status


def strerror(status: int) -> str:
    return load().fp8opt_strerror(status).decode()


def timing_enable(on: bool) -> None:
    """Start (clearing the record) or stop per-kernel event timing."""
    check(load().fp8opt_timing_enable(1 if on else 0))


def timing_read(kernel: str):
    """(launches, total milliseconds) of one kernel since timing_enable(True)."""
    n, ms = C.c_int(0), C.c_double(0.0)
    check(load().fp8opt_timing_read(kernel.encode(), C.byref(n), C.byref(ms)))
    return n.value, ms.value


def release() -> None:
    load().fp8opt_release()


def release_stream(stream) -> None:
    """Frees the workspace of one stream (a torch.cuda.Stream or a raw
    cudaStream_t), e.g. after the CUDA graphs captured on it are destroyed."""
    ptr = getattr(stream, "cuda_stream", stream)
    load().fp8opt_release_stream(ptr or None)
