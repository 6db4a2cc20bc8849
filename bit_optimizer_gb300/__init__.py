"""libfp8opt for GB300: the MS-AMP-style scaled FP8 cast and FP8-state AdamW
step as hand-written sm_103a CUDA kernels behind a C ABI (include/fp8opt.h).

Importing the package loads the in-tree shared library and fails if it has
not been built: there is no fallback path.
"""
from ._lib import (BF16, E4M3, E5M2, EXPORTS, F16, F32, KERNELS, Fp8OptError,
                   LIB_PATH, load, release, release_stream, strerror,
                   timing_enable, timing_read)
from .api import (AdamWPlan, CastPlan, CastStepPlan, Fp8AdamW, ReducePlan,
                  StepState, arena_views, fp8_adamw_step, fp8_cast_scaled,
                  fp8_reduce_scaled)

load()

__all__ = ["fp8_cast_scaled", "fp8_adamw_step", "fp8_reduce_scaled",
           "CastPlan", "AdamWPlan", "CastStepPlan", "ReducePlan", "StepState",
           "Fp8AdamW", "arena_views", "E4M3", "E5M2", "F32", "BF16", "F16",
           "Fp8OptError", "strerror", "release", "release_stream", "load",
           "LIB_PATH", "EXPORTS",
           "KERNELS", "timing_enable", "timing_read"]
