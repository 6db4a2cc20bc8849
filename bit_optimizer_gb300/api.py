"""PyTorch-facing binding of libfp8opt.

PyTorch supplies device memory and streams only; every step of the cast and
the optimizer runs in the library's CUDA kernels, reached through the C ABI.

* ``fp8_cast_scaled`` / ``CastPlan``: per-tensor just-in-time scaled FP8 cast
  of a tensor list (MS-AMP O1 gradients in FP8).
* ``fp8_adamw_step`` / ``AdamWPlan``: one multi-tensor AdamW step with E4M3
  first moment and FP16 second moment (MS-AMP O2), FP16 master plus E4M3
  weight copy for O3, and the GradScaler inf/NaN skip.
* ``fp8_reduce_scaled`` / ``ReducePlan``: local reduction of k FP8 shards per
  tensor (the arithmetic half of an FP8 all-reduce), re-encoded with a
  just-in-time scale.
* ``Fp8AdamW``: an optimizer object that owns the low-bit state in flat,
  256-byte-aligned arenas and runs cast + step for a list of FP16 weights,
  with ``state_dict`` / ``load_state_dict`` for checkpoint and resume.

A "plan" marshals its tensor list into the C records once; calling it again
passes the same records, so a repeated call costs one ctypes call and, inside
the library, no table upload.
"""
from __future__ import annotations

import ctypes as C
import math
from typing import Dict, List, Optional, Sequence

import torch

from . import _lib
from ._lib import (BF16, E4M3, E5M2, F16, F32, CastItem, Param, ReduceItem,
                   check, load)

FMTS = {"e4m3": E4M3, "e5m2": E5M2, E4M3: E4M3, E5M2: E5M2}
_DT = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}

__all__ = ["fp8_cast_scaled", "fp8_adamw_step", "fp8_reduce_scaled",
           "clip_coef", "CastPlan", "AdamWPlan", "CastStepPlan", "ReducePlan",
           "Fp8AdamW", "arena_views", "FMTS"]


def _fmt(f) -> int:
    try:
        return FMTS[f]
    except KeyError:
        raise ValueError(f"unknown FP8 format {f!r}") from None


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> Optional[int]:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream or None


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _slot_ptr(t: torch.Tensor, i: int, name: str) -> int:
    """Address of element i of a float32 vector (one scale/amax per tensor)."""
    _cuda(t, name)
    if t.dtype != torch.float32 or t.numel() <= i:
        raise ValueError(f"{name} must be float32 with one element per tensor")
    return t.data_ptr() + 4 * i


def arena_views(numels: Sequence[int], dtype: torch.dtype, device,
                align_bytes: int = 256, fill=None, return_base=False):
    """One flat allocation cut into per-tensor views, each starting on an
    ``align_bytes`` boundary (the vector path wants 16-byte starts).  With
    ``return_base`` also returns the flat buffer."""
    isz = torch.empty((), dtype=dtype).element_size()
    step = max(1, align_bytes // isz)
    offs, total = [], 0
    for n in numels:
        offs.append(total)
        total += (n + step - 1) // step * step
    buf = (torch.empty(max(total, 1), dtype=dtype, device=device)
           if fill is None else
           torch.full((max(total, 1),), fill, dtype=dtype, device=device))
    views = [buf[o:o + n] for o, n in zip(offs, numels)]
    return (views, buf) if return_base else views


def _ptr_or_none(t: Optional[torch.Tensor], name: str, dtype) -> Optional[int]:
    if t is None:
        return None
    _cuda(t, name)
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    return t.data_ptr()


# ------------------------------------------------------------------- cast

class CastPlan:
    """A marshalled ``fp8_cast_scaled`` over fixed buffers.

    srcs: contiguous CUDA tensors (float32, bfloat16 or float16);
    codes: uint8 CUDA tensors with the same numels; amax, scale: float32 CUDA
    vectors with one entry per tensor.
    """

    def __init__(self, srcs, codes, amax, scale, fmt="e4m3"):
        n = len(srcs)
        if len(codes) != n:
            raise ValueError("srcs and codes differ in length")
        self.fmt = _fmt(fmt)
        self.n = n
        self._keep = (list(srcs), list(codes), amax, scale)
        self._items = (CastItem * max(n, 1))()
        for i, (s, c) in enumerate(zip(srcs, codes)):
            _cuda(s, "src")
            _cuda(c, "codes")
            if s.dtype not in _DT:
                raise TypeError(f"src {i}: unsupported dtype {s.dtype}")
            if c.dtype != torch.uint8 or c.numel() != s.numel():
                raise ValueError(f"codes {i} must be uint8 with the src numel")
            it = self._items[i]
            it.src, it.numel, it.dtype = s.data_ptr(), s.numel(), _DT[s.dtype]
            it.codes = c.data_ptr()
            it.amax = _slot_ptr(amax, i, "amax")
            it.scale = _slot_ptr(scale, i, "scale")

    def __call__(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        check(load().fp8_cast_scaled(self._items, self.n, self.fmt,
                                     _stream_ptr(stream)))


def fp8_cast_scaled(srcs: Sequence[torch.Tensor], fmt="e4m3", codes=None,
                    amax=None, scale=None, stream=None):
    """Scaled FP8 cast of each tensor: returns (codes list, amax, scale).

    amax[i] = max |srcs[i]|; scale[i] = fp8_max / amax[i] (1.0 for a zero or
    non-finite amax); codes[i] = RNE-saturating FP8 encode of srcs[i] * scale.
    """
    srcs = list(srcs)
    dev = srcs[0].device if srcs else torch.device("cuda")
    if codes is None:
        codes = [torch.empty(s.numel(), dtype=torch.uint8, device=dev) for s in srcs]
    if amax is None:
        amax = torch.empty(max(len(srcs), 1), dtype=torch.float32, device=dev)
    if scale is None:
        scale = torch.empty(max(len(srcs), 1), dtype=torch.float32, device=dev)
    CastPlan(srcs, codes, amax, scale, fmt)(stream)
    return codes, amax, scale


# ------------------------------------------------------------- reduction

class ReducePlan:
    """A marshalled ``fp8_reduce_scaled`` over fixed buffers.

    shards: per tensor a uint8 CUDA tensor of shape [k, numel] whose rows are
    the k shards (unit stride within a row; the row stride may exceed numel,
    e.g. a slice of a padded receive buffer); scales: per tensor the k shard
    scales, as a float32 CUDA tensor [n, k] (row i for tensor i) or a list of
    k-element float32 CUDA vectors; codes: uint8 CUDA tensors of numel (one
    may be row 0 of its shards for an in-place reduction); amax, scale:
    float32 CUDA vectors with one entry per tensor.  post multiplies the sum
    (1 / k for a mean).
    """

    def __init__(self, shards, scales, codes, amax, scale, in_fmt="e4m3",
                 out_fmt="e4m3", post=1.0):
        n = len(shards)
        if len(codes) != n or len(scales) != n:
            raise ValueError("shards, scales and codes differ in length")
        ks = {int(t.shape[0]) for t in shards} if n else {1}
        if len(ks) != 1:
            raise ValueError("every tensor needs the same number of shards")
        self.k = ks.pop()
        self.in_fmt, self.out_fmt = _fmt(in_fmt), _fmt(out_fmt)
        self.post = float(post)
        self.n = n
        self._keep = (list(shards), scales, list(codes), amax, scale)
        self._items = (ReduceItem * max(n, 1))()
        for i in range(n):
            sh, c, sc = shards[i], codes[i], scales[i]
            if not isinstance(sh, torch.Tensor) or not sh.is_cuda:
                raise TypeError("shards must be CUDA tensors")
            if sh.dtype != torch.uint8 or sh.dim() != 2 or (
                    sh.shape[1] > 1 and sh.stride(1) != 1):
                raise ValueError(f"shards[{i}] must be uint8 [k, numel] with unit row stride")
            _cuda(c, "codes")
            ne = int(sh.shape[1])
            if c.dtype != torch.uint8 or c.numel() != ne:
                raise ValueError(f"codes[{i}] must be uint8 with numel {ne}")
            _cuda(sc, "scales")
            if sc.dtype != torch.float32 or sc.numel() != self.k:
                raise ValueError(f"scales[{i}] must be float32 with k elements")
            it = self._items[i]
            it.src, it.numel = sh.data_ptr(), ne
            # (the library rejects a row stride below numel; an empty tensor's
            # stride does not matter)
            it.stride = (sh.stride(0) if ne else 0) if self.k > 1 else ne
            it.src_scale = sc.data_ptr()
            it.codes = c.data_ptr()
            it.amax = _slot_ptr(amax, i, "amax")
            it.scale = _slot_ptr(scale, i, "scale")

    def __call__(self, stream: Optional[torch.cuda.Stream] = None,
                 norm_terms: Optional[torch.Tensor] = None,
                 found: Optional[torch.Tensor] = None,
                 inv_loss_scale: float = 1.0) -> None:
        """One reduction.  With norm_terms (float64 CUDA, one per tensor):
        also the norm terms of the outputs and, in found (int32 CUDA scalar,
        optional), their found_inf (fp8_reduce_scaled_norm)."""
        if norm_terms is None:
            check(load().fp8_reduce_scaled(self._items, self.n, self.k,
                                           self.in_fmt, self.out_fmt, self.post,
                                           _stream_ptr(stream)))
            return
        if norm_terms.numel() < self.n:
            raise ValueError("norm_terms needs one float64 per tensor")
        check(load().fp8_reduce_scaled_norm(
            self._items, self.n, self.k, self.in_fmt, self.out_fmt, self.post,
            inv_loss_scale, _ptr_or_none(norm_terms, "norm_terms", torch.float64),
            _ptr_or_none(found, "found", torch.int32), _stream_ptr(stream)))

    # The reduction split at its amax, for tensors reduced in pieces on
    # several ranks (fp8_reduce_scaled_begin / _finish).  amax_bits: int32
    # CUDA, one per item (fp32 bits); limbs: int64 CUDA, four per item;
    # found: int32 CUDA scalar.  Neither waits for the stream.

    def begin(self, amax_bits: torch.Tensor, stream=None) -> None:
        if amax_bits.numel() < self.n:
            raise ValueError("amax_bits needs one int32 per item")
        check(load().fp8_reduce_scaled_begin(
            self._items, self.n, self.k, self.in_fmt, self.post,
            _ptr_or_none(amax_bits, "amax_bits", torch.int32), _stream_ptr(stream)))

    def finish(self, amax_bits: torch.Tensor, inv_loss_scale: float = 1.0,
               limbs: Optional[torch.Tensor] = None,
               found: Optional[torch.Tensor] = None, stream=None) -> None:
        if amax_bits.numel() < self.n or (limbs is not None and
                                          limbs.numel() < 4 * self.n):
            raise ValueError("amax_bits needs one int32 and limbs four int64 per item")
        check(load().fp8_reduce_scaled_finish(
            self._items, self.n, self.k, self.in_fmt, self.out_fmt, self.post,
            _ptr_or_none(amax_bits, "amax_bits", torch.int32), inv_loss_scale,
            _ptr_or_none(limbs, "limbs", torch.int64),
            _ptr_or_none(found, "found", torch.int32), _stream_ptr(stream)))


def fp8_reduce_scaled(shards: Sequence[torch.Tensor], scales, in_fmt="e4m3",
                      out_fmt="e4m3", post=1.0, codes=None, amax=None,
                      scale=None, stream=None):
    """Reduce k FP8 shards per tensor: returns (codes list, amax, scale).

    y = post * sum_j decode(shards[i][j]) / scales[i][j] (fp32, shard order);
    amax[i] = max |y|; scale[i] = fp8_max(out_fmt) / amax[i]; codes[i] =
    encode(y * scale[i]).
    """
    shards = list(shards)
    dev = shards[0].device if shards else torch.device("cuda")
    if codes is None:
        codes = [torch.empty(int(s.shape[1]), dtype=torch.uint8, device=dev)
                 for s in shards]
    if amax is None:
        amax = torch.empty(max(len(shards), 1), dtype=torch.float32, device=dev)
    if scale is None:
        scale = torch.empty(max(len(shards), 1), dtype=torch.float32, device=dev)
    ReducePlan(shards, scales, codes, amax, scale, in_fmt, out_fmt, post)(stream)
    return codes, amax, scale


# ------------------------------------------------------------------- step

class StepState:
    """fp8opt_step_state in device memory: lr, inv_loss_scale and the step
    count read by the *_dev step calls at run (or graph replay) time.
    ``lr`` and ``inv_loss_scale`` are float32 CUDA scalars, ``step`` an int64
    CUDA scalar (steps taken so far), all views of one 16-byte buffer.  Write
    them with tensor operations (``state.lr.fill_(x)``,
    ``state.inv_loss_scale.copy_(t)``), inside or outside a captured graph."""

    def __init__(self, lr=1e-3, inv_loss_scale=1.0, step=0, device=None):
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.buf = torch.zeros(2, dtype=torch.int64, device=dev)
        f = self.buf.view(torch.float32)
        self.lr = f[0]
        self.inv_loss_scale = f[1]
        self.step = self.buf[1]
        self.lr.fill_(float(lr))
        self.inv_loss_scale.fill_(float(inv_loss_scale))
        self.step.fill_(int(step))

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


class AdamWPlan:
    """A marshalled ``fp8_adamw_step`` over fixed state buffers.

    g: uint8 gradient codes per tensor; g_scale: float32 vector (n);
    m: uint8 E4M3 first moments; m_scale: float32 vector (n); v: float16
    second moments; w: float16 weights (O2) or masters (O3).  O3 when w8 (uint8
    per tensor), w8_scale and w8_amax (float32 vectors) are given.  A scaled
    second moment when v_bound (float32 vector, one bound per tensor, 0 with
    v = 0 at the start) is given.
    """

    def __init__(self, g, g_scale, m, m_scale, v, w, w8=None, w8_scale=None,
                 w8_amax=None, g_fmt="e4m3", v_bound=None):
        n = len(g)
        if not (len(m) == len(v) == len(w) == n):
            raise ValueError("g, m, v and w differ in length")
        o3 = w8 is not None
        if o3 and (w8_scale is None or w8_amax is None or len(w8) != n):
            raise ValueError("O3 needs w8, w8_scale and w8_amax")
        self.n = n
        self.o3 = o3
        self._keep = (list(g), g_scale, list(m), m_scale, list(v), list(w),
                      None if w8 is None else list(w8), w8_scale, w8_amax,
                      v_bound)
        fmts = g_fmt if isinstance(g_fmt, (list, tuple)) else [g_fmt] * n
        self._params = (Param * max(n, 1))()
        for i in range(n):
            ne = w[i].numel()
            for name, t, dt in (("g", g[i], torch.uint8), ("m", m[i], torch.uint8),
                                ("v", v[i], torch.float16),
                                ("w", w[i], torch.float16)):
                _cuda(t, name)
                if t.dtype != dt or t.numel() != ne:
                    raise ValueError(f"{name}[{i}] must be {dt} with numel {ne}")
            p = self._params[i]
            p.numel = ne
            p.g, p.g_fmt = g[i].data_ptr(), _fmt(fmts[i])
            p.g_scale = _slot_ptr(g_scale, i, "g_scale")
            p.m, p.m_scale = m[i].data_ptr(), _slot_ptr(m_scale, i, "m_scale")
            p.v, p.w = v[i].data_ptr(), w[i].data_ptr()
            if o3:
                _cuda(w8[i], "w8")
                if w8[i].dtype != torch.uint8 or w8[i].numel() != ne:
                    raise ValueError(f"w8[{i}] must be uint8 with numel {ne}")
                p.w8 = w8[i].data_ptr()
                p.w8_scale = _slot_ptr(w8_scale, i, "w8_scale")
                p.w8_amax = _slot_ptr(w8_amax, i, "w8_amax")
            if v_bound is not None:
                p.v_bound = _slot_ptr(v_bound, i, "v_bound")
        self._found = C.c_int(0)
        self._norm = C.c_double(0.0)
        self.last_grad_norm: Optional[float] = None

    def __call__(self, lr, beta1, beta2, eps, wd, step, inv_loss_scale=1.0,
                 found_inf_dev: Optional[torch.Tensor] = None, sync=True,
                 stream=None, l2=False, max_grad_norm=None,
                 grad_norm_dev: Optional[torch.Tensor] = None) -> Optional[int]:
        """Runs one step: AdamW, or Adam with L2 decay when l2.  sync=True
        returns found_inf (0/1) after waiting for the stream; sync=False
        returns None without waiting (found_inf is then only in
        found_inf_dev, a uint32/int32 CUDA tensor, if given).
        max_grad_norm: clip the unscaled gradient to this global L2 norm
        (0 reports the norm without clipping); the norm is then left in
        ``last_grad_norm`` (sync=True) and in grad_norm_dev (float32 CUDA
        scalar), if given."""
        fdev = None
        if found_inf_dev is not None:
            _cuda(found_inf_dev, "found_inf_dev")
            fdev = found_inf_dev.data_ptr()
        fptr = C.byref(self._found) if sync else None
        if max_grad_norm is None:
            fn = load().fp8_adam_step if l2 else load().fp8_adamw_step
            check(fn(self._params, self.n, lr, beta1, beta2, eps, wd, int(step),
                     inv_loss_scale, fptr, fdev, _stream_ptr(stream)))
        else:
            ndev = None
            if grad_norm_dev is not None:
                ndev = _slot_ptr(grad_norm_dev, 0, "grad_norm_dev")
            nptr = C.byref(self._norm) if sync else None
            check(load().fp8_adam_step_clipped(
                self._params, self.n, lr, beta1, beta2, eps, wd, int(step),
                inv_loss_scale, 1 if l2 else 0, float(max_grad_norm), nptr, ndev,
                fptr, fdev, _stream_ptr(stream)))
            self.last_grad_norm = self._norm.value if nptr is not None else None
        return self._found.value if sync else None

    def step_dev(self, state: StepState, beta1, beta2, eps, wd, l2=False,
                 found_inf_dev: Optional[torch.Tensor] = None,
                 stream=None) -> None:
        """One step with lr, inv_loss_scale and the step count read from
        ``state`` on the device (fp8_adam_step_dev): capturable into a CUDA
        graph that serves every step.  Never waits for the stream; found_inf
        goes to found_inf_dev, if given, and the step count advances on the
        device unless the step was skipped."""
        fdev = None
        if found_inf_dev is not None:
            fdev = _cuda(found_inf_dev, "found_inf_dev").data_ptr()
        check(load().fp8_adam_step_dev(self._params, self.n, beta1, beta2, eps,
                                       wd, 1 if l2 else 0, state.ptr, fdev,
                                       _stream_ptr(stream)))

    def grad_norm(self, inv_loss_scale=1.0, norm_dev=None, sync=True,
                  stream=None):
        """The global L2 norm of the unscaled gradient codes (no step):
        returns (found_inf, norm) with sync=True, else None (the norm is then
        only in norm_dev, a float32 CUDA scalar, if given)."""
        ndev = None if norm_dev is None else _slot_ptr(norm_dev, 0, "norm_dev")
        nptr = C.byref(self._norm) if sync else None
        fptr = C.byref(self._found) if sync else None
        check(load().fp8_grad_norm(self._params, self.n, inv_loss_scale, nptr,
                                   ndev, fptr, _stream_ptr(stream)))
        return (self._found.value, self._norm.value) if sync else None

    # The step split at the exchange between ranks (fp8_grad_norm_terms,
    # fp8_adam_step_begin, fp8_adam_step_finish).  hp = (lr, beta1, beta2,
    # eps, wd, step, inv_loss_scale, l2); clip, found_in: float32 / int32 CUDA
    # scalars or None; terms: float64 CUDA, one per record; found: int32 CUDA
    # scalar out, or None.  None of these waits for the stream.

    def norm_terms(self, inv_loss_scale, terms: torch.Tensor,
                   found: Optional[torch.Tensor] = None, stream=None) -> None:
        if terms.numel() < self.n:
            raise ValueError("terms needs one float64 per record")
        check(load().fp8_grad_norm_terms(
            self._params, self.n, inv_loss_scale,
            _ptr_or_none(terms, "terms", torch.float64),
            _ptr_or_none(found, "found", torch.int32), _stream_ptr(stream)))

    # maxima: int32 CUDA, 2n (begin: out, finish: in; the fp32 bits of each
    # record's first-moment amax, then of its max |g|); master_amax: int32
    # CUDA, n (finish: out, then copy: in), for records that are pieces of
    # tensors cut across ranks.

    def begin(self, hp, clip=None, found=None, stream=None,
              maxima: Optional[torch.Tensor] = None) -> None:
        lr, b1, b2, eps, wd, step, ils, l2 = hp
        if maxima is not None and maxima.numel() < 2 * self.n:
            raise ValueError("maxima needs two int32 per record")
        check(load().fp8_adam_step_begin(
            self._params, self.n, lr, b1, b2, eps, wd, int(step), ils, int(l2),
            _ptr_or_none(clip, "clip", torch.float32),
            _ptr_or_none(found, "found", torch.int32),
            _ptr_or_none(maxima, "maxima", torch.int32), _stream_ptr(stream)))

    def finish(self, hp, clip=None, found_in=None, found=None,
               stream=None, maxima: Optional[torch.Tensor] = None,
               master_amax: Optional[torch.Tensor] = None) -> None:
        lr, b1, b2, eps, wd, step, ils, l2 = hp
        if (maxima is not None and maxima.numel() < 2 * self.n) or (
                master_amax is not None and master_amax.numel() < self.n):
            raise ValueError("maxima needs two and master_amax one int32 per record")
        check(load().fp8_adam_step_finish(
            self._params, self.n, lr, b1, b2, eps, wd, int(step), ils, int(l2),
            _ptr_or_none(clip, "clip", torch.float32),
            _ptr_or_none(found_in, "found_in", torch.int32),
            _ptr_or_none(found, "found", torch.int32),
            _ptr_or_none(maxima, "maxima", torch.int32),
            _ptr_or_none(master_amax, "master_amax", torch.int32),
            _stream_ptr(stream)))

    def copy(self, master_amax: torch.Tensor, stream=None) -> None:
        if master_amax.numel() < self.n:
            raise ValueError("master_amax needs one int32 per record")
        check(load().fp8_adam_step_copy(
            self._params, self.n, _ptr_or_none(master_amax, "master_amax", torch.int32),
            _stream_ptr(stream)))


def fp8_adamw_step(g, g_scale, m, m_scale, v, w, lr, beta1, beta2, eps, wd,
                   step, inv_loss_scale=1.0, w8=None, w8_scale=None,
                   w8_amax=None, g_fmt="e4m3", found_inf_dev=None, sync=True,
                   stream=None):
    """One FP8-state AdamW step over a tensor list; returns found_inf."""
    plan = AdamWPlan(g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax, g_fmt)
    return plan(lr, beta1, beta2, eps, wd, step, inv_loss_scale, found_inf_dev,
                sync, stream)


class CastStepPlan:
    """A marshalled ``fp8_cast_adamw_step``: the cast of ``cast`` and the step
    of ``step`` in one call (one pass fewer over memory).  The cast plan's
    codes and scales must be the step plan's ``g`` and ``g_scale``, with the
    same format; the library checks this and raises otherwise."""

    def __init__(self, cast: CastPlan, step: AdamWPlan):
        if cast.n != step.n:
            raise ValueError("cast and step plans differ in length")
        self.cast = cast
        self.step_plan = step
        self._found = C.c_int(0)
        self._norm = C.c_double(0.0)
        self.last_grad_norm: Optional[float] = None

    def __call__(self, lr, beta1, beta2, eps, wd, step, inv_loss_scale=1.0,
                 found_inf_dev: Optional[torch.Tensor] = None, sync=True,
                 stream=None, l2=False, max_grad_norm=None,
                 grad_norm_dev: Optional[torch.Tensor] = None) -> Optional[int]:
        """AdamW through fp8_cast_adamw_step; with l2 or max_grad_norm (0
        reports the norm without clipping), Adam / AdamW with the gradient
        norm through fp8_cast_adam_step_clipped, the norm then left in
        ``last_grad_norm`` (sync=True) and grad_norm_dev, if given."""
        fdev = None
        if found_inf_dev is not None:
            _cuda(found_inf_dev, "found_inf_dev")
            fdev = found_inf_dev.data_ptr()
        fptr = C.byref(self._found) if sync else None
        if not l2 and max_grad_norm is None:
            check(load().fp8_cast_adamw_step(
                self.cast._items, self.step_plan._params, self.cast.n,
                self.cast.fmt, lr, beta1, beta2, eps, wd, int(step),
                inv_loss_scale, fptr, fdev, _stream_ptr(stream)))
        else:
            ndev = (None if grad_norm_dev is None
                    else _slot_ptr(grad_norm_dev, 0, "grad_norm_dev"))
            nptr = (C.byref(self._norm)
                    if sync and max_grad_norm is not None else None)
            check(load().fp8_cast_adam_step_clipped(
                self.cast._items, self.step_plan._params, self.cast.n,
                self.cast.fmt, lr, beta1, beta2, eps, wd, int(step),
                inv_loss_scale, 1 if l2 else 0,
                0.0 if max_grad_norm is None else float(max_grad_norm), nptr,
                ndev, fptr, fdev, _stream_ptr(stream)))
            self.last_grad_norm = self._norm.value if nptr is not None else None
        return self._found.value if sync else None


    def step_dev(self, state: StepState, beta1, beta2, eps, wd,
                 found_inf_dev: Optional[torch.Tensor] = None, stream=None,
                 l2=False, max_grad_norm=None,
                 grad_norm_dev: Optional[torch.Tensor] = None) -> None:
        """The cast and a step with lr, inv_loss_scale and the step count
        read from ``state`` on the device: AdamW through
        fp8_cast_adamw_step_dev; with l2, max_grad_norm or grad_norm_dev
        through fp8_cast_adam_step_clipped_dev (the norm then in
        grad_norm_dev, a float32 CUDA scalar, if given).  Capturable, never
        waits (see AdamWPlan.step_dev)."""
        fdev = None
        if found_inf_dev is not None:
            fdev = _cuda(found_inf_dev, "found_inf_dev").data_ptr()
        if not l2 and max_grad_norm is None and grad_norm_dev is None:
            check(load().fp8_cast_adamw_step_dev(
                self.cast._items, self.step_plan._params, self.cast.n,
                self.cast.fmt, beta1, beta2, eps, wd, state.ptr, fdev,
                _stream_ptr(stream)))
            return
        ndev = (None if grad_norm_dev is None
                else _slot_ptr(grad_norm_dev, 0, "grad_norm_dev"))
        check(load().fp8_cast_adam_step_clipped_dev(
            self.cast._items, self.step_plan._params, self.cast.n, self.cast.fmt,
            beta1, beta2, eps, wd, 1 if l2 else 0,
            0.0 if max_grad_norm is None else float(max_grad_norm), state.ptr,
            ndev, fdev, _stream_ptr(stream)))


# -------------------------------------------------------------- optimizer

class Fp8AdamW:
    """AdamW over a list of FP16 weights with MS-AMP low-bit state.

    level "O2": FP16 weights updated in place; E4M3 first moment, FP16 second
    moment.  level "O3": the FP16 tensors are master weights, and after each
    step ``w8`` / ``w8_scale`` hold their E4M3 copies for forward/backward.
    ``scaled_v``: the FP16 second moment is kept relative to a per-tensor
    bound (``v_bound``), so small gradients do not underflow it.  ``l2``:
    Adam with L2 weight decay (torch.optim.Adam) instead of AdamW.
    ``max_grad_norm``: clip the unscaled gradient to this global L2 norm
    (torch's clip_grad_norm_; 0 only measures it); ``last_grad_norm`` holds
    the norm after a synchronous step.  With ``fused`` (the default) a step
    is one library call; otherwise the cast and the step are two.

    ``step(grads, inv_loss_scale)`` casts the gradients to FP8 (per-tensor
    just-in-time scale) and runs the update; it returns found_inf and, like a
    GradScaler step, leaves every state tensor and the step count unchanged
    when found_inf is 1.

    ``capturable``: lr, inv_loss_scale and the step count live on the device
    (``self.state``, a StepState), so ``step`` can be captured into a CUDA
    graph once and replayed every step.  ``step`` then never waits: it returns
    None, takes inv_loss_scale from ``self.state`` (write it there) and
    reports found_inf only through found_inf_dev and, with max_grad_norm,
    the norm only through ``grad_norm_dev``.  Set the learning rate with
    ``set_lr``.  With max_grad_norm it needs ``fused``.
    """

    def __init__(self, params: Sequence[torch.Tensor], lr=1e-3,
                 betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01, level="O2",
                 grad_fmt="e4m3", fused=True, scaled_v=False, l2=False,
                 max_grad_norm=None, capturable=False):
        if level not in ("O2", "O3"):
            raise ValueError("level must be 'O2' or 'O3'")
        if capturable and max_grad_norm is not None and not fused:
            raise ValueError("capturable with max_grad_norm needs fused=True")
        self.params = list(params)
        for i, p in enumerate(self.params):
            _cuda(p, f"params[{i}]")
            if p.dtype != torch.float16:
                raise TypeError("params must be float16")
        self.lr, (self.beta1, self.beta2) = lr, betas
        self.eps, self.wd = eps, weight_decay
        self.level, self.grad_fmt = level, grad_fmt
        self.l2 = l2
        self.max_grad_norm = max_grad_norm
        # one call per step: fp8_cast_adamw_step, or fp8_cast_adam_step_clipped
        # with l2 or clipping
        self.fused = fused
        self.last_grad_norm: Optional[float] = None
        self.step_count = 0
        n = len(self.params)
        dev = self.params[0].device if n else torch.device("cuda")
        numels = [p.numel() for p in self.params]
        self.g_codes = arena_views(numels, torch.uint8, dev)
        self.m = arena_views(numels, torch.uint8, dev, fill=0)
        self.v = arena_views(numels, torch.float16, dev, fill=0)
        self.g_amax = torch.zeros(max(n, 1), dtype=torch.float32, device=dev)
        self.g_scale = torch.ones(max(n, 1), dtype=torch.float32, device=dev)
        self.m_scale = torch.ones(max(n, 1), dtype=torch.float32, device=dev)
        w = [p.view(-1) for p in self.params]
        if level == "O3":
            self.w8 = arena_views(numels, torch.uint8, dev, fill=0)
            self.w8_scale = torch.ones(max(n, 1), dtype=torch.float32, device=dev)
            self.w8_amax = torch.zeros(max(n, 1), dtype=torch.float32, device=dev)
        else:
            self.w8 = self.w8_scale = self.w8_amax = None
        self.v_bound = (torch.zeros(max(n, 1), dtype=torch.float32, device=dev)
                        if scaled_v else None)
        self._plan = AdamWPlan(self.g_codes, self.g_scale, self.m, self.m_scale,
                               self.v, w, self.w8, self.w8_scale, self.w8_amax,
                               grad_fmt, self.v_bound)
        self._cast_key = None
        self._cast = None
        self._cast_step = None
        self.capturable = capturable
        self.state = StepState(lr, 1.0, 0, dev) if capturable else None
        self.grad_norm_dev = (torch.zeros(1, dtype=torch.float32, device=dev)
                              if capturable and max_grad_norm is not None
                              else None)

    def set_lr(self, lr: float) -> None:
        """The learning rate of the next step (on the device when
        capturable)."""
        self.lr = lr
        if self.state is not None:
            self.state.lr.fill_(float(lr))

    def _cast_plan(self, grads: Sequence[torch.Tensor]) -> CastPlan:
        key = tuple((g.data_ptr(), g.numel(), g.dtype) for g in grads)
        if key != self._cast_key:
            flat = [g.view(-1) for g in grads]
            self._cast = CastPlan(flat, self.g_codes, self.g_amax, self.g_scale,
                                  self.grad_fmt)
            self._cast_step = CastStepPlan(self._cast, self._plan)
            self._cast_key = key
        return self._cast

    def step(self, grads: Sequence[torch.Tensor], inv_loss_scale=1.0,
             found_inf_dev=None, sync=True, stream=None):
        """Cast ``grads`` to FP8 and apply one AdamW step.  Returns found_inf
        (sync=True) or None (sync=False; the step count then advances
        unconditionally and the caller reads found_inf_dev)."""
        if len(grads) != len(self.params):
            raise ValueError("one gradient per parameter")
        cast = self._cast_plan(grads)
        if self.capturable:
            if inv_loss_scale != 1.0:
                raise ValueError("capturable: write inv_loss_scale into "
                                 "self.state.inv_loss_scale")
            # fused: one call (AdamW, or Adam-L2 / clipping through the
            # clipped form); fused=False: the cast, then the step
            if self.fused:
                self._cast_step.step_dev(self.state, self.beta1, self.beta2,
                                         self.eps, self.wd, found_inf_dev, stream,
                                         l2=self.l2,
                                         max_grad_norm=self.max_grad_norm,
                                         grad_norm_dev=self.grad_norm_dev)
            else:
                cast(stream)
                self._plan.step_dev(self.state, self.beta1, self.beta2, self.eps,
                                    self.wd, self.l2, found_inf_dev, stream)
            return None
        t = self.step_count + 1
        if self.fused:
            found = self._cast_step(self.lr, self.beta1, self.beta2, self.eps,
                                    self.wd, t, inv_loss_scale, found_inf_dev,
                                    sync, stream, l2=self.l2,
                                    max_grad_norm=self.max_grad_norm)
            self.last_grad_norm = self._cast_step.last_grad_norm
        else:
            cast(stream)
            found = self._plan(self.lr, self.beta1, self.beta2, self.eps, self.wd,
                               t, inv_loss_scale, found_inf_dev, sync, stream,
                               l2=self.l2, max_grad_norm=self.max_grad_norm)
            self.last_grad_norm = self._plan.last_grad_norm
        if not sync or found == 0:
            self.step_count = t
        return found

    def state_dict(self) -> Dict[str, object]:
        if self.state is not None:
            self.step_count = int(self.state.step.item())
            self.lr = float(self.state.lr.item())
        d = {"step": self.step_count, "level": self.level,
             "grad_fmt": self.grad_fmt,
             "hparams": (self.lr, self.beta1, self.beta2, self.eps, self.wd),
             "m": [t.clone() for t in self.m], "v": [t.clone() for t in self.v],
             "m_scale": self.m_scale.clone(), "l2": self.l2,
             "max_grad_norm": self.max_grad_norm,
             "v_bound": None if self.v_bound is None else self.v_bound.clone()}
        if self.level == "O3":
            d["w8"] = [t.clone() for t in self.w8]
            d["w8_scale"] = self.w8_scale.clone()
            d["w8_amax"] = self.w8_amax.clone()
        return d

    def load_state_dict(self, d: Dict[str, object]) -> None:
        if d["level"] != self.level or len(d["m"]) != len(self.m):
            raise ValueError("state dict does not match this optimizer")
        self.step_count = int(d["step"])
        self.lr, self.beta1, self.beta2, self.eps, self.wd = d["hparams"]
        if self.state is not None:
            self.state.step.fill_(self.step_count)
            self.state.lr.fill_(float(self.lr))
        for dst, src in zip(self.m, d["m"]):
            dst.copy_(src)
        for dst, src in zip(self.v, d["v"]):
            dst.copy_(src)
        self.m_scale.copy_(d["m_scale"])
        if (d.get("v_bound") is None) != (self.v_bound is None):
            raise ValueError("state dict and optimizer differ in scaled_v")
        if self.v_bound is not None:
            self.v_bound.copy_(d["v_bound"])
        if self.level == "O3":
            for dst, src in zip(self.w8, d["w8"]):
                dst.copy_(src)
            self.w8_scale.copy_(d["w8_scale"])
            self.w8_amax.copy_(d["w8_amax"])

    @staticmethod
    def state_bytes_per_param(level="O2") -> int:
        """Optimizer-state bytes per parameter: 1 (E4M3 m) + 2 (FP16 v)."""
        return 1 + 2


def norm_terms_from_limbs(limbs: torch.Tensor, amax_bits: torch.Tensor, fmt,
                          inv_loss_scale: float, terms: torch.Tensor,
                          stream=None) -> None:
    """fp8_norm_terms_from_limbs: the norm term of every tensor (float64 CUDA,
    one per tensor) from its exact sum of squares as limbs (int64 CUDA, four
    per tensor, possibly summed over ranks) and its reduced codes' amax
    (int32 CUDA, fp32 bits, one per tensor)."""
    n = terms.numel()
    if limbs.numel() < 4 * n or amax_bits.numel() < n:
        raise ValueError("limbs needs four int64 and amax_bits one int32 per term")
    check(load().fp8_norm_terms_from_limbs(
        _ptr_or_none(limbs, "limbs", torch.int64),
        _ptr_or_none(amax_bits, "amax_bits", torch.int32), n, _fmt(fmt),
        inv_loss_scale, _ptr_or_none(terms, "terms", torch.float64),
        _stream_ptr(stream)))


def clip_coef(terms: torch.Tensor, max_grad_norm: float, clip: torch.Tensor,
              norm: Optional[torch.Tensor] = None,
              found: Optional[torch.Tensor] = None, stream=None) -> None:
    """fp8_clip_coef: the global norm (float64 CUDA scalar, optional) and the
    clip coefficient (float32 CUDA scalar) from the terms of every record
    (float64 CUDA, in record order); found (int32 CUDA scalar, optional)
    nonzero makes the norm +inf."""
    check(load().fp8_clip_coef(
        _ptr_or_none(terms, "terms", torch.float64), terms.numel(),
        _ptr_or_none(found, "found", torch.int32), float(max_grad_norm),
        _ptr_or_none(norm, "norm", torch.float64),
        _ptr_or_none(clip, "clip", torch.float32), _stream_ptr(stream)))
