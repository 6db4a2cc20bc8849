"""Data-parallel sharding of the FP8 optimizer step (ZeRO-1 style).

MS-AMP's O3 level keeps an FP16 master weight per parameter and an FP8 weight
for forward/backward, and broadcasts the 8-bit weights (the "Optimization
Level" page, O3 paragraph).  Here every rank owns the optimizer state (E4M3
first moment, FP16 second moment, FP16 master) of a contiguous range of whole
tensors, balanced by size; a step on each rank is

  1. the FP8 cast of its local gradients, an all-to-all that brings every
     tensor's codes from all ranks to its owner, and the FP8 mean of those
     shards (with clipping, that reduction also gives the owned tensors' norm
     terms and found_inf);
  2. the step's first pass over its own tensors (``begin``), giving found_inf;
  3. one exchange: found_inf MAX over ranks (and, with clipping, the per-tensor
     norm terms, each held by exactly one rank, summed so every rank holds all
     of them and takes the same norm and clip coefficient);
  4. the update and the O3 weight copy of its own tensors (``finish``), skipped
     on every rank when any rank found a non-finite gradient;
  5. the E4M3 weight copies and their scales broadcast from their owners.

Because the partition is tensor-aligned, every per-tensor quantity (amax,
scale, bound) is computed whole on one rank, and the result on every rank is
the unsharded step's, bit for bit.

The collectives are torch.distributed calls on an initialised process group
(NCCL between GPUs; gloo works for host-side tests).  The arithmetic is behind
an engine object: ``LibEngine`` calls the CUDA library; tests may pass another
engine with the same methods.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple


def partition(numels: Sequence[int], world: int) -> List[Tuple[int, int]]:
    """Contiguous, tensor-aligned ranges [lo, hi) of the tensor list, one per
    rank in rank order, that minimise the largest rank's element count (every
    tensor of a step moves the same bytes per element, so this balances
    bytes).  Ranks past the last tensor get empty ranges.  Deterministic:
    every rank computes the same answer."""
    if world < 1:
        raise ValueError("world must be >= 1")
    n = len(numels)
    if any(x < 0 for x in numels):
        raise ValueError("negative numel")
    # the smallest capacity whose greedy packing fits in `world` ranges
    w = [max(int(x), 1) for x in numels]   # an empty tensor still has a record

    def fits(cap):
        parts, load = 1, 0
        for x in w:
            if x > cap:
                return False
            if load + x > cap:
                parts += 1
                load = x
            else:
                load += x
        return parts <= world

    lo, hi = max(w, default=1), max(sum(w), 1)
    while lo < hi:
        mid = (lo + hi) // 2
        if fits(mid):
            hi = mid
        else:
            lo = mid + 1
    cap = lo
    ranges, start, load = [], 0, 0
    for i, x in enumerate(w):
        if load + x > cap and i > start:
            ranges.append((start, i))
            start, load = i, 0
        load += x
    ranges.append((start, n))
    while len(ranges) < world:
        ranges.append((n, n))
    return ranges


# ------------------------------------------------------------ collectives

class TorchDistComm:
    """The sharded step's collectives on a torch.distributed process group
    (NCCL for CUDA tensors, gloo for host tensors)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self._dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_to_all(self, out, inp, out_splits, in_splits):
        self._dist.all_to_all_single(out, inp, list(out_splits), list(in_splits),
                                     group=self.group)

    def all_reduce_sum(self, t):
        self._dist.all_reduce(t, op=self._dist.ReduceOp.SUM, group=self.group)

    def all_reduce_max(self, t):
        self._dist.all_reduce(t, op=self._dist.ReduceOp.MAX, group=self.group)

    def broadcast(self, t, src):
        self._dist.broadcast(t, src=self._dist.get_global_rank(self.group, src)
                             if self.group is not None else src,
                             group=self.group)


# ------------------------------------------------------------------ engine

class LibEngine:
    """The sharded step's arithmetic through the CUDA library: each factory
    returns the binding's plan over fixed buffers."""

    def make_cast(self, srcs, codes, amax, scale, fmt):
        from .api import CastPlan
        return CastPlan(srcs, codes, amax, scale, fmt)

    def make_reduce(self, shards, scales, codes, amax, scale, in_fmt, out_fmt,
                    post):
        from .api import ReducePlan
        return ReducePlan(shards, scales, codes, amax, scale, in_fmt, out_fmt,
                          post)

    def make_step(self, g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                  g_fmt, v_bound):
        from .api import AdamWPlan
        return AdamWPlan(g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                         g_fmt, v_bound)

    def clip_coef(self, terms, max_grad_norm, clip, norm, found):
        from .api import clip_coef
        clip_coef(terms, max_grad_norm, clip, norm, found)


# ------------------------------------------------------------ the step loop

def _offsets(views, base) -> List[int]:
    """Element offsets of arena views in their base buffer."""
    isz = base.element_size()
    return [(v.data_ptr() - base.data_ptr()) // isz for v in views]


class ShardedFp8AdamW:
    """One rank of the data-parallel FP8 optimizer step (MS-AMP O2 / O3 with
    ZeRO-1 sharding of the optimizer state).

    weights: every tensor's FP16 weight (the same on every rank); they are
    copied into the optimizer's flat arena, whose views ``weights`` the
    forward pass uses (O2), or which holds the FP16 masters of this rank's
    tensors (O3; the E4M3 copies of all tensors are ``w8`` / ``w8_scale``).

    ``step(grads)`` takes this rank's local gradients of every tensor (BF16,
    FP16 or FP32), casts them to FP8 (per-tensor just-in-time scales), sends
    each tensor's codes to its owner (one all-to-all of the codes and one of
    the scales), reduces the ranks' shards to their mean in FP8, and steps the
    owned tensors.  found_inf is combined over ranks (every rank skips
    together) and, with ``max_grad_norm``, the gradient is clipped to a
    global L2 norm taken over every rank's tensors.  The owners then
    broadcast the new FP16 weights (O2) or E4M3 weights and scales (O3).
    """

    def __init__(self, weights: Sequence, comm, lr=1e-3, betas=(0.9, 0.999),
                 eps=1e-8, weight_decay=0.01, level="O2", grad_fmt="e4m3",
                 l2=False, scaled_v=False, max_grad_norm=None, engine=None,
                 device=None):
        import torch
        from .api import arena_views
        if level not in ("O2", "O3"):
            raise ValueError("level must be 'O2' or 'O3'")
        self.comm = comm
        self.engine = engine if engine is not None else LibEngine()
        self.rank, self.world = comm.rank, comm.world
        self.lr, (self.beta1, self.beta2) = lr, betas
        self.eps, self.wd = eps, weight_decay
        self.level, self.grad_fmt, self.l2 = level, grad_fmt, l2
        self.max_grad_norm = max_grad_norm
        self.step_count = 0
        self.last_grad_norm: Optional[float] = None
        weights = list(weights)
        dev = device if device is not None else (weights[0].device if weights
                                                 else torch.device("cuda"))
        self.device = dev
        numels = [int(w.numel()) for w in weights]
        self.numels = numels
        n = len(numels)
        self.n = n
        self.ranges = partition(numels, self.world)
        lo, hi = self.ranges[self.rank]
        self.own = (lo, hi)
        f32 = dict(dtype=torch.float32, device=dev)

        # every tensor: weights (O2) / masters (O3) and the local cast codes
        self.weights, self._w_flat = arena_views(numels, torch.float16, dev,
                                                 return_base=True)
        for dst, src in zip(self.weights, weights):
            dst.copy_(src.reshape(-1))
        self._gc, self._gc_flat = arena_views(numels, torch.uint8, dev,
                                              return_base=True)
        self._g_amax = torch.zeros(max(n, 1), **f32)
        self._g_scale = torch.ones(max(n, 1), **f32)
        # element offsets (the same in every uint8 / float16 arena: both pad
        # each tensor to 256 bytes, i.e. 256 and 128 elements)
        off8 = _offsets(self._gc, self._gc_flat) + [self._gc_flat.numel()]
        off16 = _offsets(self.weights, self._w_flat) + [self._w_flat.numel()]
        if n:
            off8[-1] = off8[n - 1] + -(-numels[n - 1] // 256) * 256
            off16[-1] = off16[n - 1] + -(-numels[n - 1] // 128) * 128
        self._off8, self._off16 = off8, off16
        self._bytes = [off8[b] - off8[a] for a, b in self.ranges]
        self._counts = [b - a for a, b in self.ranges]
        own_bytes = self._bytes[self.rank]
        n_own = hi - lo

        # the shards of this rank's tensors from every rank, and their scales
        self._recv = torch.zeros(max(self.world * own_bytes, 1), dtype=torch.uint8,
                                 device=dev)
        self._recv_scale = torch.ones(max(self.world * n_own, 1), **f32)
        self._scale_t = torch.ones((max(n_own, 1), self.world), **f32)
        rows = self._recv[:self.world * own_bytes].view(self.world, own_bytes)
        shards = [rows[:, off8[t] - off8[lo]: off8[t] - off8[lo] + numels[t]]
                  for t in range(lo, hi)]
        own_numels = numels[lo:hi]
        self._g_own = arena_views(own_numels, torch.uint8, dev)
        self._g_own_amax = torch.zeros(max(n_own, 1), **f32)
        self._g_own_scale = torch.ones(max(n_own, 1), **f32)
        self._reduce = self.engine.make_reduce(
            shards, [self._scale_t[j] for j in range(n_own)], self._g_own,
            self._g_own_amax, self._g_own_scale, grad_fmt, grad_fmt,
            1.0 / self.world)

        # this rank's optimizer state
        self.m = arena_views(own_numels, torch.uint8, dev, fill=0)
        self.v = arena_views(own_numels, torch.float16, dev, fill=0)
        self.m_scale = torch.ones(max(n_own, 1), **f32)
        self.v_bound = torch.zeros(max(n_own, 1), **f32) if scaled_v else None
        if level == "O3":
            self.w8, self._w8_flat = arena_views(numels, torch.uint8, dev, fill=0,
                                                 return_base=True)
            self.w8_scale = torch.ones(max(n, 1), **f32)
            self.w8_amax = torch.zeros(max(n, 1), **f32)
            w8_own = self.w8[lo:hi]
            w8s, w8a = self.w8_scale[lo:max(hi, lo + 1)], self.w8_amax[lo:max(hi, lo + 1)]
        else:
            self.w8 = self.w8_scale = self.w8_amax = None
            w8_own = w8s = w8a = None
        self._step = self.engine.make_step(
            self._g_own, self._g_own_scale, self.m, self.m_scale, self.v,
            self.weights[lo:hi], w8_own, w8s, w8a, grad_fmt, self.v_bound)
        self._found = torch.zeros(1, dtype=torch.int32, device=dev)
        self._found_out = torch.zeros(1, dtype=torch.int32, device=dev)
        self._terms = torch.zeros(max(n, 1), dtype=torch.float64, device=dev)
        self._norm = torch.zeros(1, dtype=torch.float64, device=dev)
        self._clip = torch.ones(1, **f32)
        self._cast_key = None
        self._cast = None

    def _cast_plan(self, grads):
        key = tuple((g.data_ptr(), g.numel(), g.dtype) for g in grads)
        if key != self._cast_key:
            self._cast = self.engine.make_cast([g.reshape(-1) for g in grads],
                                               self._gc, self._g_amax,
                                               self._g_scale, self.grad_fmt)
            self._cast_key = key
        return self._cast

    def step(self, grads: Sequence, inv_loss_scale=1.0) -> int:
        """One data-parallel step from this rank's local gradients; returns
        found_inf (combined over ranks)."""
        if len(grads) != self.n:
            raise ValueError("one gradient per tensor")
        lo, hi = self.own
        comm, world = self.comm, self.world
        t = self.step_count + 1
        hp = (self.lr, self.beta1, self.beta2, self.eps, self.wd, t,
              inv_loss_scale, self.l2)
        # 1. FP8 cast of every local gradient
        self._cast_plan(grads)()
        # 2. each tensor's codes and scale to its owner
        total = self._off8[self.n] if self.n else 0
        comm.all_to_all(self._recv[:world * self._bytes[self.rank]],
                        self._gc_flat[:total],
                        [self._bytes[self.rank]] * world, self._bytes)
        n_own = hi - lo
        comm.all_to_all(self._recv_scale[:world * n_own], self._g_scale[:self.n],
                        [n_own] * world, self._counts)
        if n_own:
            self._scale_t[:n_own].copy_(
                self._recv_scale[:world * n_own].view(world, n_own).t())
        # 3. the mean of the ranks' shards, re-encoded (with clipping, the
        #    encode pass also gives the owned tensors' norm terms)
        clip = None
        if self.max_grad_norm is not None:
            self._terms.zero_()
            self._reduce(norm_terms=self._terms[lo:max(hi, lo + 1)],
                         found=self._found, inv_loss_scale=inv_loss_scale)
        else:
            self._reduce()
        # 4. found_inf (and the global norm) over ranks, then the step
        if self.max_grad_norm is not None:
            comm.all_reduce_sum(self._terms)
            comm.all_reduce_max(self._found)
            self.engine.clip_coef(self._terms[:self.n], self.max_grad_norm,
                                  self._clip, self._norm, self._found)
            clip = self._clip
            self._step.begin(hp, clip, None)
        else:
            self._step.begin(hp, None, self._found)
            comm.all_reduce_max(self._found)
        self._step.finish(hp, clip, self._found, self._found_out)
        # 5. the owners' new weights to every rank
        for r, (a, b) in enumerate(self.ranges):
            if a == b:
                continue
            if self.level == "O3":
                comm.broadcast(self._w8_flat[self._off8[a]:self._off8[b]], r)
                comm.broadcast(self.w8_scale[a:b], r)
                comm.broadcast(self.w8_amax[a:b], r)
            else:
                comm.broadcast(self._w_flat[self._off16[a]:self._off16[b]], r)
        found = int(self._found_out.item())
        if self.max_grad_norm is not None:
            self.last_grad_norm = float(self._norm.item())
        if found == 0:
            self.step_count = t
        return found
