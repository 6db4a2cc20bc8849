"""Data-parallel sharding of the FP8 optimizer step (ZeRO-1 style).

MS-AMP's O3 level keeps an FP16 master weight per parameter and an FP8 weight
for forward/backward, names ZeRO among the strategies it supports, and
broadcasts the 8-bit weights (the "Optimization Level" page, O3 paragraph).
Here the tensors of the list are laid end to end in one element space, each
from a 256-element boundary, and rank r owns the optimizer state (E4M3 first
moment, FP16 second moment, FP16 master) of the elements [r*S, (r+1)*S) of
that space: every rank holds the same number of elements, and a tensor that
crosses a segment boundary is cut into pieces on two or more ranks.  A step
on each rank is

  1. the FP8 cast of its local gradients of every tensor, one all-to-all that
     sends every rank its segment of the codes, and an all-gather of the
     per-tensor scales;
  2. the FP8 mean of the ranks' shards of its pieces, in two passes: each
     piece's amax, combined per tensor by MAX over ranks, then the encode with
     the whole tensor's amax (with clipping, the encode also gives each
     piece's exact sum of squares, combined per tensor by an exact SUM over
     ranks, so that every rank takes the same norm and clip coefficient);
  3. the step's first pass over its pieces; per tensor, the amax of the new
     first moment and max |g| combined by MAX over ranks, with found_inf;
  4. the update of its pieces with the whole tensors' maxima, skipped on every
     rank when any rank found a non-finite gradient; for O3 the new masters'
     amax combined by MAX, then the E4M3 weight copy;
  5. one all-gather that returns every rank's segment of the new FP16 weights
     (O2) or E4M3 weights (O3, their per-tensor scales combined by MAX).

Every per-tensor quantity is therefore the whole tensor's, and the result on
every rank is the unsharded pipeline's, bit for bit.  On one rank a step is
the cast and the step in one call (no exchange, no reduction).

The collectives are torch.distributed calls on an initialised process group
(NCCL between GPUs; gloo works for host-side tests).  The arithmetic is behind
an engine object: ``LibEngine`` calls the CUDA library; tests may pass another
engine with the same methods.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

ALIGN = 256   # elements: 256 B of codes, 512 B of FP16


def layout(numels: Sequence[int], world: int, align: int = ALIGN):
    """The element space of a tensor list for `world` ranks.

    Returns (off, seg, pieces): tensor t starts at element off[t] (a multiple
    of `align`; tensors follow one another in list order, each padded to a
    multiple of `align`); every rank owns `seg` elements (a multiple of
    `align`, world * seg covering the space), rank r the range [r*seg,
    (r+1)*seg); pieces[r] lists rank r's (tensor, a, b), the tensor's
    elements [a, b) inside that range, in tensor order.  An empty tensor is a
    piece (t, 0, 0) of the rank whose range holds its offset, so that its
    per-tensor outputs are written.  Deterministic: every rank computes the
    same answer."""
    if world < 1:
        raise ValueError("world must be >= 1")
    if any(int(x) < 0 for x in numels):
        raise ValueError("negative numel")
    off, pos = [], 0
    for x in numels:
        off.append(pos)
        pos += -(-int(x) // align) * align
    share = -(-pos // world)
    seg = max(align, -(-share // align) * align)
    pieces: List[List[Tuple[int, int, int]]] = [[] for _ in range(world)]
    for t, x in enumerate(numels):
        x = int(x)
        if x == 0:
            pieces[min(off[t] // seg, world - 1)].append((t, 0, 0))
            continue
        for r in range(off[t] // seg, (off[t] + x - 1) // seg + 1):
            pieces[r].append((t, max(0, r * seg - off[t]),
                              min(x, (r + 1) * seg - off[t])))
    return off, seg, pieces


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

    def all_gather(self, out, inp):
        """out = the ranks' inp, concatenated in rank order (inp may be this
        rank's part of out)."""
        self._dist.all_gather_into_tensor(out, inp, group=self.group)

    def all_reduce_sum(self, t):
        self._dist.all_reduce(t, op=self._dist.ReduceOp.SUM, group=self.group)

    def all_reduce_max(self, t):
        self._dist.all_reduce(t, op=self._dist.ReduceOp.MAX, group=self.group)


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

    def make_cast_step(self, cast, step):
        from .api import CastStepPlan
        return CastStepPlan(cast, step)

    def norm_terms_from_limbs(self, limbs, amax_bits, fmt, inv_loss_scale, terms):
        from .api import norm_terms_from_limbs
        norm_terms_from_limbs(limbs, amax_bits, fmt, inv_loss_scale, terms)

    def clip_coef(self, terms, max_grad_norm, clip, norm, found):
        from .api import clip_coef
        clip_coef(terms, max_grad_norm, clip, norm, found)


# ------------------------------------------------------------ the step loop

class ShardedFp8AdamW:
    """One rank of the data-parallel FP8 optimizer step (MS-AMP O2 / O3 with
    ZeRO-1 sharding of the optimizer state over equal element ranges).

    weights: every tensor's FP16 weight (the same on every rank); they are
    copied into the optimizer's flat arena, whose views ``weights`` the
    forward pass uses (O2), or which holds the FP16 masters of this rank's
    pieces (O3; the E4M3 copies of all tensors are ``w8`` / ``w8_scale``).
    ``pieces`` lists this rank's (tensor, a, b); ``m``, ``v``, ``m_scale``
    (and ``v_bound``) hold their optimizer state, one entry per piece.

    ``step(grads)`` takes this rank's local gradients of every tensor (BF16,
    FP16 or FP32) and runs the step of the module docstring; found_inf is
    combined over ranks (every rank skips together) and, with
    ``max_grad_norm``, the gradient is clipped to a global L2 norm taken over
    every rank's pieces.
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
        self.off, self.seg, self.layout_pieces = layout(numels, self.world)
        self.pieces = self.layout_pieces[self.rank]
        world, seg, off, rank = self.world, self.seg, self.off, self.rank
        space = world * seg
        f32 = dict(dtype=torch.float32, device=dev)
        i32 = dict(dtype=torch.int32, device=dev)

        # every tensor in the element space: FP16 weights (O2) / masters
        # (O3), the local cast codes, and (O3) the E4M3 weight copies
        self._w_flat = torch.zeros(space, dtype=torch.float16, device=dev)
        self.weights = [self._w_flat[off[t]:off[t] + numels[t]] for t in range(n)]
        for dst, src in zip(self.weights, weights):
            dst.copy_(src.reshape(-1))
        self._gc_flat = torch.zeros(space, dtype=torch.uint8, device=dev)
        self._gc = [self._gc_flat[off[t]:off[t] + numels[t]] for t in range(n)]
        self._g_amax = torch.zeros(max(n, 1), **f32)
        self._g_scale = torch.ones(max(n, 1), **f32)
        o3 = level == "O3"
        if o3:
            self._w8_flat = torch.zeros(space, dtype=torch.uint8, device=dev)
            self.w8 = [self._w8_flat[off[t]:off[t] + numels[t]] for t in range(n)]
            self.w8_scale = torch.ones(max(n, 1), **f32)
            self.w8_amax = torch.zeros(max(n, 1), **f32)
        else:
            self.w8 = self.w8_scale = self.w8_amax = None
        self._found = torch.zeros(1, **i32)
        self._found_out = torch.zeros(1, **i32)
        self._cast_key = None
        self._cast = None
        self._fused, self._fused_for = None, None

        pieces = self.pieces
        npc = len(pieces)
        sizes = [b - a for _, a, b in pieces]
        self.m = arena_views(sizes, torch.uint8, dev, fill=0)
        self.v = arena_views(sizes, torch.float16, dev, fill=0)
        self.m_scale = torch.ones(max(npc, 1), **f32)
        self.v_bound = torch.zeros(max(npc, 1), **f32) if scaled_v else None
        w_pieces = [self._w_flat[off[t] + a:off[t] + b] for t, a, b in pieces]
        if world == 1:
            # one rank: the cast's codes and scales feed the step directly
            self._step = self.engine.make_step(
                self._gc, self._g_scale, self.m, self.m_scale, self.v, w_pieces,
                self.w8 if o3 else None, self.w8_scale, self.w8_amax, grad_fmt,
                self.v_bound)
            return

        self._piece_t = torch.tensor([t for t, _, _ in pieces] or [0],
                                     dtype=torch.int64, device=dev)[:npc]
        # every rank's codes of this rank's segment, and every rank's scales
        self._recv = torch.zeros(space, dtype=torch.uint8, device=dev)
        rows = self._recv.view(world, seg)
        shards = [rows[:, off[t] + a - rank * seg:off[t] + b - rank * seg]
                  for t, a, b in pieces]
        self._scales_all = torch.ones(world * max(n, 1), **f32)
        self._scales_t = torch.ones((max(n, 1), world), **f32)
        self._g_own = arena_views(sizes, torch.uint8, dev)
        self._g_own_amax = torch.zeros(max(npc, 1), **f32)
        self._g_own_scale = torch.ones(max(npc, 1), **f32)
        self._reduce = self.engine.make_reduce(
            shards, [self._scales_t[t] for t, _, _ in pieces], self._g_own,
            self._g_own_amax, self._g_own_scale, grad_fmt, grad_fmt, 1.0 / world)
        if o3:
            w8_pieces = [self._w8_flat[off[t] + a:off[t] + b] for t, a, b in pieces]
            self._w8s_own = torch.ones(max(npc, 1), **f32)
            self._w8a_own = torch.zeros(max(npc, 1), **f32)
        else:
            w8_pieces = self._w8s_own = self._w8a_own = None
        self._step = self.engine.make_step(
            self._g_own, self._g_own_scale, self.m, self.m_scale, self.v,
            w_pieces, w8_pieces, self._w8s_own, self._w8a_own, grad_fmt,
            self.v_bound)
        # exchange buffers: per piece (local) and per tensor (exchanged)
        self._amax_local = torch.zeros(max(npc, 1), **i32)
        self._amax_vec = torch.zeros(max(n, 1), **i32)
        self._maxima_local = torch.zeros(2 * max(npc, 1), **i32)
        self._maxima_vec = torch.zeros(2 * n + 1, **i32)
        self._limbs_local = torch.zeros(4 * max(npc, 1), dtype=torch.int64, device=dev)
        self._limbs_vec = torch.zeros(4 * n + 1, dtype=torch.int64, device=dev)
        self._master_local = torch.zeros(max(npc, 1), **i32)
        self._master_vec = torch.zeros(max(n, 1), **i32)
        self._w8_vec = torch.zeros(2 * max(n, 1), **i32)
        self._terms = torch.zeros(max(n, 1), dtype=torch.float64, device=dev)
        self._norm = torch.zeros(1, dtype=torch.float64, device=dev)
        self._clip = torch.ones(1, **f32)

    def state_dict(self) -> dict:
        """This rank's optimizer state: its pieces' E4M3 first moments, FP16
        second moments, their scales (and second-moment bounds); for O3 the
        FP16 masters of its pieces and every tensor's E4M3 weight copy with
        its scale and amax; the step count and hyperparameters; and the
        layout the state belongs to (ranks, this rank, the tensors' sizes),
        which load_state_dict checks.  The O2 weights are the model's: every
        rank holds all of them after a step."""
        d = {"step": self.step_count, "level": self.level,
             "grad_fmt": self.grad_fmt,
             "hparams": (self.lr, self.beta1, self.beta2, self.eps, self.wd),
             "l2": self.l2, "max_grad_norm": self.max_grad_norm,
             "world": self.world, "rank": self.rank,
             "numels": list(self.numels), "pieces": list(self.pieces),
             "m": [t.clone() for t in self.m], "v": [t.clone() for t in self.v],
             "m_scale": self.m_scale.clone(),
             "v_bound": None if self.v_bound is None else self.v_bound.clone()}
        if self.level == "O3":
            off = self.off
            d["master"] = [self._w_flat[off[t] + a:off[t] + b].clone()
                           for t, a, b in self.pieces]
            d["w8"] = [t.clone() for t in self.w8]
            d["w8_scale"] = self.w8_scale.clone()
            d["w8_amax"] = self.w8_amax.clone()
        return d

    def load_state_dict(self, d: dict) -> None:
        """Restores a state_dict of the same rank of the same layout (level,
        number of ranks, tensor sizes); raises ValueError otherwise."""
        if (d["level"] != self.level or d["world"] != self.world or
                d["rank"] != self.rank or list(d["numels"]) != self.numels or
                [tuple(p) for p in d["pieces"]] != [tuple(p) for p in self.pieces]):
            raise ValueError("state dict does not match this optimizer's level, "
                             "ranks or tensors")
        if (d.get("v_bound") is None) != (self.v_bound is None):
            raise ValueError("state dict and optimizer differ in scaled_v")
        self.step_count = int(d["step"])
        self.lr, self.beta1, self.beta2, self.eps, self.wd = d["hparams"]
        for dst, src in zip(self.m, d["m"]):
            dst.copy_(src)
        for dst, src in zip(self.v, d["v"]):
            dst.copy_(src)
        self.m_scale.copy_(d["m_scale"])
        if self.v_bound is not None:
            self.v_bound.copy_(d["v_bound"])
        if self.level == "O3":
            off = self.off
            for (t, a, b), src in zip(self.pieces, d["master"]):
                self._w_flat[off[t] + a:off[t] + b].copy_(src)
            for dst, src in zip(self.w8, d["w8"]):
                dst.copy_(src)
            self.w8_scale.copy_(d["w8_scale"])
            self.w8_amax.copy_(d["w8_amax"])

    def _cast_plan(self, grads):
        key = tuple((g.data_ptr(), g.numel(), g.dtype) for g in grads)
        if key != self._cast_key:
            self._cast = self.engine.make_cast([g.reshape(-1) for g in grads],
                                               self._gc, self._g_amax,
                                               self._g_scale, self.grad_fmt)
            self._cast_key = key
        return self._cast

    def _max_over_ranks(self, local, vec, parts=1, flag=None):
        """Per-tensor MAX over ranks of per-piece int32 values: `parts`
        blocks of one value per piece in `local` go to their tensors' slots
        in `vec` (zero elsewhere, below every value), the ranks' vectors are
        combined by MAX in one collective, and each piece takes its tensor's
        result back.  flag (an int32 scalar, optional) rides along in the
        entry after the blocks and takes the MAX over ranks too."""
        n, npc, idx = self.n, len(self.pieces), self._piece_t
        vec.zero_()
        for j in range(parts):
            vec[j * n:(j + 1) * n].index_copy_(0, idx, local[j * npc:(j + 1) * npc])
        if flag is not None:
            vec[parts * n:parts * n + 1].copy_(flag)
        self.comm.all_reduce_max(vec)
        for j in range(parts):
            local[j * npc:(j + 1) * npc].copy_(vec[j * n:(j + 1) * n].index_select(0, idx))
        if flag is not None:
            flag.copy_(vec[parts * n:parts * n + 1])

    def step(self, grads: Sequence, inv_loss_scale=1.0) -> int:
        """One data-parallel step from this rank's local gradients; returns
        found_inf (combined over ranks)."""
        if len(grads) != self.n:
            raise ValueError("one gradient per tensor")
        if self.n == 0:
            return 0
        t = self.step_count + 1
        hp = (self.lr, self.beta1, self.beta2, self.eps, self.wd, t,
              inv_loss_scale, self.l2)
        cast = self._cast_plan(grads)
        found = (self._step_one_rank(cast, hp) if self.world == 1
                 else self._step_ranks(cast, hp))
        if found == 0:
            self.step_count = t
        return found

    def _step_one_rank(self, cast, hp) -> int:
        if self._fused_for is not cast:
            self._fused = self.engine.make_cast_step(cast, self._step)
            self._fused_for = cast
        lr, b1, b2, eps, wd, t, ils, l2 = hp
        found = self._fused(lr, b1, b2, eps, wd, t, ils,
                            found_inf_dev=self._found_out, l2=l2,
                            max_grad_norm=self.max_grad_norm)
        if self.max_grad_norm is not None:
            self.last_grad_norm = self._fused.last_grad_norm
        return int(found)

    def _step_ranks(self, cast, hp) -> int:
        import torch
        comm, world, seg, rank, n = self.comm, self.world, self.seg, self.rank, self.n
        npc = len(self.pieces)
        ils = hp[6]
        clipped = self.max_grad_norm is not None
        # 1. FP8 cast of every local gradient; each rank's segment of the
        #    codes to it; every rank's per-tensor scales to every rank
        cast()
        comm.all_to_all(self._recv, self._gc_flat, [seg] * world, [seg] * world)
        comm.all_gather(self._scales_all[:world * n], self._g_scale[:n])
        self._scales_t[:n].copy_(self._scales_all[:world * n].view(world, n).t())
        # 2. the FP8 mean of the ranks' shards: pieces' amax, MAX per tensor,
        #    then the encode (with clipping, the exact sums and found_inf)
        self._reduce.begin(self._amax_local)
        self._max_over_ranks(self._amax_local, self._amax_vec)
        clip = None
        self._found.zero_()
        if clipped:
            self._reduce.finish(self._amax_local, ils, self._limbs_local, self._found)
            vec = self._limbs_vec
            vec.zero_()
            vec[:4 * n].view(n, 4).index_copy_(
                0, self._piece_t, self._limbs_local[:4 * npc].view(npc, 4))
            vec[4 * n:].copy_(self._found)
            comm.all_reduce_sum(vec)
            self._found.copy_((vec[4 * n:] != 0).to(torch.int32))
            self.engine.norm_terms_from_limbs(vec[:4 * n], self._amax_vec[:n],
                                              self.grad_fmt, ils, self._terms[:n])
            self.engine.clip_coef(self._terms[:n], self.max_grad_norm, self._clip,
                                  self._norm, self._found)
            clip = self._clip
        else:
            self._reduce.finish(self._amax_local)
        # 3. the first pass; the maxima and found_inf over ranks
        found_local = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._step.begin(hp, clip, found_local, maxima=self._maxima_local)
        self._found.copy_(torch.maximum(found_local, self._found))
        self._max_over_ranks(self._maxima_local, self._maxima_vec, parts=2,
                             flag=self._found)
        # 4. the update with the whole tensors' maxima; O3: the masters'
        #    amax over ranks, then the weight copy
        o3 = self.level == "O3"
        self._step.finish(hp, clip, self._found, self._found_out,
                          maxima=self._maxima_local,
                          master_amax=self._master_local if o3 else None)
        if o3:
            self._max_over_ranks(self._master_local, self._master_vec)
            self._step.copy(self._master_local)
        # 5. every rank's segment of the new weights to every rank
        if o3:
            comm.all_gather(self._w8_flat, self._w8_flat[rank * seg:(rank + 1) * seg])
            wv = self._w8_vec
            wv.zero_()
            if npc:
                wv[:n].index_copy_(0, self._piece_t, self._w8s_own[:npc].view(torch.int32))
                wv[n:2 * n].index_copy_(0, self._piece_t,
                                        self._w8a_own[:npc].view(torch.int32))
            comm.all_reduce_max(wv)
            self.w8_scale[:n].copy_(wv[:n].view(torch.float32))
            self.w8_amax[:n].copy_(wv[n:2 * n].view(torch.float32))
        else:
            comm.all_gather(self._w_flat, self._w_flat[rank * seg:(rank + 1) * seg])
        found = int(self._found_out.item())
        if clipped:
            self.last_grad_norm = float(self._norm.item())
        return found
