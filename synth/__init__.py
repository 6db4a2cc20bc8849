"""Seeded synthetic inputs for the scaled FP8 cast and the FP8-state AdamW step.

This module is shared by the tests, the bench and the smoke check.  It holds
tensor-list shapes, value distributions and seeds only: none of the method's
arithmetic (no encoding, no scaling rule, no optimizer math).  Every draw is
made with a ``torch.Generator`` seeded per (workload seed, tensor index, role,
step), so any single tensor can be regenerated on its own.  The same call on
the CPU and on a GPU gives different (but each reproducible) streams, so a
test that compares two sides draws once and copies the values across.

Workloads (transformer-shaped lists, GPT-2/GPT-3 naming):

* ``tiny``        3 tensors [64,64], [64], [256,64]; FP32 grads N(0, 1e-3);
                  FP16 weights N(0, 0.02); lr 1e-3, betas (0.9, 0.999),
                  eps 1e-8, wd 0.01; 10 steps, seed 0.
* ``gpt2_cast``   12 layers, d 768, ffn 3072, vocab 50257, ctx 1024 (148
                  tensors, 124,439,808 elements); BF16 grads, per-tensor
                  N(0, sigma), sigma log-uniform in [1e-6, 1e-1].
* ``o2_350m``     24 layers, d 1024, ffn 4096, vocab 50304, ctx 2048 (292
                  tensors); grads N(0, sigma) sigma log-uniform [1e-5, 1e-2],
                  multiplied by the loss scale 65536 before the cast; one
                  gradient element is +inf.
* ``o3_1p3b``     24 layers, d 2048, ffn 8192, vocab 50304 (292 tensors);
                  grads N(0, sigma), sigma log-uniform [1e-5, 1e-2]; FP16
                  master weights N(0, 0.02); O3 (emits an E4M3 weight copy).
* ``fp8_reduce``  the ``gpt2_cast`` list with ``ranks`` = 8 data-parallel
                  gradient copies per tensor (``rank_grad``), each a BF16
                  N(0, sigma_t * f_r) draw, f_r log-uniform in [1/2, 2]: the
                  shards an FP8 all-reduce sums once each is cast to FP8.
* ``o2_6p7b_tail`` 32 layers, d 4096, ffn 16384, vocab 50304 (388 tensors),
                  plus 200 tiny tensors with sizes log-uniform in [1, 4096]
                  and one all-zero-gradient tensor of 4096 elements (589
                  tensors); grads sigma_t * Student-t(nu=3), sigma_t
                  log-uniform [1e-5, 1e-2]; 10 steps.

Every builder takes the model dimensions as arguments, so tests can build the
same structure at sizes a scalar CPU implementation finishes in seconds.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

__all__ = [
    "Workload", "gpt_shapes", "tiny", "gpt2_cast", "fp8_reduce", "o2_350m",
    "o3_1p3b",
    "o2_6p7b_tail", "WORKLOADS", "tensor_seed",
]


def _mix64(x: int) -> int:
    """A 64-bit integer mixer (splitmix64 finaliser) used only to derive seeds."""
    x &= 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return x ^ (x >> 31)


_ROLES = {"grad": 1, "weight": 2, "sigma": 3, "tail": 4, "m": 5, "v": 6,
          "rank": 7}


def tensor_seed(seed: int, index: int, role: str, step: int = 0) -> int:
    """Seed of the stream that draws ``role`` values of tensor ``index``."""
    h = _mix64(seed * 0x9E3779B97F4A7C15 + 0x1234567)
    h = _mix64(h ^ (index + 1) * 0xD1B54A32D192ED03)
    h = _mix64(h ^ _ROLES[role] * 0xA24BAED4963EE407)
    h = _mix64(h ^ (step + 1) * 0x9FB21C651E98DF25)
    return h & 0x7FFFFFFFFFFFFFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def gpt_shapes(n_layer: int, d: int, ffn: int, vocab: int,
               ctx: int) -> List[Tuple[str, Tuple[int, ...]]]:
    """Parameter list of a GPT-2/GPT-3-style decoder, embedding first."""
    out = [("wte", (vocab, d)), ("wpe", (ctx, d))]
    for i in range(n_layer):
        p = f"h{i}."
        out += [
            (p + "ln1.w", (d,)), (p + "ln1.b", (d,)),
            (p + "qkv.w", (3 * d, d)), (p + "qkv.b", (3 * d,)),
            (p + "proj.w", (d, d)), (p + "proj.b", (d,)),
            (p + "ln2.w", (d,)), (p + "ln2.b", (d,)),
            (p + "fc.w", (ffn, d)), (p + "fc.b", (ffn,)),
            (p + "fc2.w", (d, ffn)), (p + "fc2.b", (d,)),
        ]
    out += [("lnf.w", (d,)), ("lnf.b", (d,))]
    return out


@dataclass
class Workload:
    """A named tensor list with its value recipe and optimizer settings."""
    name: str
    names: List[str]
    shapes: List[Tuple[int, ...]]
    seed: int
    grad_dtype: torch.dtype = torch.bfloat16
    grad_dist: str = "normal"             # "normal" or "student_t3"
    sigma_fixed: Optional[float] = None   # one std for every tensor
    sigma_range: Tuple[float, float] = (1e-5, 1e-2)  # log-uniform per tensor
    grad_mult: float = 1.0                # e.g. the loss scale
    zero_grad_tensors: Tuple[int, ...] = ()
    inf_site: Optional[Tuple[int, int]] = None  # (tensor, element) set to +inf
    weight_std: float = 0.02
    level: str = "O2"                     # "O2" or "O3"
    grad_fmt: str = "e4m3"
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    wd: float = 0.01
    inv_loss_scale: float = 1.0
    steps: int = 1
    warmup_steps: int = 0
    ranks: int = 1                        # data-parallel gradient copies

    @property
    def numels(self) -> List[int]:
        return [math.prod(s) for s in self.shapes]

    @property
    def n_params(self) -> int:
        return sum(self.numels)

    def sigma(self, i: int) -> float:
        if self.sigma_fixed is not None:
            return self.sigma_fixed
        lo, hi = self.sigma_range
        r = random.Random(tensor_seed(self.seed, i, "sigma"))
        return math.exp(r.uniform(math.log(lo), math.log(hi)))

    def grad(self, i: int, step: int, device="cpu") -> torch.Tensor:
        """Pre-cast gradient of tensor ``i`` at ``step`` (1-based), flat."""
        n = self.numels[i]
        if i in self.zero_grad_tensors:
            return torch.zeros(n, dtype=self.grad_dtype, device=device)
        g = _gen(device, tensor_seed(self.seed, i, "grad", step))
        if self.grad_dist == "normal":
            x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        elif self.grad_dist == "student_t3":
            # t = Z / sqrt(chi2_3 / 3), chi2_3 a sum of three squared normals
            z = torch.randn(4, n, generator=g, device=device, dtype=torch.float32)
            chi2 = z[1].square() + z[2].square() + z[3].square()
            x = z[0] / torch.sqrt(chi2 / 3.0)
            del z, chi2
        else:
            raise ValueError(self.grad_dist)
        x.mul_(self.sigma(i) * self.grad_mult)
        if self.inf_site is not None and self.inf_site[0] == i:
            x[self.inf_site[1]] = float("inf")
        return x.to(self.grad_dtype)

    def grads(self, step: int, device="cpu") -> List[torch.Tensor]:
        return [self.grad(i, step, device) for i in range(len(self.shapes))]

    def rank_grad(self, i: int, step: int, rank: int, device="cpu") -> torch.Tensor:
        """Pre-cast gradient of tensor ``i`` on data-parallel rank ``rank``:
        an independent draw per rank from the tensor's distribution, with the
        rank's std the tensor's times a factor log-uniform in [1/2, 2]."""
        n = self.numels[i]
        if i in self.zero_grad_tensors:
            return torch.zeros(n, dtype=self.grad_dtype, device=device)
        g = _gen(device, tensor_seed(self.seed, i, "rank", step * 4096 + rank))
        f = math.exp(random.Random(tensor_seed(self.seed, i, "rank", rank))
                     .uniform(-math.log(2.0), math.log(2.0)))
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        return x.mul_(self.sigma(i) * f * self.grad_mult).to(self.grad_dtype)

    def weight(self, i: int, device="cpu") -> torch.Tensor:
        """Initial FP16 weight (O2) or FP16 master weight (O3), flat."""
        g = _gen(device, tensor_seed(self.seed, i, "weight"))
        x = torch.randn(self.numels[i], generator=g, device=device,
                        dtype=torch.float32)
        return x.mul_(self.weight_std).to(torch.float16)

    def weights(self, device="cpu") -> List[torch.Tensor]:
        return [self.weight(i, device) for i in range(len(self.shapes))]

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2,
                    eps=self.eps, wd=self.wd,
                    inv_loss_scale=self.inv_loss_scale)


def _tail_sizes(seed: int, count: int, hi: int = 4096) -> List[int]:
    r = random.Random(tensor_seed(seed, 0, "tail"))
    return [max(1, min(hi, int(round(math.exp(r.uniform(0.0, math.log(hi)))))))
            for _ in range(count)]


def tiny() -> Workload:
    shapes = [(64, 64), (64,), (256, 64)]
    return Workload("tiny", ["w0", "b0", "w1"], shapes, seed=0,
                    grad_dtype=torch.float32, sigma_fixed=1e-3, steps=10)


def gpt2_cast(n_layer=12, d=768, ffn=3072, vocab=50257, ctx=1024,
              seed=2) -> Workload:
    nm, sh = zip(*gpt_shapes(n_layer, d, ffn, vocab, ctx))
    return Workload("gpt2_cast", list(nm), list(sh), seed=seed,
                    grad_dtype=torch.bfloat16, sigma_range=(1e-6, 1e-1))


def fp8_reduce(ranks=8, n_layer=12, d=768, ffn=3072, vocab=50257, ctx=1024,
               seed=6) -> Workload:
    nm, sh = zip(*gpt_shapes(n_layer, d, ffn, vocab, ctx))
    return Workload("fp8_reduce", list(nm), list(sh), seed=seed,
                    grad_dtype=torch.bfloat16, sigma_range=(1e-6, 1e-1),
                    ranks=ranks)


def o2_350m(n_layer=24, d=1024, ffn=4096, vocab=50304, ctx=2048,
            seed=3) -> Workload:
    nm, sh = zip(*gpt_shapes(n_layer, d, ffn, vocab, ctx))
    numel5 = math.prod(sh[5])
    return Workload("o2_350m", list(nm), list(sh), seed=seed,
                    grad_dtype=torch.bfloat16, sigma_range=(1e-5, 1e-2),
                    grad_mult=65536.0, inv_loss_scale=1.0 / 65536.0,
                    inf_site=(5, numel5 // 3), warmup_steps=5)


def o3_1p3b(n_layer=24, d=2048, ffn=8192, vocab=50304, ctx=2048,
            seed=4) -> Workload:
    nm, sh = zip(*gpt_shapes(n_layer, d, ffn, vocab, ctx))
    return Workload("o3_1p3b", list(nm), list(sh), seed=seed,
                    grad_dtype=torch.bfloat16, sigma_range=(1e-5, 1e-2),
                    level="O3", warmup_steps=2)


def o2_6p7b_tail(n_layer=32, d=4096, ffn=16384, vocab=50304, ctx=2048,
                 n_tail=200, tail_max=4096, zero_numel=4096,
                 seed=5) -> Workload:
    nm, sh = zip(*gpt_shapes(n_layer, d, ffn, vocab, ctx))
    names, shapes = list(nm), list(sh)
    for j, s in enumerate(_tail_sizes(seed, n_tail, tail_max)):
        names.append(f"tail{j}")
        shapes.append((s,))
    names.append("zero")
    shapes.append((zero_numel,))
    return Workload("o2_6p7b_tail", names, shapes, seed=seed,
                    grad_dtype=torch.bfloat16, grad_dist="student_t3",
                    sigma_range=(1e-5, 1e-2),
                    zero_grad_tensors=(len(shapes) - 1,), steps=10)


WORKLOADS = {
    "tiny": tiny, "gpt2_cast": gpt2_cast, "fp8_reduce": fp8_reduce,
    "o2_350m": o2_350m,
    "o3_1p3b": o3_1p3b, "o2_6p7b_tail": o2_6p7b_tail,
}
