"""Drives the oracle and the CUDA library on the same synthetic inputs.

Inputs come from ``synth`` (seeded, drawn on the CPU or on the GPU with
torch's generators); oracle inputs and expected values never come from the
CUDA library: where the library's step consumes gradient codes, the codes the
oracle produced are uploaded for it.
"""
from typing import List, Sequence

import numpy as np
import torch

import oracle
from parity import (bf16_bits, check_codes, check_f16, check_f32_exact,
                    check_master, from_np_u16, to_np_u16, to_np_u8)

DT = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16,
      torch.float16: oracle.F16}


def host_src(t: torch.Tensor):
    """A CPU tensor as the oracle's input array and dtype code."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy(), oracle.F32
    return bf16_bits(t), DT[t.dtype]


def oracle_cast(grads: Sequence[torch.Tensor], fmt: int):
    codes, amax, scale = [], [], []
    for g in grads:
        a, dt = host_src(g)
        c, am, sc = oracle.cast_scaled(a, dt, fmt)
        codes.append(c)
        amax.append(am)
        scale.append(sc)
    return codes, np.array(amax, np.float32), np.array(scale, np.float32)


def fresh_states(weights: Sequence[torch.Tensor], o3: bool, g_fmt=oracle.E4M3,
                 scaled_v=False):
    out = []
    for w in weights:
        n = w.numel()
        out.append(oracle.StepState(
            np.zeros(n, np.uint8), 1.0, np.zeros(n, np.uint8), 1.0,
            np.zeros(n, np.uint16), to_np_u16(w.cpu()), g_fmt=g_fmt, o3=o3,
            scaled_v=scaled_v))
    return out


def set_grads(states, codes, scales):
    for s, c, sc in zip(states, codes, scales):
        s.g = np.ascontiguousarray(c, np.uint8)
        s.g_scale = float(np.float32(sc))


def oracle_step(states, wl, step, ils=None, l2=False):
    return oracle.adamw_step(states, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd,
                             step, wl.inv_loss_scale if ils is None else ils,
                             l2=l2)


def oracle_step_threads(states, wl, step, pool, workers):
    """oracle_step over a long list on the host's cores: the tensors are
    dealt, largest first, into `workers` groups of about equal size, and each
    group is one oracle call in a thread of `pool` (ctypes releases the GIL).
    With every gradient finite, each tensor's result is the one of a single
    call over the whole list; returns the largest found_inf of the groups."""
    groups = [[] for _ in range(workers)]
    load = [0] * workers
    for i in sorted(range(len(states)), key=lambda i: -states[i].numel):
        j = load.index(min(load))
        groups[j].append(states[i])
        load[j] += states[i].numel
    found = list(pool.map(lambda g: oracle_step(g, wl, step) if g else 0, groups))
    return max(found)


class GpuState:
    """The library's view of a list of oracle states, on the device."""

    def __init__(self, states, device="cuda", misalign=()):
        import bit_optimizer_gb300 as bo
        self.states = states
        n = len(states)
        self.o3 = states[0].w8 is not None if n else False
        f32 = dict(dtype=torch.float32, device=device)
        self.g_scale = torch.tensor([s.g_scale for s in states] or [1.0], **f32)
        self.m_scale = torch.tensor([s.m_scale[0] for s in states] or [1.0], **f32)

        def put(a, i, kind):
            # `misalign` lists tensor indices whose buffers start off the
            # vector alignment (one element past an aligned start)
            off = 1 if i in misalign else 0
            if kind == "u8":
                buf = torch.zeros(a.size + off, dtype=torch.uint8, device=device)
                buf[off:] = torch.from_numpy(a).to(device)
            else:
                buf = torch.zeros(a.size + off, dtype=torch.float16, device=device)
                buf[off:] = from_np_u16(a, device)
            return buf[off:]

        self.g = [put(s.g, i, "u8") for i, s in enumerate(states)]
        self.m = [put(s.m, i, "u8") for i, s in enumerate(states)]
        self.v = [put(s.v, i, "f16") for i, s in enumerate(states)]
        self.w = [put(s.w, i, "f16") for i, s in enumerate(states)]
        if self.o3:
            self.w8 = [put(s.w8, i, "u8") for i, s in enumerate(states)]
            self.w8_scale = torch.tensor([s.w8_scale[0] for s in states], **f32)
            self.w8_amax = torch.tensor([s.w8_amax[0] for s in states], **f32)
        else:
            self.w8 = self.w8_scale = self.w8_amax = None
        self.scaled_v = n > 0 and states[0].v_bound is not None
        self.v_bound = (torch.tensor([s.v_bound[0] for s in states], **f32)
                        if self.scaled_v else None)
        fmts = [s.g_fmt for s in states]
        self.plan = bo.AdamWPlan(self.g, self.g_scale, self.m, self.m_scale,
                                 self.v, self.w, self.w8, self.w8_scale,
                                 self.w8_amax, g_fmt=fmts, v_bound=self.v_bound)
        self.found_dev = torch.full((1,), 7, dtype=torch.int32, device=device)

    def step(self, wl, step, ils=None, l2=False):
        found = self.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, step,
                          wl.inv_loss_scale if ils is None else ils,
                          found_inf_dev=self.found_dev, l2=l2)
        assert int(self.found_dev.item()) == found
        return found

    def compare(self, ref_states, master_rel=False):
        """Compare every output against oracle states; returns exact rates."""
        m_scale = self.m_scale.cpu().numpy()[:len(ref_states)]
        check_f32_exact(m_scale, [s.m_scale[0] for s in ref_states], "m_scale")
        if self.scaled_v:
            check_f32_exact(self.v_bound.cpu().numpy()[:len(ref_states)],
                            [s.v_bound[0] for s in ref_states], "v_bound")
        rates = {"m": [], "v": [], "w": [], "w8": []}
        for i, s in enumerate(ref_states):
            rates["m"].append(check_codes(to_np_u8(self.m[i]), s.m, name=f"m[{i}]"))
            rates["v"].append(check_f16(to_np_u16(self.v[i]), s.v, name=f"v[{i}]"))
            w = to_np_u16(self.w[i])
            if self.o3:
                check_master(w, s.w, name=f"master[{i}]")
            rates["w"].append(check_f16(w, s.w, name=f"w[{i}]"))
            if self.o3:
                rates["w8"].append(check_codes(to_np_u8(self.w8[i]), s.w8,
                                               name=f"w8[{i}]"))
        if self.o3:
            check_f32_exact(self.w8_scale.cpu().numpy(),
                            [s.w8_scale[0] for s in ref_states], "w8_scale")
            check_f32_exact(self.w8_amax.cpu().numpy(),
                            [s.w8_amax[0] for s in ref_states], "w8_amax")
        return {k: (min(v) if v else 1.0) for k, v in rates.items()}

    def load_state(self, states):
        """Overwrite the device state with oracle states (same tensors)."""
        for i, s in enumerate(states):
            self.g[i].copy_(torch.from_numpy(s.g))
            self.m[i].copy_(torch.from_numpy(s.m))
            self.v[i].copy_(from_np_u16(s.v, self.v[i].device))
            self.w[i].copy_(from_np_u16(s.w, self.w[i].device))
        self.g_scale[:len(states)].copy_(torch.tensor([s.g_scale for s in states]))
        self.m_scale[:len(states)].copy_(torch.tensor([s.m_scale[0] for s in states]))
        if self.scaled_v:
            self.v_bound[:len(states)].copy_(
                torch.tensor([s.v_bound[0] for s in states]))


class DeviceList:
    """A whole workload resident on the device, in 256-byte-aligned arenas, run
    through the same plans ``bench.py`` times (CastPlan + AdamWPlan).  The
    oracle follows a sample of whole tensors: before each step their device
    state is overwritten with the oracle's, so every compared output is one
    step of the library from the oracle's inputs."""

    def __init__(self, wl, device="cuda", scaled_v=False):
        import bit_optimizer_gb300 as bo
        self.wl = wl
        self.device = device
        self.scaled_v = scaled_v
        self.o3 = wl.level == "O3"
        self.fmt = oracle.FMT[wl.grad_fmt]
        n = len(wl.shapes)
        numels = wl.numels
        f32 = dict(dtype=torch.float32, device=device)
        self.w = bo.arena_views(numels, torch.float16, device)
        for i, w in enumerate(self.w):
            w.copy_(wl.weight(i, device))
        self.src = bo.arena_views(numels, wl.grad_dtype, device)
        self.g = bo.arena_views(numels, torch.uint8, device)
        self.m = bo.arena_views(numels, torch.uint8, device, fill=0)
        self.v = bo.arena_views(numels, torch.float16, device, fill=0)
        self.g_amax = torch.zeros(n, **f32)
        self.g_scale = torch.ones(n, **f32)
        self.m_scale = torch.ones(n, **f32)
        if self.o3:
            self.w8 = bo.arena_views(numels, torch.uint8, device, fill=0)
            self.w8_scale = torch.ones(n, **f32)
            self.w8_amax = torch.zeros(n, **f32)
        else:
            self.w8 = self.w8_scale = self.w8_amax = None
        self.v_bound = torch.zeros(n, **f32) if scaled_v else None
        self.cast = bo.CastPlan(self.src, self.g, self.g_amax, self.g_scale,
                                wl.grad_fmt)
        self.plan = bo.AdamWPlan(self.g, self.g_scale, self.m, self.m_scale,
                                 self.v, self.w, self.w8, self.w8_scale,
                                 self.w8_amax, wl.grad_fmt, self.v_bound)
        self.found_dev = torch.zeros(1, dtype=torch.int32, device=device)

    def gen_grads(self, step, wl=None):
        wl = wl or self.wl
        for i, s in enumerate(self.src):
            s.copy_(wl.grad(i, step, self.device))

    def fresh_oracle(self, i):
        n = self.wl.numels[i]
        return oracle.StepState(np.zeros(n, np.uint8), 1.0, np.zeros(n, np.uint8),
                                1.0, np.zeros(n, np.uint16), to_np_u16(self.w[i]),
                                g_fmt=self.fmt, o3=self.o3, scaled_v=self.scaled_v)

    def cast_and_check(self, sample, states):
        """GPU cast of every tensor; the oracle casts the sampled ones from
        the same values and its codes become their step inputs."""
        self.cast()
        torch.cuda.synchronize()
        amax = self.g_amax.cpu().numpy()
        scale = self.g_scale.cpu().numpy()
        for i in sample:
            a, dt = host_src(self.src[i])
            codes, am, sc = oracle.cast_scaled(a, dt, self.fmt)
            check_f32_exact(amax[i:i + 1], [am], f"grad amax[{i}]")
            check_f32_exact(scale[i:i + 1], [sc], f"grad scale[{i}]")
            check_codes(to_np_u8(self.g[i]), codes, self.fmt, name=f"grad[{i}]")
            states[i].g = codes
            states[i].g_scale = float(sc)

    def put(self, i, st):
        self.g[i].copy_(torch.from_numpy(st.g))
        self.g_scale[i] = st.g_scale
        self.m[i].copy_(torch.from_numpy(st.m))
        self.m_scale[i] = float(st.m_scale[0])
        self.v[i].copy_(from_np_u16(st.v, self.device))
        self.w[i].copy_(from_np_u16(st.w, self.device))
        if self.scaled_v:
            self.v_bound[i] = float(st.v_bound[0])

    def step(self, t, ils=None):
        wl = self.wl
        return self.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
                         wl.inv_loss_scale if ils is None else ils,
                         found_inf_dev=self.found_dev)

    def cast_step(self, t, ils=None):
        """The cast of every tensor and the step in one fp8_cast_adamw_step
        call (the bench's configuration)."""
        import bit_optimizer_gb300 as bo
        wl = self.wl
        if not hasattr(self, "fused"):
            self.fused = bo.CastStepPlan(self.cast, self.plan)
        return self.fused(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, t,
                          wl.inv_loss_scale if ils is None else ils,
                          found_inf_dev=self.found_dev)

    def check_cast(self, sample, states):
        """After a fused call: the sampled tensors' codes, amax and scale
        against the oracle's cast of the same values, which become the
        oracle's step inputs."""
        amax = self.g_amax.cpu().numpy()
        scale = self.g_scale.cpu().numpy()
        for i in sample:
            a, dt = host_src(self.src[i])
            codes, am, sc = oracle.cast_scaled(a, dt, self.fmt)
            check_f32_exact(amax[i:i + 1], [am], f"grad amax[{i}]")
            check_f32_exact(scale[i:i + 1], [sc], f"grad scale[{i}]")
            check_codes(to_np_u8(self.g[i]), codes, self.fmt, name=f"grad[{i}]")
            states[i].g = codes
            states[i].g_scale = float(sc)

    def compare(self, i, st):
        check_f32_exact(self.m_scale[i:i + 1].cpu().numpy(), st.m_scale, f"m_scale[{i}]")
        if self.scaled_v:
            check_f32_exact(self.v_bound[i:i + 1].cpu().numpy(), st.v_bound,
                            f"v_bound[{i}]")
        check_codes(to_np_u8(self.m[i]), st.m, name=f"m[{i}]")
        check_f16(to_np_u16(self.v[i]), st.v, name=f"v[{i}]")
        w = to_np_u16(self.w[i])
        check_f16(w, st.w, name=f"w[{i}]")
        if self.o3:
            check_master(w, st.w, name=f"master[{i}]")
            check_codes(to_np_u8(self.w8[i]), st.w8, name=f"w8[{i}]")
            check_f32_exact(self.w8_scale[i:i + 1].cpu().numpy(), st.w8_scale,
                            f"w8_scale[{i}]")
            check_f32_exact(self.w8_amax[i:i + 1].cpu().numpy(), st.w8_amax,
                            f"w8_amax[{i}]")

    def invariants(self):
        """Properties of a finished step that hold for every tensor at any
        size: the just-in-time scale puts each nonzero first moment's largest
        element on the E4M3 maximum, no moment is NaN, v is non-negative, and
        the weights are finite."""
        for i in range(len(self.m)):
            if self.m[i].numel() == 0:
                continue
            mag = self.m[i] & 0x7F
            top = int(mag.max().item())
            assert top in (0, 0x7E), f"tensor {i}: largest |m| code {top:#x}"
            assert not bool((mag == 0x7F).any().item()), f"tensor {i}: NaN m"
            v = self.v[i]
            assert not bool((v < 0).any().item()), f"tensor {i}: negative v"
            assert bool(torch.isfinite(self.w[i]).all().item()), f"tensor {i}: w"
            if self.o3:
                top8 = int((self.w8[i] & 0x7F).max().item())
                assert top8 in (0, 0x7E), f"tensor {i}: largest |w8| code {top8:#x}"
