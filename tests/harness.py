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


def fresh_states(weights: Sequence[torch.Tensor], o3: bool, g_fmt=oracle.E4M3):
    out = []
    for w in weights:
        n = w.numel()
        out.append(oracle.StepState(
            np.zeros(n, np.uint8), 1.0, np.zeros(n, np.uint8), 1.0,
            np.zeros(n, np.uint16), to_np_u16(w.cpu()), g_fmt=g_fmt, o3=o3))
    return out


def set_grads(states, codes, scales):
    for s, c, sc in zip(states, codes, scales):
        s.g = np.ascontiguousarray(c, np.uint8)
        s.g_scale = float(np.float32(sc))


def oracle_step(states, wl, step, ils=None):
    return oracle.adamw_step(states, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd,
                             step, wl.inv_loss_scale if ils is None else ils)


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
        fmts = [s.g_fmt for s in states]
        self.plan = bo.AdamWPlan(self.g, self.g_scale, self.m, self.m_scale,
                                 self.v, self.w, self.w8, self.w8_scale,
                                 self.w8_amax, g_fmt=fmts)
        self.found_dev = torch.full((1,), 7, dtype=torch.int32, device=device)

    def step(self, wl, step, ils=None):
        found = self.plan(wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, step,
                          wl.inv_loss_scale if ils is None else ils,
                          found_inf_dev=self.found_dev)
        assert int(self.found_dev.item()) == found
        return found

    def compare(self, ref_states, master_rel=False):
        """Compare every output against oracle states; returns exact rates."""
        m_scale = self.m_scale.cpu().numpy()[:len(ref_states)]
        check_f32_exact(m_scale, [s.m_scale[0] for s in ref_states], "m_scale")
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
