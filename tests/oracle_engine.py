"""The sharded step's arithmetic by the oracle, on host tensors: an engine
with the methods of ``bit_optimizer_gb300.sharded.LibEngine``, so the sharded
step loop's host logic (partition, exchanges, skip, broadcasts) can run on CPU
ranks over gloo.  Test infrastructure only."""
import math

import numpy as np
import torch

import oracle
from harness import host_src


def _u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _put_u16(t, a):
    t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.dtype))


class OracleEngine:
    def make_cast(self, srcs, codes, amax, scale, fmt):
        f = oracle.FMT[fmt]

        def run():
            for i, (s, c) in enumerate(zip(srcs, codes)):
                a, dt = host_src(s)
                cc, am, sc = oracle.cast_scaled(a, dt, f)
                c.copy_(torch.from_numpy(cc))
                amax[i] = float(am)
                scale[i] = float(sc)
        return run

    def make_reduce(self, shards, scales, codes, amax, scale, in_fmt, out_fmt,
                    post):
        fi, fo = oracle.FMT[in_fmt], oracle.FMT[out_fmt]

        def run(stream=None, norm_terms=None, found=None, inv_loss_scale=1.0):
            for i, sh in enumerate(shards):
                cc, am, sc = oracle.reduce_scaled(sh.contiguous().numpy(),
                                                  scales[i].numpy(), fi, fo, post)
                codes[i].copy_(torch.from_numpy(cc))
                amax[i] = float(am)
                scale[i] = float(sc)
            if norm_terms is not None:
                states = [oracle.StepState(c.numpy(), float(scale[i]),
                                           np.zeros(c.numel(), np.uint8), 1.0,
                                           np.zeros(c.numel(), np.uint16),
                                           np.zeros(c.numel(), np.uint16), g_fmt=fo)
                          for i, c in enumerate(codes)]
                f, tt = oracle.grad_norm_terms(states, inv_loss_scale)
                norm_terms[:len(codes)] = torch.from_numpy(tt.copy())
                if found is not None:
                    found[0] = f
        return run

    def make_step(self, g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                  g_fmt, v_bound):
        return OracleStep(g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                          oracle.FMT[g_fmt], v_bound)

    def clip_coef(self, terms, max_grad_norm, clip, norm, found):
        total = 0.0
        for t in terms.tolist():
            total += t
        inf = found is not None and int(found[0]) != 0
        nv = math.inf if inf else math.sqrt(total)
        if norm is not None:
            norm[0] = nv
        clip[0] = 1.0 if inf else oracle.clip_coef(nv, max_grad_norm)


class OracleStep:
    def __init__(self, g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                 g_fmt, v_bound):
        self.t = dict(g=g, g_scale=g_scale, m=m, m_scale=m_scale, v=v, w=w,
                      w8=w8, w8_scale=w8_scale, w8_amax=w8_amax, v_bound=v_bound)
        self.fmt = g_fmt
        self.n = len(g)
        self._begun = 0

    def _states(self):
        t = self.t
        out = []
        for i in range(self.n):
            st = oracle.StepState(t["g"][i].numpy(), float(t["g_scale"][i]),
                                  t["m"][i].numpy(), float(t["m_scale"][i]),
                                  _u16(t["v"][i]), _u16(t["w"][i]), g_fmt=self.fmt,
                                  o3=t["w8"] is not None,
                                  scaled_v=t["v_bound"] is not None,
                                  v_bound=(float(t["v_bound"][i])
                                           if t["v_bound"] is not None else 0.0))
            out.append(st)
        return out

    def _write(self, states):
        t = self.t
        for i, st in enumerate(states):
            t["m"][i].copy_(torch.from_numpy(st.m))
            t["m_scale"][i] = float(st.m_scale[0])
            _put_u16(t["v"][i], st.v)
            _put_u16(t["w"][i], st.w)
            if t["w8"] is not None:
                t["w8"][i].copy_(torch.from_numpy(st.w8))
                t["w8_scale"][i] = float(st.w8_scale[0])
                t["w8_amax"][i] = float(st.w8_amax[0])
            if t["v_bound"] is not None:
                t["v_bound"][i] = float(st.v_bound[0])

    def norm_terms(self, inv_loss_scale, terms, found=None, stream=None):
        f, tt = oracle.grad_norm_terms(self._states(), inv_loss_scale)
        terms[:self.n] = torch.from_numpy(tt.copy())
        if found is not None:
            found[0] = f

    def begin(self, hp, clip=None, found=None, stream=None):
        self._begun = oracle.grad_norm(self._states(), hp[6])[0]
        if found is not None:
            found[0] = self._begun

    def finish(self, hp, clip=None, found_in=None, found=None, stream=None):
        lr, b1, b2, eps, wd, step, ils, l2 = hp
        f = self._begun or (found_in is not None and int(found_in[0]) != 0)
        if not f:
            states = self._states()
            c = float(clip[0]) if clip is not None else 1.0
            assert oracle.adam_step_coef(states, lr, b1, b2, eps, wd, step, ils,
                                         c, l2=l2) == 0
            self._write(states)
        if found is not None:
            found[0] = int(f)
