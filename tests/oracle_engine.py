"""The sharded step's arithmetic by the oracle, on host tensors: an engine
with the methods of ``bit_optimizer_gb300.sharded.LibEngine``, so the sharded
step loop's host logic (layout, exchanges, skip, all-gathers) can run on CPU
ranks over gloo.  Each phase is the oracle's phase of the same name: the
reduction's amax and its encode with a given amax, the step's maxima, its
update from given maxima and the weight copy from a given master amax.
Test infrastructure only."""
import math

import numpy as np
import torch

import oracle
from harness import host_src


def _u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _put_u16(t, a):
    t.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(t.dtype))


def _bits(values):
    """float32 values as the int32 bit patterns the exchanges carry."""
    return torch.from_numpy(np.ascontiguousarray(values, np.float32).view(np.int32))


def _floats(bits):
    return bits.numpy().astype(np.int32).view(np.float32)


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
        return OracleReduce(shards, scales, codes, amax, scale,
                            oracle.FMT[in_fmt], oracle.FMT[out_fmt], post)

    def make_step(self, g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                  g_fmt, v_bound):
        return OracleStep(g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                          oracle.FMT[g_fmt], v_bound)

    def make_cast_step(self, cast, step):
        return OracleCastStep(cast, step)

    def norm_terms_from_limbs(self, limbs, amax_bits, fmt, inv_loss_scale, terms):
        f = oracle.FMT[fmt]
        lb = [int(x) for x in limbs.tolist()]
        am = _floats(amax_bits)
        for t in range(terms.numel()):
            s = sum(lb[4 * t + j] << (32 * j) for j in range(4))
            sc = np.float32(oracle.scale_from_amax(float(am[t]), f))
            k = float(np.float32(np.float32(inv_loss_scale) / sc))
            terms[t] = (k * k) * (float(s) * 2.0 ** -32)

    def clip_coef(self, terms, max_grad_norm, clip, norm, found):
        total = 0.0
        for t in terms.tolist():
            total += t
        inf = found is not None and int(found[0]) != 0
        nv = math.inf if inf else math.sqrt(total)
        if norm is not None:
            norm[0] = nv
        clip[0] = 1.0 if inf else oracle.clip_coef(nv, max_grad_norm)


class OracleReduce:
    def __init__(self, shards, scales, codes, amax, scale, fi, fo, post):
        self.shards, self.scales = shards, scales
        self.codes, self.amax, self.scale = codes, amax, scale
        self.fi, self.fo, self.post = fi, fo, post

    def begin(self, amax_bits, stream=None):
        for i, sh in enumerate(self.shards):
            _, am, _ = oracle.reduce_scaled(sh.contiguous().numpy(),
                                            self.scales[i].numpy(), self.fi,
                                            self.fo, self.post)
            amax_bits[i] = int(_bits([am])[0])

    def finish(self, amax_bits, inv_loss_scale=1.0, limbs=None, found=None,
               stream=None):
        am = _floats(amax_bits)
        any_bad = 0
        for i, sh in enumerate(self.shards):
            cc, sc = oracle.reduce_scaled_given(sh.contiguous().numpy(),
                                                self.scales[i].numpy(), self.fi,
                                                self.fo, self.post, float(am[i]))
            self.codes[i].copy_(torch.from_numpy(cc))
            self.amax[i] = float(am[i])
            self.scale[i] = float(sc)
            if limbs is not None:
                s = oracle.fp8_sq_sum(cc, self.fo)
                for j in range(4):
                    limbs[4 * i + j] = (s >> (32 * j)) & 0xFFFFFFFF
                st = oracle.StepState(cc, float(sc), np.zeros(cc.size, np.uint8), 1.0,
                                      np.zeros(cc.size, np.uint16),
                                      np.zeros(cc.size, np.uint16), g_fmt=self.fo)
                any_bad |= oracle.grad_norm_terms([st], inv_loss_scale)[0]
        if found is not None:
            found[0] = any_bad


class OracleStep:
    def __init__(self, g, g_scale, m, m_scale, v, w, w8, w8_scale, w8_amax,
                 g_fmt, v_bound):
        self.t = dict(g=g, g_scale=g_scale, m=m, m_scale=m_scale, v=v, w=w,
                      w8=w8, w8_scale=w8_scale, w8_amax=w8_amax, v_bound=v_bound)
        self.fmt = g_fmt
        self.n = len(g)
        self._begun = 0
        self._skipped = 0

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
            if st.w8 is not None:
                st.w8 = t["w8"][i].numpy().copy()
                st.w8_scale[0] = float(t["w8_scale"][i])
                st.w8_amax[0] = float(t["w8_amax"][i])
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

    def begin(self, hp, clip=None, found=None, stream=None, maxima=None):
        lr, b1, b2, eps, wd, step, ils, l2 = hp
        c = float(clip[0]) if clip is not None else 1.0
        f, am, gm = oracle.step_maxima(self._states(), lr, b1, b2, wd, step, ils,
                                       clip=c, l2=l2)
        self._begun = f
        if found is not None:
            found[0] = f
        if maxima is not None:
            maxima[:2 * self.n] = 0
            if f == 0 and self.n:
                maxima[:self.n] = _bits(am)
                maxima[self.n:2 * self.n] = _bits(gm)

    def finish(self, hp, clip=None, found_in=None, found=None, stream=None,
               maxima=None, master_amax=None):
        lr, b1, b2, eps, wd, step, ils, l2 = hp
        f = self._begun or (found_in is not None and int(found_in[0]) != 0)
        self._skipped = int(f)
        if not f:
            states = self._states()
            c = float(clip[0]) if clip is not None else 1.0
            if maxima is not None:
                am, gm = _floats(maxima[:self.n]), _floats(maxima[self.n:2 * self.n])
            else:
                _, am, gm = oracle.step_maxima(states, lr, b1, b2, wd, step, ils,
                                               clip=c, l2=l2)
            wm = oracle.step_update(states, lr, b1, b2, eps, wd, step, ils, am, gm,
                                    clip=c, l2=l2)
            if master_amax is not None:
                master_amax[:self.n] = _bits(wm)
            else:
                oracle.weight_copy(states, wm)
            self._write(states)
        if found is not None:
            found[0] = int(f)

    def copy(self, master_amax, stream=None):
        if self._skipped:
            return
        states = self._states()
        oracle.weight_copy(states, _floats(master_amax[:self.n]))
        self._write(states)


class OracleCastStep:
    """The cast and the step in one call (the one-rank path)."""

    def __init__(self, cast, step):
        self.cast, self.step = cast, step
        self.last_grad_norm = None

    def __call__(self, lr, b1, b2, eps, wd, step, ils, found_inf_dev=None,
                 sync=True, stream=None, l2=False, max_grad_norm=None,
                 grad_norm_dev=None):
        self.cast()
        states = self.step._states()
        if max_grad_norm is not None:
            f, nv = oracle.adam_step_clipped(states, lr, b1, b2, eps, wd, step, ils,
                                             max_grad_norm, l2=l2)
            self.last_grad_norm = nv
        else:
            f = oracle.adamw_step(states, lr, b1, b2, eps, wd, step, ils, l2=l2)
        if f == 0:
            self.step._write(states)
        if found_inf_dev is not None:
            found_inf_dev[0] = f
        return f
