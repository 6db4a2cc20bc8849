// FP8-state AdamW step over a tensor list (MS-AMP O2, and O3 with an FP16
// master and an FP8 weight copy), with the GradScaler inf/NaN skip.
//
// Three persistent kernels over the chunk table:
//   step_amax_kernel    reads g and m codes; recomputes this step's fp32 first
//                       moment and reduces its per-tensor amax (the scale of
//                       the new E4M3 moment is just in time, so it must be
//                       known before any moment is written); sets found_inf
//                       when an unscaled gradient is not finite.  2 B/param.
//   step_update_kernel  exits at once when found_inf is set; otherwise the
//                       fused dequantize + unscale + Adam moments + bias
//                       correction + decoupled weight decay update, writing
//                       E4M3 m, FP16 v and the FP16 weight (O2) / master (O3),
//                       and for O3 the per-tensor amax of the FP16 master.
//                       Reads 6 B, writes 5 B per param.
//   step_w8_kernel      O3 only: w8 = E4M3 encode of master * 448 / amax.
//                       Reads 2 B, writes 1 B per param.
// The update walks the chunk table backwards and the O3 pass forwards, so
// each pass starts on the chunks the previous one left in L2.
//
// Arithmetic per element, in fp32 (each operation rounded once; fma rounds
// the product and the sum once together):
//   g = dec(g_code) * k                       k = inv_loss_scale / g_scale
//                                             (times the clip coefficient
//                                             when the call clips)
//   [Adam with L2 decay: g = fma(wd, w_old, g)]
//   m = fma(beta1, dec(m_code) * minv, (1 - beta1) * g)   minv = 1 / m_scale
//   v = fma(beta2, v_old, (1 - beta2) * (g * g))
//   u = m / fma(sqrt(v), inv_sbc2, eps)
//   w = fma(-step_size, u, w_old * decay)     decay = 1 - lr * wd, or 1 (L2)
// A scaled second moment (v_bound set) keeps a per-tensor bound B on max v:
// B_new = fma(beta2, B_old, (1 - beta2) * gmax * gmax) with gmax = max |g|
// from the first pass; v_old = FP16 * (B_old * 2^-14) and v is stored as FP16
// of v * (2^14 / B_new).
// Elements are processed in pairs with the paired fp32 instructions, which
// round each lane like the scalar ones, so the first moment, its amax and its
// scale are bit-identical to a scalar fp32 evaluation of the same lines.
//
// Device-resident step (DEVS instantiations, the *_dev calls): lr,
// inv_loss_scale and the step count live in device memory.
// step_scalars_kernel turns them into step_size, inv_sbc2, decay and ils with
// the host's arithmetic.  The passes read those four from the device.  The
// update stores the new step count unless found_inf skipped the step.  A
// CUDA graph of such a call then serves every step.
#include "fp8opt_internal.cuh"

namespace fp8opt {

namespace {

// Tunables (compile-time): 8-element groups each thread keeps in flight per
// tile in the amax and update passes, and the update kernel's CTA size and
// resident CTAs per SM (which cap its registers a thread).  The update kernel
// is latency-bound, so what counts is the warps an SM holds: at 72 registers
// an SM holds 28 warps as seven CTAs of 128 threads but 24 as three of 256
// (76 registers).  Measured on the 6.7B list: 11.56 ms against 12.16 ms.
#ifndef FP8OPT_STEP_AMAX_GROUPS
#define FP8OPT_STEP_AMAX_GROUPS 8
#endif
#ifndef FP8OPT_UPD_GROUPS
#define FP8OPT_UPD_GROUPS 2
#endif
#ifndef FP8OPT_UPD_THREADS
#define FP8OPT_UPD_THREADS 128
#endif
#ifndef FP8OPT_UPD_MIN_BLOCKS
#define FP8OPT_UPD_MIN_BLOCKS 7
#endif
// The same for the scaled-second-moment, L2 and device-resident-step
// instantiations.  These need a few more registers: at 7 CTAs/SM they spill
// 8 to 52 bytes, at 6 they do not.  7 is still faster.  Measured on the O3
// 1.3B step with the scaled second moment: 4.04 ms at 7 CTAs/SM, 4.13 at 6.
// Measured on Adam-L2 over 350M: 1.127 ms at 7, 1.142 at 6.
#ifndef FP8OPT_UPD_MIN_BLOCKS_VAR
#define FP8OPT_UPD_MIN_BLOCKS_VAR 7
#endif
// Tiles ahead of the current one that the update and amax passes prefetch
// into L2 (0: none).  Measured on the 6.7B list: the update pass is 7 %
// slower with a prefetch one or two tiles ahead, and the amax pass 4 - 5 %
// slower, so both are off.  The amax pass (clipped 6.7B step, a separate
// run): 2.13 ms with eight groups in flight, 2.21 with four, 2.26 with two.
#ifndef FP8OPT_UPD_PREFETCH
#define FP8OPT_UPD_PREFETCH 0
#endif
#ifndef FP8OPT_STEP_AMAX_PREFETCH
#define FP8OPT_STEP_AMAX_PREFETCH 0
#endif
constexpr int kAmaxGroups = FP8OPT_STEP_AMAX_GROUPS;
constexpr int kUpdGroups = FP8OPT_UPD_GROUPS;
constexpr int kUpdThreads = FP8OPT_UPD_THREADS;
constexpr int kW8Groups = 2;

// Device-resident step (DEVS): the call's DevScalars, copied into shared
// memory by thread 0 at kernel start (load_dev_scalars), so the passes read
// them without holding a pointer.
__shared__ DevScalars dev_sh;

template <bool DEVS>
__device__ __forceinline__ void load_dev_scalars(const StepScalars& s) {
  if constexpr (DEVS) {
    if (threadIdx.x == 0) dev_sh = *s.dev;
    __syncthreads();
  }
}

template <bool DEVS>
__device__ __forceinline__ float ils_of(const StepScalars& s) {
  if constexpr (DEVS) return dev_sh.ils;
  else return s.ils;
}

// The scalar forms of the lines above (tails and unaligned tensors).
__device__ __forceinline__ float m_new1(float mdec, float minv, float g,
                                        const StepScalars& s) {
  return __fmaf_rn(s.beta1, __fmul_rn(mdec, minv), __fmul_rn(s.omb1, g));
}

template <bool DEVS>
__device__ __forceinline__ void adamw1(float g, float m, float vp, float wp,
                                       const StepScalars& s, float& v,
                                       float& w) {
  v = __fmaf_rn(s.beta2, vp, __fmul_rn(s.omb2, __fmul_rn(g, g)));
  if constexpr (DEVS) {
    const float den = __fmaf_rn(__fsqrt_rn(v), dev_sh.inv_sbc2, s.eps);
    const float u = __fdiv_rn(m, den);
    w = __fmaf_rn(-dev_sh.step_size, u, __fmul_rn(wp, dev_sh.decay));
  } else {
    const float den = __fmaf_rn(__fsqrt_rn(v), s.inv_sbc2, s.eps);
    const float u = __fdiv_rn(m, den);
    w = __fmaf_rn(-s.step_size, u, __fmul_rn(wp, s.decay));
  }
}

// ------------------------------------------------------------ pass 1: amax

// found_inf is "some gradient code magnitude >= T" (overflow_threshold of
// the unclipped factor, passed as its addend `tadd`), so it needs only the
// codes, and a clip coefficient in k cannot hide an unscaled overflow.
// L2: the gradient takes the decay term fma(wd, w, g) (so w is read too).
// Besides the amax of the first moment (mx) this also reduces max |g| (gx)
// when GX: the input of a scaled second moment's bound.
template <int GF, bool L2, bool GX>
__device__ void thread_step_amax(const StepDesc& d, int64_t begin, int64_t end,
                                 float k, float minv, uint32_t tadd,
                                 const StepScalars& s, uint32_t& mx,
                                 uint32_t& gx, uint32_t& bad) {
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kAmaxGroups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  const float2 k2 = splat2(k), minv2 = splat2(minv), b1 = splat2(s.beta1),
               omb1 = splat2(s.omb1), wd2 = splat2(s.wd);
  const bool pf = FP8OPT_STEP_AMAX_PREFETCH > 0 && tid == 0 && vec &&
                  aligned16(d.g) && aligned16(d.m);
  for (int64_t base = begin; base < end; base += kTile) {
    if (pf) {
      const int64_t ahead = base + FP8OPT_STEP_AMAX_PREFETCH * kTile;
      if (ahead + kTile <= end) {
        prefetch_l2(d.g + ahead, (uint32_t)kTile);
        prefetch_l2(d.m + ahead, (uint32_t)kTile);
      }
    }
    if (vec && base + kTile <= end) {
      uint2 gc[kAmaxGroups], mc[kAmaxGroups];
      uint4 wh[kAmaxGroups];
#pragma unroll
      for (int q = 0; q < kAmaxGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        gc[q] = ld_keep2(d.g + i0);
        mc[q] = ld_keep2(d.m + i0);
        if (L2) wh[q] = ld_keep4(d.w + i0);
      }
#pragma unroll
      for (int q = 0; q < kAmaxGroups; ++q) {
        bad |= codes_at_least(gc[q].x, tadd) | codes_at_least(gc[q].y, tadd);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float2 g = mul2(dec2<GF>(code_pair(gc[q], j)), k2);
          if (L2) g = fma2(wd2, h2_to_f2(half_pair(wh[q], j)), g);
          if (GX) gx = max(gx, max(abs_bits(g.x), abs_bits(g.y)));
          const float2 m = fma2(b1, mul2(dec2<kE4M3>(code_pair(mc[q], j)), minv2),
                                mul2(omb1, g));
          mx = max(mx, max(abs_bits(m.x), abs_bits(m.y)));
        }
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < kAmaxGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          bad |= codes_at_least(d.g[i], tadd);
          float g = __fmul_rn(dec2<GF>(d.g[i]).x, k);
          if (L2) g = __fmaf_rn(s.wd, h_to_f(d.w[i]), g);
          if (GX) gx = max(gx, abs_bits(g));
          mx = max(mx, abs_bits(m_new1(dec2<kE4M3>(d.m[i]).x, minv, g, s)));
        }
      }
    }
  }
}

// k0: the unclipped factor inv_loss_scale / g_scale, which decides found_inf
// (GradScaler unscales, and finds any inf, before the norm is clipped); k:
// the factor the moments use (k0 times the clip coefficient, if any).
template <int GF, bool L2>
__device__ __forceinline__ void step_amax_dispatch(const StepDesc& d,
                                                   int64_t begin, int64_t end,
                                                   float k0, float k, float minv,
                                                   const StepScalars& s,
                                                   uint32_t& mx, uint32_t& gx,
                                                   uint32_t& bad) {
  const uint32_t tadd = threshold_addend(overflow_threshold<GF>(k0));
  if (d.v_bound != nullptr)
    thread_step_amax<GF, L2, true>(d, begin, end, k, minv, tadd, s, mx, gx, bad);
  else
    thread_step_amax<GF, L2, false>(d, begin, end, k, minv, tadd, s, mx, gx, bad);
}

template <bool L2, bool DEVS>
__global__ void __launch_bounds__(kThreads)
step_amax_kernel(const StepDesc* __restrict__ descs,
                 const Chunk* __restrict__ chunks, uint32_t nchunks,
                 StepScratch sc, StepScalars s, uint32_t epoch) {
  __shared__ uint32_t red[kThreads / 32];
  load_dev_scalars<DEVS>(s);
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const StepDesc d = descs[ch.tensor];
    const float gs = *d.g_scale, ms = *d.m_scale;
    if (ch.begin == 0 && threadIdx.x == 0) {
      sc.old_m_scale[ch.tensor] = ms;
      if (d.v_bound != nullptr) sc.old_v_bound[ch.tensor] = *d.v_bound;
    }
    const float k0 = __fdiv_rn(ils_of<DEVS>(s), gs);
    const float k = s.clip != nullptr ? __fmul_rn(k0, *s.clip) : k0;
    const float minv = __frcp_rn(ms);
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    uint32_t mx = 0, gx = 0, bad = 0;
    if (d.g_fmt == kE4M3)
      step_amax_dispatch<kE4M3, L2>(d, begin, end, k0, k, minv, s, mx, gx, bad);
    else
      step_amax_dispatch<kE5M2, L2>(d, begin, end, k0, k, minv, s, mx, gx, bad);
    mx = block_max_u32(mx, red);
    if (d.v_bound != nullptr) {   // uniform over the CTA
      gx = block_max_u32(gx, red);
      if (threadIdx.x == 0 && gx != 0)
        atomicMax(&sc.amax_g[ch.tensor], slot_tag(epoch, canon_amax_bits(gx)));
    }
    const int any_bad = __syncthreads_or(bad != 0);
    if (threadIdx.x == 0) {
      if (mx != 0) atomicMax(&sc.amax_m[ch.tensor], slot_tag(epoch, canon_amax_bits(mx)));
      if (any_bad) atomicMax(sc.found, slot_tag(epoch, 1u));
    }
  }
}

// ---------------------------------------------------------- pass 2: update

// Per-chunk constants of the update, as paired lanes.
struct UpdConsts {
  float2 k2, minv2, b1, omb1, b2, omb2, isbc2, eps2, nstep, decay, msc2, wd2,
      vinv2, vsc2;
};

template <bool DEVS>
__device__ __forceinline__ UpdConsts upd_consts(float k, float minv, float msc,
                                                float vinv, float vsc,
                                                const StepScalars& s) {
  UpdConsts c;
  c.k2 = splat2(k);
  c.minv2 = splat2(minv);
  c.b1 = splat2(s.beta1);
  c.omb1 = splat2(s.omb1);
  c.b2 = splat2(s.beta2);
  c.omb2 = splat2(s.omb2);
  if constexpr (DEVS) c.isbc2 = splat2(dev_sh.inv_sbc2);
  else c.isbc2 = splat2(s.inv_sbc2);
  c.eps2 = splat2(s.eps);
  if constexpr (DEVS) {
    c.nstep = splat2(-dev_sh.step_size);
    c.decay = splat2(dev_sh.decay);
  } else {
    c.nstep = splat2(-s.step_size);
    c.decay = splat2(s.decay);
  }
  c.msc2 = splat2(msc);
  c.wd2 = splat2(s.wd);
  c.vinv2 = splat2(vinv);
  c.vsc2 = splat2(vsc);
  return c;
}

// The update of eight elements: gradient codes gc, moment codes mc, FP16 v
// and w in; new moment codes, v and w out.  MCHECK: the first moment holds a
// non-finite value (its amax is not finite), so its codes take the explicit
// NaN code.  O3: also reduce the FP16 master's max |bits| per 16-bit lane
// into hmax.  VS: the second moment is scaled (read as FP16 * vinv, stored as
// FP16 of v * vsc).  L2: the gradient takes the decay term fma(wd, w, g).
template <int GF, bool O3, bool MCHECK, bool VS, bool L2>
__device__ __forceinline__ void update8(uint2 gc, uint2 mc, uint4 vh, uint4 wh,
                                        const UpdConsts& c, uint2& mo2,
                                        uint4& vo4, uint4& wo4, uint32_t& hmax) {
  uint32_t mo[4], vo[4], wo[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 g = mul2(dec2<GF>(code_pair(gc, j)), c.k2);
    if (L2) g = fma2(c.wd2, h2_to_f2(half_pair(wh, j)), g);
    const float2 m = fma2(c.b1, mul2(dec2<kE4M3>(code_pair(mc, j)), c.minv2),
                          mul2(c.omb1, g));
    float2 vp = h2_to_f2(half_pair(vh, j));
    if (VS) vp = mul2(vp, c.vinv2);
    const float2 v = fma2(c.b2, vp, mul2(c.omb2, mul2(g, g)));
    float2 sq;
    sq.x = __fsqrt_rn(v.x);
    sq.y = __fsqrt_rn(v.y);
    const float2 den = fma2(sq, c.isbc2, c.eps2);
    float2 u;
    u.x = __fdiv_rn(m.x, den.x);
    u.y = __fdiv_rn(m.y, den.y);
    const float2 w = fma2(c.nstep, u, mul2(h2_to_f2(half_pair(wh, j)), c.decay));
    const float2 mt = mul2(m, c.msc2);
    mo[j] = MCHECK ? (enc1_checked<kE4M3>(mt.x) | (enc1_checked<kE4M3>(mt.y) << 8))
                   : enc2<kE4M3>(mt.x, mt.y);
    vo[j] = f2_to_h2(VS ? mul2(v, c.vsc2) : v);
    wo[j] = f2_to_h2(w);
  }
  mo2 = make_uint2(mo[0] | (mo[1] << 16), mo[2] | (mo[3] << 16));
  vo4 = make_uint4(vo[0], vo[1], vo[2], vo[3]);
  wo4 = make_uint4(wo[0], wo[1], wo[2], wo[3]);
  if (O3) {
#pragma unroll
    for (int j = 0; j < 4; ++j) hmax = __vmaxu2(hmax, wo[j] & 0x7FFF7FFFu);
  }
}

// The update of this thread's share of [begin, end) from global memory.
template <int GF, bool O3, bool MCHECK, bool VS, bool L2, bool DEVS>
__device__ void thread_update(const StepDesc& d, int64_t begin, int64_t end,
                              float k, float minv, float msc, float vinv,
                              float vsc, const StepScalars& s, uint32_t& hmax) {
  constexpr int64_t kTile = (int64_t)kUpdThreads * kGroup * kUpdGroups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  // built here, so an instantiation keeps only the constants it uses
  const UpdConsts c = upd_consts<DEVS>(k, minv, msc, vinv, vsc, s);
  // One thread asks L2 for the tile FP8OPT_UPD_PREFETCH tiles ahead (whole
  // tiles of 16-byte-aligned tensors only), so the loads below find their
  // lines on chip while the DRAM reads for later tiles are already running.
  const bool pf = FP8OPT_UPD_PREFETCH > 0 && tid == 0 && vec &&
                  aligned16(d.g) && aligned16(d.m) && aligned16(d.v) &&
                  aligned16(d.w);
  for (int64_t base = begin; base < end; base += kTile) {
    if (pf) {
      const int64_t ahead = base + FP8OPT_UPD_PREFETCH * kTile;
      if (ahead + kTile <= end) {
        prefetch_l2(d.g + ahead, (uint32_t)kTile);
        prefetch_l2(d.m + ahead, (uint32_t)kTile);
        prefetch_l2(d.v + ahead, (uint32_t)(2 * kTile));
        prefetch_l2(d.w + ahead, (uint32_t)(2 * kTile));
      }
    }
    if (vec && base + kTile <= end) {
      uint2 gc[kUpdGroups], mc[kUpdGroups];
      uint4 vh[kUpdGroups], wh[kUpdGroups];
#pragma unroll
      for (int q = 0; q < kUpdGroups; ++q) {
        const int64_t i0 = base + q * (kUpdThreads * kGroup) + tid * kGroup;
        gc[q] = ld_once2(d.g + i0);
        mc[q] = ld_once2(d.m + i0);
        vh[q] = ld_once4(d.v + i0);
        wh[q] = ld_once4(d.w + i0);
      }
#pragma unroll
      for (int q = 0; q < kUpdGroups; ++q) {
        const int64_t i0 = base + q * (kUpdThreads * kGroup) + tid * kGroup;
        uint2 mo;
        uint4 vo, wo;
        update8<GF, O3, MCHECK, VS, L2>(gc[q], mc[q], vh[q], wh[q], c, mo, vo, wo,
                                        hmax);
        // streaming stores (evict-first): the new state is not read again
        // in this call.  Measured on the 6.7B list: 11.43 ms against 11.53.
        __stcs(reinterpret_cast<uint2*>(d.m + i0), mo);
        __stcs(reinterpret_cast<uint4*>(d.v + i0), vo);
        __stcs(reinterpret_cast<uint4*>(d.w + i0), wo);
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < kUpdGroups; ++q) {
        const int64_t i0 = base + q * (kUpdThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          const float wp = h_to_f(d.w[i]);
          float g = __fmul_rn(dec2<GF>(d.g[i]).x, k);
          if (L2) g = __fmaf_rn(s.wd, wp, g);
          const float m = m_new1(dec2<kE4M3>(d.m[i]).x, minv, g, s);
          float vp = h_to_f(d.v[i]);
          if (VS) vp = __fmul_rn(vp, vinv);
          float v, w;
          adamw1<DEVS>(g, m, vp, wp, s, v, w);
          const float mt = __fmul_rn(m, msc);
          d.m[i] = (uint8_t)(MCHECK ? enc1_checked<kE4M3>(mt)
                                    : (enc2<kE4M3>(mt, 0.0f) & 0xFFu));
          d.v[i] = f_to_h(VS ? __fmul_rn(v, vsc) : v);
          const uint16_t wn = f_to_h(w);
          d.w[i] = wn;
          if (O3) hmax = __vmaxu2(hmax, wn & 0x7FFFu);
        }
      }
    }
  }
}

template <int GF, bool O3, bool MCHECK, bool ANY_VS, bool L2, bool DEVS>
__device__ __forceinline__ void update_dispatch3(const StepDesc& d,
                                                 int64_t begin, int64_t end,
                                                 float k, float minv, float msc,
                                                 float vinv, float vsc,
                                                 const StepScalars& s,
                                                 uint32_t& hmax) {
  if (ANY_VS && d.v_bound != nullptr)
    thread_update<GF, O3, MCHECK, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc,
                                                    vinv, vsc, s, hmax);
  else
    thread_update<GF, O3, MCHECK, false, L2, DEVS>(d, begin, end, k, minv, msc,
                                                   vinv, vsc, s, hmax);
}

template <int GF, bool O3, bool ANY_VS, bool L2, bool DEVS>
__device__ __forceinline__ void update_dispatch2(const StepDesc& d,
                                                 int64_t begin, int64_t end,
                                                 float k, float minv, float msc,
                                                 float vinv, float vsc,
                                                 bool mcheck,
                                                 const StepScalars& s,
                                                 uint32_t& hmax) {
  if (mcheck)
    update_dispatch3<GF, O3, true, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc,
                                                     vinv, vsc, s, hmax);
  else
    update_dispatch3<GF, O3, false, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc,
                                                      vinv, vsc, s, hmax);
}

template <int GF, bool ANY_VS, bool L2, bool DEVS>
__device__ __forceinline__ void update_dispatch(const StepDesc& d,
                                                int64_t begin, int64_t end,
                                                float k, float minv, float msc,
                                                float vinv, float vsc,
                                                bool mcheck,
                                                const StepScalars& s,
                                                uint32_t& hmax) {
  if (d.o3)
    update_dispatch2<GF, true, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc, vinv,
                                                 vsc, mcheck, s, hmax);
  else
    update_dispatch2<GF, false, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc, vinv,
                                                  vsc, mcheck, s, hmax);
}

__device__ __forceinline__ bool found_set(const StepScratch& sc, uint32_t epoch) {
  return *reinterpret_cast<const volatile unsigned long long*>(sc.found) ==
         slot_tag(epoch, 1u);
}

// Several resident CTAs per SM keep enough warps to hide the latency of the
// square root and division sequences.  ANY_VS: some tensor of the call has a
// scaled second moment; L2: Adam with L2 decay.  Separate instantiations keep
// the plain AdamW kernel free of the other variants' registers.
template <bool ANY_VS, bool L2, bool DEVS>
__global__ void __launch_bounds__(kUpdThreads, (ANY_VS || L2 || DEVS)
                                                   ? FP8OPT_UPD_MIN_BLOCKS_VAR
                                                   : FP8OPT_UPD_MIN_BLOCKS)
step_update_kernel(const StepDesc* __restrict__ descs,
                   const Chunk* __restrict__ chunks, uint32_t nchunks,
                   StepScratch sc, StepScalars s, uint32_t epoch,
                   uint32_t* found_dev) {
  __shared__ uint32_t red[kUpdThreads / 32];
  const bool found = found_set(sc, epoch);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (found_dev != nullptr) *found_dev = found ? 1u : 0u;
    // the step count advances only when the step is taken
    if constexpr (DEVS) {
      if (!found) *s.step_out = s.dev->t;
    }
  }
  if (found) return;
  load_dev_scalars<DEVS>(s);
  for (uint32_t r = blockIdx.x; r < nchunks; r += gridDim.x) {
    const Chunk ch = chunks[nchunks - 1 - r];
    const StepDesc d = descs[ch.tensor];
    float k = __fdiv_rn(ils_of<DEVS>(s), *d.g_scale);
    if (s.clip != nullptr) k = __fmul_rn(k, *s.clip);
    const float minv = __frcp_rn(sc.old_m_scale[ch.tensor]);
    const uint32_t am = slot_value(sc.amax_m[ch.tensor], epoch);
    const float msc = scale_from_amax_bits(am, 448.0f);
    float vinv = 1.0f, vsc = 1.0f;
    if (ANY_VS && d.v_bound != nullptr) {
      // bound of this step: fma(beta2, old bound, (1 - beta2) * gmax^2)
      const float b_old = sc.old_v_bound[ch.tensor];
      const float gmax = __uint_as_float(slot_value(sc.amax_g[ch.tensor], epoch));
      const float b_new = __fmaf_rn(s.beta2, b_old,
                                    __fmul_rn(s.omb2, __fmul_rn(gmax, gmax)));
      vinv = __fmul_rn(b_old, 0x1p-14f);
      vsc = v_scale_from_bound(b_new);
      if (ch.begin == 0 && threadIdx.x == 0) *d.v_bound = b_new;
    }
    if (ch.begin == 0 && threadIdx.x == 0) *d.m_scale = msc;
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    const bool mcheck = am >= 0x7F800000u;
    uint32_t hmax = 0;
    if (d.g_fmt == kE4M3)
      update_dispatch<kE4M3, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc, vinv,
                                               vsc, mcheck, s, hmax);
    else
      update_dispatch<kE5M2, ANY_VS, L2, DEVS>(d, begin, end, k, minv, msc, vinv,
                                               vsc, mcheck, s, hmax);
    if (d.o3) {   // uniform over the CTA
      uint32_t h = max(hmax & 0xFFFFu, hmax >> 16);
      h = block_max_u32<kUpdThreads>(h, red);
      if (threadIdx.x == 0 && h != 0) {
        const uint32_t fb = h > 0x7C00u ? 0x7FC00000u
                                        : __float_as_uint(h_to_f((uint16_t)h));
        atomicMax(&sc.amax_w[ch.tensor], slot_tag(epoch, fb));
      }
    }
  }
}

// ------------------------------------------------- pass 3: O3 weight copy

template <bool CHECKED>
__device__ void thread_w8(const StepDesc& d, int64_t begin, int64_t end,
                          float scale) {
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kW8Groups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  const float2 sc2 = splat2(scale);
  for (int64_t base = begin; base < end; base += kTile) {
    if (vec && base + kTile <= end) {
      uint4 wh[kW8Groups];
#pragma unroll
      for (int q = 0; q < kW8Groups; ++q)
        wh[q] = ld_once4(d.w + base + q * (kThreads * kGroup) + tid * kGroup);
#pragma unroll
      for (int q = 0; q < kW8Groups; ++q) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 t = mul2(h2_to_f2(half_pair(wh[q], j)), sc2);
          o[j] = CHECKED ? (enc1_checked<kE4M3>(t.x) | (enc1_checked<kE4M3>(t.y) << 8))
                         : enc2<kE4M3>(t.x, t.y);
        }
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        *reinterpret_cast<uint2*>(d.w8 + i0) =
            make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < kW8Groups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          const float t = __fmul_rn(h_to_f(d.w[i]), scale);
          d.w8[i] = (uint8_t)(CHECKED ? enc1_checked<kE4M3>(t)
                                      : (enc2<kE4M3>(t, 0.0f) & 0xFFu));
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads)
step_w8_kernel(const StepDesc* __restrict__ descs,
               const Chunk* __restrict__ chunks, uint32_t nchunks,
               StepScratch sc, uint32_t epoch) {
  if (found_set(sc, epoch)) return;
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const StepDesc d = descs[ch.tensor];
    const uint32_t ab = slot_value(sc.amax_w[ch.tensor], epoch);
    const float scale = scale_from_amax_bits(ab, 448.0f);
    if (ch.begin == 0 && threadIdx.x == 0) {
      *d.w8_amax = __uint_as_float(ab);
      *d.w8_scale = scale;
    }
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    if (ab >= 0x7F800000u)
      thread_w8<true>(d, begin, end, scale);
    else
      thread_w8<false>(d, begin, end, scale);
  }
}

}  // namespace

// The update pass, then (for O3 chunks) the weight-copy pass.  any_vs: some
// record has a scaled second moment.  grid_update sizes the plain AdamW
// instantiation, grid_update_var the scaled-v, L2 and device-resident ones.
cudaError_t launch_step_update(const StepDesc* descs, const Chunk* chunks,
                               uint32_t nchunks, const Chunk* chunks_o3,
                               uint32_t nchunks_o3, const StepScratch& sc,
                               const StepScalars& s, uint32_t epoch,
                               uint32_t* found_dev, int grid_update,
                               int grid_update_var, int grid_w8,
                               bool any_vs, cudaStream_t stream,
                               LaunchMark mark) {
  if (mark) mark(kStepUpdateK, 0, stream);
  const bool dev = s.dev != nullptr;
  const uint32_t g = grid_min(
      (uint32_t)(any_vs || s.l2 || dev ? grid_update_var : grid_update), nchunks);
  const int v = (any_vs ? 4 : 0) | (s.l2 ? 2 : 0) | (dev ? 1 : 0);
  switch (v) {
#define FP8OPT_UPDATE_CASE(VS, L2, DEVS)                                     \
  case (VS ? 4 : 0) | (L2 ? 2 : 0) | (DEVS ? 1 : 0):                         \
    step_update_kernel<VS, L2, DEVS><<<g, kUpdThreads, 0, stream>>>(         \
        descs, chunks, nchunks, sc, s, epoch, found_dev);                    \
    break;
    FP8OPT_UPDATE_CASE(false, false, false)
    FP8OPT_UPDATE_CASE(false, false, true)
    FP8OPT_UPDATE_CASE(false, true, false)
    FP8OPT_UPDATE_CASE(false, true, true)
    FP8OPT_UPDATE_CASE(true, false, false)
    FP8OPT_UPDATE_CASE(true, false, true)
    FP8OPT_UPDATE_CASE(true, true, false)
    FP8OPT_UPDATE_CASE(true, true, true)
#undef FP8OPT_UPDATE_CASE
  }
  if (mark) mark(kStepUpdateK, 1, stream);
  if (nchunks_o3 != 0) {
    if (mark) mark(kStepW8K, 0, stream);
    step_w8_kernel<<<grid_min((uint32_t)grid_w8, nchunks_o3), kThreads, 0,
                     stream>>>(descs, chunks_o3, nchunks_o3, sc, epoch);
    if (mark) mark(kStepW8K, 1, stream);
  }
  return cudaGetLastError();
}

// The O3 weight-copy pass alone, for an update pass launched without it
// (the split step: the master's amax is combined over ranks in between).
cudaError_t launch_step_w8(const StepDesc* descs, const Chunk* chunks_o3,
                           uint32_t nchunks_o3, const StepScratch& sc,
                           uint32_t epoch, int grid_w8, cudaStream_t stream,
                           LaunchMark mark) {
  if (nchunks_o3 == 0) return cudaSuccess;
  if (mark) mark(kStepW8K, 0, stream);
  step_w8_kernel<<<grid_min((uint32_t)grid_w8, nchunks_o3), kThreads, 0, stream>>>(
      descs, chunks_o3, nchunks_o3, sc, epoch);
  if (mark) mark(kStepW8K, 1, stream);
  return cudaGetLastError();
}

// The first pass alone (found_inf, the amax of the new first moment, max |g|).
cudaError_t launch_step_amax(const StepDesc* descs, const Chunk* chunks,
                             uint32_t nchunks, const StepScratch& sc,
                             const StepScalars& s, uint32_t epoch, int grid_amax,
                             cudaStream_t stream, LaunchMark mark) {
  if (nchunks == 0) return cudaSuccess;
  if (mark) mark(kStepAmaxK, 0, stream);
  const uint32_t ga = grid_min((uint32_t)grid_amax, nchunks);
  if (s.l2 && s.dev)
    step_amax_kernel<true, true><<<ga, kThreads, 0, stream>>>(descs, chunks,
                                                              nchunks, sc, s, epoch);
  else if (s.l2)
    step_amax_kernel<true, false><<<ga, kThreads, 0, stream>>>(descs, chunks,
                                                               nchunks, sc, s, epoch);
  else if (s.dev)
    step_amax_kernel<false, true><<<ga, kThreads, 0, stream>>>(descs, chunks,
                                                               nchunks, sc, s, epoch);
  else
    step_amax_kernel<false, false><<<ga, kThreads, 0, stream>>>(descs, chunks,
                                                                nchunks, sc, s, epoch);
  if (mark) mark(kStepAmaxK, 1, stream);
  return cudaGetLastError();
}

cudaError_t launch_step(const StepDesc* descs, const Chunk* chunks,
                        uint32_t nchunks, const Chunk* chunks_o3,
                        uint32_t nchunks_o3, const StepScratch& sc,
                        const StepScalars& s, uint32_t epoch,
                        uint32_t* found_dev, int grid_amax, int grid_update,
                        int grid_update_var,
                        int grid_w8, bool any_vs, cudaStream_t stream,
                        LaunchMark mark) {
  if (nchunks == 0) {
    if (found_dev) return cudaMemsetAsync(found_dev, 0, sizeof(uint32_t), stream);
    return cudaSuccess;
  }
  cudaError_t e = launch_step_amax(descs, chunks, nchunks, sc, s, epoch,
                                   grid_amax, stream, mark);
  if (e != cudaSuccess) return e;
  return launch_step_update(descs, chunks, nchunks, chunks_o3, nchunks_o3, sc, s,
                            epoch, found_dev, grid_update, grid_update_var,
                            grid_w8, any_vs,
                            stream, mark);
}

namespace {

// beta^t in double by binary exponentiation, each product rounded to double:
// the host's bias power, bit for bit.
__device__ double bias_power(double b, long long t) {
  double r = 1.0;
  while (t > 0) {
    if (t & 1) r = __dmul_rn(r, b);
    b = __dmul_rn(b, b);
    t >>= 1;
  }
  return r;
}

// One thread: the scalars of step t = state->step + 1 from the caller's
// device-resident lr and inv_loss_scale, with the host's arithmetic (the
// bias corrections in double, each result rounded to float once).  commit:
// also store t (a call with no chunks, whose update pass does not run).
__global__ void step_scalars_kernel(DevState* state, float beta1, float beta2,
                                    float wd, int l2, DevScalars* out,
                                    int commit) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const long long t = state->step + 1;
  const float lr = state->lr;
  const double bc1 = __dsub_rn(1.0, bias_power((double)beta1, t));
  const double bc2 = __dsub_rn(1.0, bias_power((double)beta2, t));
  DevScalars d;
  d.step_size = (float)__ddiv_rn((double)lr, bc1);
  d.inv_sbc2 = (float)__ddiv_rn(1.0, __dsqrt_rn(bc2));
  d.decay = l2 ? 1.0f : __fsub_rn(1.0f, __fmul_rn(lr, wd));
  d.ils = state->inv_loss_scale;
  d.t = t;
  *out = d;
  if (commit) state->step = t;
}

}  // namespace

// Writes the scalars of the next step of `state` to `out` (one thread).
cudaError_t launch_step_scalars(DevState* state, float beta1, float beta2,
                                float wd, bool l2, DevScalars* out, bool commit,
                                cudaStream_t stream) {
  step_scalars_kernel<<<1, 32, 0, stream>>>(state, beta1, beta2, wd, l2 ? 1 : 0,
                                            out, commit ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t step_occupancy(int* amax_per_sm, int* update_per_sm,
                           int* update_var_per_sm, int* w8_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      amax_per_sm, step_amax_kernel<false, false>, kThreads, 0);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      update_per_sm, step_update_kernel<false, false, false>, kUpdThreads, 0);
  if (e != cudaSuccess) return e;
  // the least of the instantiations that share grid_update_var
  int lo = 0;
  const void* vars[] = {
      (const void*)step_update_kernel<false, false, true>,
      (const void*)step_update_kernel<false, true, false>,
      (const void*)step_update_kernel<false, true, true>,
      (const void*)step_update_kernel<true, false, false>,
      (const void*)step_update_kernel<true, false, true>,
      (const void*)step_update_kernel<true, true, false>,
      (const void*)step_update_kernel<true, true, true>};
  for (const void* k : vars) {
    int b = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k, kUpdThreads, 0);
    if (e != cudaSuccess) return e;
    lo = (lo == 0 || b < lo) ? b : lo;
  }
  *update_var_per_sm = lo;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(w8_per_sm,
                                                       step_w8_kernel, kThreads, 0);
}

}  // namespace fp8opt
