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
// Every product and sum is rounded on its own (the file is compiled without
// multiply-add contraction), in the order of the definition, so the first
// moment, and with it its amax and scale, is bit-identical to a scalar fp32
// evaluation of the same expression.
#include "fp8opt_internal.cuh"

namespace fp8opt {

namespace {

constexpr int kAmaxGroups = 2;   // 8-element groups per thread per tile
constexpr int kUpdGroups = 2;

// Unscaled gradients of eight codes: decode, times 1/g_scale, times the
// inverse loss scale.
template <int GF>
__device__ __forceinline__ void grad8(uint2 gc, float ginv, float ils,
                                      float (&g)[8]) {
  dec8<GF>(gc, g);
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = __fmul_rn(__fmul_rn(g[j], ginv), ils);
}

__device__ __forceinline__ float m_new(float mdec, float minv, float g,
                                       const StepScalars& s) {
  const float mp = __fmul_rn(mdec, minv);
  return __fadd_rn(__fmul_rn(s.beta1, mp), __fmul_rn(s.omb1, g));
}

__device__ __forceinline__ uint32_t nonfinite(float x) {
  return (__float_as_uint(x) & 0x7FFFFFFFu) >= 0x7F800000u;
}

// ------------------------------------------------------------ pass 1: amax

// SAFE: every finite gradient code unscales to a finite value (checked once
// per chunk from the largest code), so found_inf only needs the codes.
template <int GF, bool SAFE>
__device__ void thread_step_amax(const StepDesc& d, int64_t begin, int64_t end,
                                 float ginv, float minv, const StepScalars& s,
                                 uint32_t& mx, uint32_t& bad) {
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kAmaxGroups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  for (int64_t base = begin; base < end; base += kTile) {
    if (vec && base + kTile <= end) {
      uint2 gc[kAmaxGroups], mc[kAmaxGroups];
#pragma unroll
      for (int k = 0; k < kAmaxGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        gc[k] = ld_keep2(d.g + i0);
        mc[k] = ld_keep2(d.m + i0);
      }
#pragma unroll
      for (int k = 0; k < kAmaxGroups; ++k) {
        float g[8], md[8];
        grad8<GF>(gc[k], ginv, s.ils, g);
        dec8<kE4M3>(mc[k], md);
        if (SAFE) {
          bad |= nonfinite_code_bytes<GF>(gc[k].x) | nonfinite_code_bytes<GF>(gc[k].y);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (!SAFE) bad |= nonfinite(g[j]);
          mx = max(mx, __float_as_uint(m_new(md[j], minv, g[j], s)) & 0x7FFFFFFFu);
        }
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < kAmaxGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          const float gd = dec2<GF>(d.g[i]).x;
          const float g = __fmul_rn(__fmul_rn(gd, ginv), s.ils);
          bad |= nonfinite(g);
          const float md = dec2<kE4M3>(d.m[i]).x;
          mx = max(mx, __float_as_uint(m_new(md, minv, g, s)) & 0x7FFFFFFFu);
        }
      }
    }
  }
}

template <int GF>
__device__ __forceinline__ void step_amax_dispatch(const StepDesc& d,
                                                   int64_t begin, int64_t end,
                                                   float ginv, float minv,
                                                   const StepScalars& s,
                                                   uint32_t& mx, uint32_t& bad) {
  // The largest finite code unscales to the largest |g|; rounding is
  // monotonic, so if that is finite every finite code gives a finite g.
  const float gmax = __fmul_rn(__fmul_rn(fp8_max_of<GF>(), ginv), fabsf(s.ils));
  if (!nonfinite(__fmul_rn(fp8_max_of<GF>(), ginv)) && !nonfinite(gmax))
    thread_step_amax<GF, true>(d, begin, end, ginv, minv, s, mx, bad);
  else
    thread_step_amax<GF, false>(d, begin, end, ginv, minv, s, mx, bad);
}

__global__ void __launch_bounds__(kThreads)
step_amax_kernel(const StepDesc* __restrict__ descs,
                 const Chunk* __restrict__ chunks, uint32_t nchunks,
                 StepScratch sc, StepScalars s, uint32_t epoch) {
  __shared__ uint32_t red[kThreads / 32];
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const StepDesc d = descs[ch.tensor];
    const float gs = *d.g_scale, ms = *d.m_scale;
    if (ch.index == 0 && threadIdx.x == 0) sc.old_m_scale[ch.tensor] = ms;
    const float ginv = __frcp_rn(gs), minv = __frcp_rn(ms);
    const int64_t begin = (int64_t)ch.index * kChunkElems;
    const int64_t end = min(begin + kChunkElems, d.numel);
    uint32_t mx = 0, bad = 0;
    if (d.g_fmt == kE4M3)
      step_amax_dispatch<kE4M3>(d, begin, end, ginv, minv, s, mx, bad);
    else
      step_amax_dispatch<kE5M2>(d, begin, end, ginv, minv, s, mx, bad);
    mx = block_max_u32(mx, red);
    const int any_bad = __syncthreads_or(bad != 0);
    if (threadIdx.x == 0) {
      if (mx != 0) atomicMax(&sc.amax_m[ch.tensor], slot_tag(epoch, canon_amax_bits(mx)));
      if (any_bad) atomicMax(sc.found, slot_tag(epoch, 1u));
    }
  }
}

// ---------------------------------------------------------- pass 2: update

// The update of one element; returns the new fp32 m, v and w.
__device__ __forceinline__ void adamw1(float g, float mdec, float minv,
                                       float vp, float wp, const StepScalars& s,
                                       float& m, float& v, float& w) {
  m = m_new(mdec, minv, g, s);
  v = __fadd_rn(__fmul_rn(s.beta2, vp), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.sbc2), s.eps);
  const float upd = __fdiv_rn(__fdiv_rn(m, s.bc1), denom);
  w = __fsub_rn(__fmul_rn(wp, s.decay), __fmul_rn(s.lr, upd));
}

// MCHECK: the first moment holds a non-finite value (its amax is not
// finite), so its codes take the explicit NaN code.  O3: also reduce the
// FP16 master's max |bits| per 16-bit lane into hmax.
template <int GF, bool O3, bool MCHECK>
__device__ void thread_update(const StepDesc& d, int64_t begin, int64_t end,
                              float ginv, float minv, float msc,
                              const StepScalars& s, uint32_t& hmax) {
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kUpdGroups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  for (int64_t base = begin; base < end; base += kTile) {
    if (vec && base + kTile <= end) {
      uint2 gc[kUpdGroups], mc[kUpdGroups];
      uint4 vh[kUpdGroups], wh[kUpdGroups];
#pragma unroll
      for (int k = 0; k < kUpdGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        gc[k] = ld_once2(d.g + i0);
        mc[k] = ld_once2(d.m + i0);
        vh[k] = ld_once4(d.v + i0);
        wh[k] = ld_once4(d.w + i0);
      }
#pragma unroll
      for (int k = 0; k < kUpdGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        float g[8], md[8], vp[8], wp[8], m[8], v[8], w[8];
        grad8<GF>(gc[k], ginv, s.ils, g);
        dec8<kE4M3>(mc[k], md);
        h8_to_f(vh[k], vp);
        h8_to_f(wh[k], wp);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          adamw1(g[j], md[j], minv, vp[j], wp[j], s, m[j], v[j], w[j]);
          m[j] = __fmul_rn(m[j], msc);
        }
        *reinterpret_cast<uint2*>(d.m + i0) = enc8<kE4M3, MCHECK>(m);
        *reinterpret_cast<uint4*>(d.v + i0) = f_to_h8(v);
        const uint4 wn = f_to_h8(w);
        *reinterpret_cast<uint4*>(d.w + i0) = wn;
        if (O3) {
          hmax = __vmaxu2(hmax, wn.x & 0x7FFF7FFFu);
          hmax = __vmaxu2(hmax, wn.y & 0x7FFF7FFFu);
          hmax = __vmaxu2(hmax, wn.z & 0x7FFF7FFFu);
          hmax = __vmaxu2(hmax, wn.w & 0x7FFF7FFFu);
        }
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < kUpdGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          const float gd = dec2<GF>(d.g[i]).x;
          const float g = __fmul_rn(__fmul_rn(gd, ginv), s.ils);
          const float md = dec2<kE4M3>(d.m[i]).x;
          float m, v, w;
          adamw1(g, md, minv, h_to_f(d.v[i]), h_to_f(d.w[i]), s, m, v, w);
          const float mt = __fmul_rn(m, msc);
          d.m[i] = (uint8_t)(MCHECK ? enc1_checked<kE4M3>(mt)
                                    : (enc2<kE4M3>(mt, 0.0f) & 0xFFu));
          d.v[i] = f_to_h(v);
          const uint16_t wn = f_to_h(w);
          d.w[i] = wn;
          if (O3) hmax = __vmaxu2(hmax, wn & 0x7FFFu);
        }
      }
    }
  }
}

template <int GF, bool O3>
__device__ __forceinline__ void update_dispatch2(const StepDesc& d,
                                                 int64_t begin, int64_t end,
                                                 float ginv, float minv,
                                                 float msc, bool mcheck,
                                                 const StepScalars& s,
                                                 uint32_t& hmax) {
  if (mcheck)
    thread_update<GF, O3, true>(d, begin, end, ginv, minv, msc, s, hmax);
  else
    thread_update<GF, O3, false>(d, begin, end, ginv, minv, msc, s, hmax);
}

template <int GF>
__device__ __forceinline__ void update_dispatch(const StepDesc& d,
                                                int64_t begin, int64_t end,
                                                float ginv, float minv,
                                                float msc, bool mcheck,
                                                const StepScalars& s,
                                                uint32_t& hmax) {
  if (d.w8 != nullptr)
    update_dispatch2<GF, true>(d, begin, end, ginv, minv, msc, mcheck, s, hmax);
  else
    update_dispatch2<GF, false>(d, begin, end, ginv, minv, msc, mcheck, s, hmax);
}

__device__ __forceinline__ bool found_set(const StepScratch& sc, uint32_t epoch) {
  return *reinterpret_cast<const volatile unsigned long long*>(sc.found) ==
         slot_tag(epoch, 1u);
}

__global__ void __launch_bounds__(kThreads)
step_update_kernel(const StepDesc* __restrict__ descs,
                   const Chunk* __restrict__ chunks, uint32_t nchunks,
                   StepScratch sc, StepScalars s, uint32_t epoch,
                   uint32_t* found_dev) {
  __shared__ uint32_t red[kThreads / 32];
  const bool found = found_set(sc, epoch);
  if (found_dev != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *found_dev = found ? 1u : 0u;
  if (found) return;
  for (uint32_t r = blockIdx.x; r < nchunks; r += gridDim.x) {
    const Chunk ch = chunks[nchunks - 1 - r];
    const StepDesc d = descs[ch.tensor];
    const float ginv = __frcp_rn(*d.g_scale);
    const float minv = __frcp_rn(sc.old_m_scale[ch.tensor]);
    const uint32_t am = slot_value(sc.amax_m[ch.tensor], epoch);
    const float msc = scale_from_amax_bits(am, 448.0f);
    if (ch.index == 0 && threadIdx.x == 0) *d.m_scale = msc;
    const int64_t begin = (int64_t)ch.index * kChunkElems;
    const int64_t end = min(begin + kChunkElems, d.numel);
    const bool mcheck = am >= 0x7F800000u;
    uint32_t hmax = 0;
    if (d.g_fmt == kE4M3)
      update_dispatch<kE4M3>(d, begin, end, ginv, minv, msc, mcheck, s, hmax);
    else
      update_dispatch<kE5M2>(d, begin, end, ginv, minv, msc, mcheck, s, hmax);
    if (d.w8 != nullptr) {   // uniform over the CTA
      uint32_t h = max(hmax & 0xFFFFu, hmax >> 16);
      h = block_max_u32(h, red);
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
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kUpdGroups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  for (int64_t base = begin; base < end; base += kTile) {
    if (vec && base + kTile <= end) {
      uint4 wh[kUpdGroups];
#pragma unroll
      for (int k = 0; k < kUpdGroups; ++k)
        wh[k] = ld_once4(d.w + base + k * (kThreads * kGroup) + tid * kGroup);
#pragma unroll
      for (int k = 0; k < kUpdGroups; ++k) {
        float x[8];
        h8_to_f(wh[k], x);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(x[j], scale);
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        *reinterpret_cast<uint2*>(d.w8 + i0) = enc8<kE4M3, CHECKED>(x);
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < kUpdGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
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
    if (ch.index == 0 && threadIdx.x == 0) {
      *d.w8_amax = __uint_as_float(ab);
      *d.w8_scale = scale;
    }
    const int64_t begin = (int64_t)ch.index * kChunkElems;
    const int64_t end = min(begin + kChunkElems, d.numel);
    if (ab >= 0x7F800000u)
      thread_w8<true>(d, begin, end, scale);
    else
      thread_w8<false>(d, begin, end, scale);
  }
}

}  // namespace

cudaError_t launch_step(const StepDesc* descs, const Chunk* chunks,
                        uint32_t nchunks, const Chunk* chunks_o3,
                        uint32_t nchunks_o3, const StepScratch& sc,
                        const StepScalars& s, uint32_t epoch,
                        uint32_t* found_dev, int grid_amax, int grid_update,
                        int grid_w8, cudaStream_t stream, LaunchMark mark) {
  if (nchunks == 0) {
    if (found_dev) return cudaMemsetAsync(found_dev, 0, sizeof(uint32_t), stream);
    return cudaSuccess;
  }
  if (mark) mark(kStepAmaxK, 0, stream);
  step_amax_kernel<<<grid_min((uint32_t)grid_amax, nchunks), kThreads, 0,
                     stream>>>(descs, chunks, nchunks, sc, s, epoch);
  if (mark) mark(kStepAmaxK, 1, stream);
  if (mark) mark(kStepUpdateK, 0, stream);
  step_update_kernel<<<grid_min((uint32_t)grid_update, nchunks), kThreads,
                       0, stream>>>(descs, chunks, nchunks, sc, s, epoch,
                                    found_dev);
  if (mark) mark(kStepUpdateK, 1, stream);
  if (nchunks_o3 != 0) {
    if (mark) mark(kStepW8K, 0, stream);
    step_w8_kernel<<<grid_min((uint32_t)grid_w8, nchunks_o3), kThreads, 0,
                     stream>>>(descs, chunks_o3, nchunks_o3, sc, epoch);
    if (mark) mark(kStepW8K, 1, stream);
  }
  return cudaGetLastError();
}

cudaError_t step_occupancy(int* amax_per_sm, int* update_per_sm,
                           int* w8_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      amax_per_sm, step_amax_kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      update_per_sm, step_update_kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(w8_per_sm,
                                                       step_w8_kernel, kThreads, 0);
}

}  // namespace fp8opt
