// The scaled FP8 cast of the gradients fused with the AdamW step
// (fp8_cast_adamw_step): the same results as fp8_cast_scaled followed by
// fp8_adamw_step on the codes it wrote, with one pass fewer over memory.
//
// Passes:
//   cast_amax_kernel        per-tensor gradient amax (cast_kernels.cu)
//   cast_step_amax_kernel   this file: encode the gradients with their
//                           just-in-time scale and write the codes, then, from
//                           the codes just produced, the step's first pass:
//                           found_inf and the amax of this step's fp32 first
//                           moment.  Reads 2 B (BF16/FP16) + 1 B (m), writes
//                           1 B per param, where the unfused path reads the
//                           source and writes the codes in one pass and reads
//                           the codes and m again in the next.
//   step_update_kernel      (and step_w8_kernel for O3), step_kernels.cu
// BF16 in, the whole step moves 2 + 4 + 11 = 17 B per param (O2).
//
// The arithmetic is the one of the two separate entry points, line by line:
// the cast's t = x * scale (one rounding) and its encode; the step's
// g = dec(code) * k with k = inv_loss_scale / g_scale computed from the same
// fp32 scale the cast writes; m = fma(beta1, dec(m) * minv, (1 - beta1) * g).
#include "fp8opt_internal.cuh"

namespace fp8opt {

cudaError_t launch_cast_amax(const CastDesc* descs, const Chunk* chunks,
                             uint32_t nchunks, unsigned long long* slots,
                             uint32_t epoch, int grid_amax, cudaStream_t stream,
                             LaunchMark mark);
cudaError_t launch_step_update(const StepDesc* descs, const Chunk* chunks,
                               uint32_t nchunks, const Chunk* chunks_o3,
                               uint32_t nchunks_o3, const StepScratch& sc,
                               const StepScalars& s, uint32_t epoch,
                               uint32_t* found_dev, int grid_update,
                               int grid_update_var, int grid_w8,
                               bool any_vs, cudaStream_t stream,
                               LaunchMark mark);

namespace {

constexpr int kFusedGroups = 2;   // 8-element groups per thread per tile

// Tiles ahead of the current one prefetched into L2 (0: none).
#ifndef FP8OPT_FUSED_PREFETCH
#define FP8OPT_FUSED_PREFETCH 1
#endif

// Encode eight values (CHECKED: explicit codes for non-finite inputs).
template <int FMT, bool CHECKED>
__device__ __forceinline__ uint32_t enc_pair(float2 t) {
  return CHECKED ? (enc1_checked<FMT>(t.x) | (enc1_checked<FMT>(t.y) << 8))
                 : enc2<FMT>(t.x, t.y);
}

// This thread's share of [begin, end): encode, store the codes, and fold the
// step's first pass into mx (max |m| bits), gx (max |g| bits, when GX: for a
// scaled second moment) and bad (non-finite gradient: a code magnitude at or
// above the threshold whose addend is tadd, as in the unfused first pass).
// L2 (Adam with L2 decay): the gradient takes the decay term fma(wd, w, g),
// as in the unfused first pass, so the master weights are read too.
template <int DT, int FMT, bool CHECKED, bool GX, bool L2>
__device__ void thread_cast_step(const CastDesc& cd, const StepDesc& sd,
                                 int64_t begin, int64_t end, float scale,
                                 float k, float minv, uint32_t tadd,
                                 const StepScalars& s, uint32_t& mx,
                                 uint32_t& gx, uint32_t& bad) {
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kFusedGroups;
  const int tid = threadIdx.x;
  const bool vec = cd.vec_ok != 0 && sd.vec_ok != 0;
  const float2 sc2 = splat2(scale), k2 = splat2(k), minv2 = splat2(minv),
               b1 = splat2(s.beta1), omb1 = splat2(s.omb1), wd2 = splat2(s.wd);
  constexpr uint32_t kSrcBytes = DT == kF32 ? 4 : 2;
  const bool pf = FP8OPT_FUSED_PREFETCH > 0 && tid == 0 && vec &&
                  aligned16(cd.src) && aligned16(sd.m);
  for (int64_t base = begin; base < end; base += kTile) {
    if (pf) {
      const int64_t ahead = base + FP8OPT_FUSED_PREFETCH * kTile;
      if (ahead + kTile <= end) {
        prefetch_l2(static_cast<const char*>(cd.src) + ahead * kSrcBytes,
                    (uint32_t)(kSrcBytes * kTile));
        prefetch_l2(sd.m + ahead, (uint32_t)kTile);
        if (L2) prefetch_l2(sd.w + ahead, (uint32_t)(2 * kTile));
      }
    }
    if (vec && base + kTile <= end) {
      float x[kFusedGroups][8];
      uint2 mc[kFusedGroups];
      uint4 wh[kFusedGroups];
#pragma unroll
      for (int q = 0; q < kFusedGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        load8<DT>(cd.src, i0, x[q]);
        mc[q] = ld_keep2(sd.m + i0);
        if (L2) wh[q] = ld_keep4(sd.w + i0);
      }
#pragma unroll
      for (int q = 0; q < kFusedGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          c[j] = enc_pair<FMT, CHECKED>(mul2(make_float2(x[q][2 * j], x[q][2 * j + 1]), sc2));
        const uint2 codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        *reinterpret_cast<uint2*>(cd.codes + i0) = codes;
        bad |= codes_at_least(codes.x, tadd) | codes_at_least(codes.y, tadd);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float2 g = mul2(dec2<FMT>(c[j]), k2);
          if (L2) g = fma2(wd2, h2_to_f2(half_pair(wh[q], j)), g);
          if (GX) gx = max(gx, max(abs_bits(g.x), abs_bits(g.y)));
          const float2 m = fma2(b1, mul2(dec2<kE4M3>(code_pair(mc[q], j)), minv2),
                                mul2(omb1, g));
          mx = max(mx, max(abs_bits(m.x), abs_bits(m.y)));
        }
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < kFusedGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          const float t = __fmul_rn(load1<DT>(cd.src, i), scale);
          const uint32_t code = CHECKED ? enc1_checked<FMT>(t)
                                        : (enc2<FMT>(t, 0.0f) & 0xFFu);
          cd.codes[i] = (uint8_t)code;
          bad |= codes_at_least(code, tadd);
          float g = __fmul_rn(dec2<FMT>(code).x, k);
          if (L2) g = __fmaf_rn(s.wd, h_to_f(sd.w[i]), g);
          if (GX) gx = max(gx, abs_bits(g));
          const float mp = __fmul_rn(dec2<kE4M3>(sd.m[i]).x, minv);
          mx = max(mx, abs_bits(__fmaf_rn(s.beta1, mp, __fmul_rn(s.omb1, g))));
        }
      }
    }
  }
}

template <int DT, int FMT, bool GX, bool L2>
__device__ __forceinline__ void cast_step_dispatch2(const CastDesc& cd,
                                                    const StepDesc& sd,
                                                    int64_t begin, int64_t end,
                                                    float scale, float k,
                                                    float minv, bool checked,
                                                    const StepScalars& s,
                                                    uint32_t& mx, uint32_t& gx,
                                                    uint32_t& bad) {
  // As in the unfused step: found_inf from the codes and the threshold of k.
  const uint32_t tadd = threshold_addend(overflow_threshold<FMT>(k));
  if (checked)
    thread_cast_step<DT, FMT, true, GX, L2>(cd, sd, begin, end, scale, k, minv, tadd, s, mx, gx, bad);
  else
    thread_cast_step<DT, FMT, false, GX, L2>(cd, sd, begin, end, scale, k, minv, tadd, s, mx, gx, bad);
}

template <int DT, int FMT, bool ANY_VS, bool L2>
__device__ __forceinline__ void cast_step_dispatch(const CastDesc& cd,
                                                   const StepDesc& sd,
                                                   int64_t begin, int64_t end,
                                                   float scale, float k,
                                                   float minv, bool checked,
                                                   const StepScalars& s,
                                                   uint32_t& mx, uint32_t& gx,
                                                   uint32_t& bad) {
  if (ANY_VS && sd.v_bound != nullptr)
    cast_step_dispatch2<DT, FMT, true, L2>(cd, sd, begin, end, scale, k, minv,
                                           checked, s, mx, gx, bad);
  else
    cast_step_dispatch2<DT, FMT, false, L2>(cd, sd, begin, end, scale, k, minv,
                                            checked, s, mx, gx, bad);
}

// At most 64 registers a thread: 4 resident CTAs per SM.  ANY_VS: some
// tensor of the call has a scaled second moment.  DEVS: inv_loss_scale comes
// from the device-resident step (StepScalars::dev).  L2: Adam with L2 decay.
template <int FMT, bool ANY_VS, bool DEVS, bool L2>
__global__ void __launch_bounds__(kThreads, 4)
cast_step_amax_kernel(const CastDesc* __restrict__ cdescs,
                      const StepDesc* __restrict__ sdescs,
                      const Chunk* __restrict__ chunks, uint32_t nchunks,
                      const unsigned long long* __restrict__ gslots,
                      StepScratch sc, StepScalars s, uint32_t epoch) {
  __shared__ uint32_t red[kThreads / 32];
  // backwards: the amax pass read the last chunks most recently
  for (uint32_t r = blockIdx.x; r < nchunks; r += gridDim.x) {
    const Chunk ch = chunks[nchunks - 1 - r];
    const CastDesc cd = cdescs[ch.tensor];
    const StepDesc sd = sdescs[ch.tensor];
    const uint32_t ab = slot_value(gslots[ch.tensor], epoch);
    const float scale = scale_from_amax_bits(ab, fp8_max_of<FMT>());
    const float ms = *sd.m_scale;
    if (ch.begin == 0 && threadIdx.x == 0) {
      *cd.amax_out = __uint_as_float(ab);
      *cd.scale_out = scale;
      sc.old_m_scale[ch.tensor] = ms;
      if (sd.v_bound != nullptr) sc.old_v_bound[ch.tensor] = *sd.v_bound;
    }
    const float k = __fdiv_rn(step_ils<DEVS>(s), scale), minv = __frcp_rn(ms);
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    const bool checked = ab >= 0x7F800000u;
    uint32_t mx = 0, gx = 0, bad = 0;
    if (cd.dtype == kF32)
      cast_step_dispatch<kF32, FMT, ANY_VS, L2>(cd, sd, begin, end, scale, k, minv, checked, s, mx, gx, bad);
    else if (cd.dtype == kBF16)
      cast_step_dispatch<kBF16, FMT, ANY_VS, L2>(cd, sd, begin, end, scale, k, minv, checked, s, mx, gx, bad);
    else
      cast_step_dispatch<kF16, FMT, ANY_VS, L2>(cd, sd, begin, end, scale, k, minv, checked, s, mx, gx, bad);
    mx = block_max_u32(mx, red);
    if (ANY_VS && sd.v_bound != nullptr) {   // uniform over the CTA
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

}  // namespace

cudaError_t launch_cast_step(const CastDesc* cdescs, const StepDesc* sdescs,
                             const Chunk* chunks, uint32_t nchunks,
                             const Chunk* chunks_o3, uint32_t nchunks_o3,
                             unsigned long long* gslots, const StepScratch& sc,
                             const StepScalars& s, uint32_t epoch, int fmt,
                             uint32_t* found_dev, int grid_amax, int grid_fused,
                             int grid_update, int grid_update_var, int grid_w8,
                             bool any_vs,
                             cudaStream_t stream, LaunchMark mark) {
  if (nchunks == 0) {
    if (found_dev) return cudaMemsetAsync(found_dev, 0, sizeof(uint32_t), stream);
    return cudaSuccess;
  }
  cudaError_t e = launch_cast_amax(cdescs, chunks, nchunks, gslots, epoch,
                                   grid_amax, stream, mark);
  if (e != cudaSuccess) return e;
  const uint32_t g = grid_min((uint32_t)grid_fused, nchunks);
  if (mark) mark(kCastStepAmaxK, 0, stream);
  const int v = (s.l2 ? 8 : 0) | (fmt == kE4M3 ? 0 : 4) | (any_vs ? 2 : 0) |
                (s.dev ? 1 : 0);
  switch (v) {
#define FP8OPT_CAST_STEP_CASE(L2, FMT, VS, DEVS)                             \
  case (L2 ? 8 : 0) | (FMT == kE4M3 ? 0 : 4) | (VS ? 2 : 0) | (DEVS ? 1 : 0): \
    cast_step_amax_kernel<FMT, VS, DEVS, L2><<<g, kThreads, 0, stream>>>(    \
        cdescs, sdescs, chunks, nchunks, gslots, sc, s, epoch);              \
    break;
#define FP8OPT_CAST_STEP_CASES(L2)                                           \
    FP8OPT_CAST_STEP_CASE(L2, kE4M3, false, false)                           \
    FP8OPT_CAST_STEP_CASE(L2, kE4M3, false, true)                            \
    FP8OPT_CAST_STEP_CASE(L2, kE4M3, true, false)                            \
    FP8OPT_CAST_STEP_CASE(L2, kE4M3, true, true)                             \
    FP8OPT_CAST_STEP_CASE(L2, kE5M2, false, false)                           \
    FP8OPT_CAST_STEP_CASE(L2, kE5M2, false, true)                            \
    FP8OPT_CAST_STEP_CASE(L2, kE5M2, true, false)                            \
    FP8OPT_CAST_STEP_CASE(L2, kE5M2, true, true)
    FP8OPT_CAST_STEP_CASES(false)
    FP8OPT_CAST_STEP_CASES(true)
#undef FP8OPT_CAST_STEP_CASES
#undef FP8OPT_CAST_STEP_CASE
  }
  if (mark) mark(kCastStepAmaxK, 1, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_step_update(sdescs, chunks, nchunks, chunks_o3, nchunks_o3, sc,
                            s, epoch, found_dev, grid_update, grid_update_var,
                            grid_w8, any_vs,
                            stream, mark);
}

cudaError_t cast_step_occupancy(int* per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      per_sm, cast_step_amax_kernel<kE4M3, false, false, false>, kThreads, 0);
}

}  // namespace fp8opt
