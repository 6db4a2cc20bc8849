// Global L2 norm of the unscaled gradient of a step call, and the clip
// coefficient that follows from it (torch.nn.utils.clip_grad_norm_, the run
// script's --clip-grad).
//
// grad_norm_kernel: a persistent grid over the step's chunk table.  Every
// code's value is a multiple of 2^-16, so its square is an integer count of
// 2^-32 and the sum of squares of a tensor can be taken exactly:
//   E4M3: r = |value| * 2^9 is an integer below 2^18 (taken exactly from the
//         decoded float with one fused multiply-add against 2^23), r^2 below
//         2^36 in units of 2^-18, summed in 64 bits per thread;
//   E5M2: r = |value| * 2^16 below 2^32 from the code's fields, r^2 below
//         2^64 in units of 2^-32, summed in 128 bits per thread.
// Each CTA reduces its chunk to one 128-bit sum (units of 2^-32) and adds it
// to the tensor's slot with two 64-bit atomics (the low word's carry goes to
// the high word).  Integer sums are exact and order-free, so the result does
// not depend on the schedule.  The kernel also decides found_inf exactly as
// the step's first pass does: a non-finite code, or the largest |value| of
// the chunk times k not finite (the product is monotone in |value|), both
// read from the largest code magnitude of the chunk.
//
// grad_norm_terms_kernel: one thread per record, term_t = fl64(k_t^2 *
// fl64(S_t) * 2^-32) (k_t^2 is exact in double).
// clip_coef_kernel: one CTA.  total = the terms summed in record order in
// double; norm = sqrt(total); clip = max_norm / (norm + 1e-6) rounded to
// float when below 1, else 1.  With found_inf the norm is +inf.  Across ranks
// that own disjoint records, the terms can be gathered (a sum of vectors that
// are zero outside each rank's records reproduces every term exactly) and
// every rank takes the same norm.
#include "fp8opt_internal.cuh"

namespace fp8opt {

namespace {

constexpr int kNormGroups = 4;   // 8-code groups per thread per tile
constexpr int64_t kNormTile = (int64_t)kThreads * kGroup * kNormGroups;

struct U128 {
  unsigned long long lo, hi;
};

__device__ __forceinline__ U128 add128(U128 a, U128 b) {
  U128 r;
  r.lo = a.lo + b.lo;
  r.hi = a.hi + b.hi + (r.lo < a.lo ? 1ull : 0ull);
  return r;
}

__device__ __forceinline__ U128 add64(U128 a, unsigned long long b) {
  U128 r;
  r.lo = a.lo + b;
  r.hi = a.hi + (r.lo < a.lo ? 1ull : 0ull);
  return r;
}

// Sum over the CTA; the result is valid in thread 0.  Every thread calls it.
__device__ U128 block_sum128(U128 v, unsigned long long* smem) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    U128 w;
    w.lo = __shfl_xor_sync(0xFFFFFFFFu, v.lo, o);
    w.hi = __shfl_xor_sync(0xFFFFFFFFu, v.hi, o);
    v = add128(v, w);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) {
    smem[2 * warp] = v.lo;
    smem[2 * warp + 1] = v.hi;
  }
  __syncthreads();
  U128 s = {0ull, 0ull};
  if (threadIdx.x == 0)
    for (int i = 0; i < kThreads / 32; ++i) s = add128(s, U128{smem[2 * i], smem[2 * i + 1]});
  return s;
}

// acc += r * r in one 32 x 32 -> 64-bit multiply-add.
__device__ __forceinline__ void mad_sq(unsigned long long& acc, uint32_t r) {
  asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(acc) : "r"(r));
}

// acc += r^2 over the four codes of a word (sign bits already cleared).
// E4M3: the decoded values are exact floats below 2^9; v * 512 + 2^23 is an
// exact float whose low 23 bits are the integer r.
__device__ __forceinline__ void sq_e4m3(uint32_t w, unsigned long long& acc) {
  const float2 a = dec2<kE4M3>(w & 0xFFFFu), b = dec2<kE4M3>(w >> 16);
  const float2 ta = fma2(a, splat2(512.0f), splat2(8388608.0f));
  const float2 tb = fma2(b, splat2(512.0f), splat2(8388608.0f));
  mad_sq(acc, __float_as_uint(ta.x) & 0x7FFFFFu);
  mad_sq(acc, __float_as_uint(ta.y) & 0x7FFFFFu);
  mad_sq(acc, __float_as_uint(tb.x) & 0x7FFFFFu);
  mad_sq(acc, __float_as_uint(tb.y) & 0x7FFFFFu);
}

// E5M2: r = |value| * 2^16 from the code's exponent e and mantissa m:
// (4 + m) << (e - 1) for e >= 1, m for e = 0 (non-finite codes give 0; they
// set found_inf instead).
__device__ __forceinline__ U128 sq_e5m2(uint32_t w, U128 acc) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t mag = (w >> (8 * j)) & 0x7Fu;
    const uint32_t e = mag >> 2, m = mag & 3u;
    const uint32_t r = e == 0 ? m : (e == 31 ? 0u : ((4u | m) << (e - 1)));
    acc = add64(acc, (unsigned long long)r * r);
  }
  return acc;
}

// This thread's share of [begin, end): the exact sum of squares in units of
// 2^-32 and the largest code magnitude.  A non-finite code has the largest
// magnitudes of its format (E4M3 0x7F, E5M2 0x7C and above), so the maximum
// also tells whether one was seen; its square is not meaningful, but the
// norm is then +inf anyway.
template <int GF>
__device__ void thread_norm(const uint8_t* g, int64_t begin, int64_t end,
                            bool vec, U128& sum, uint32_t& cmax) {
  const int tid = threadIdx.x;
  unsigned long long s4 = 0;   // E4M3: units of 2^-18
  U128 s5 = {0ull, 0ull};      // E5M2: units of 2^-32
  uint32_t vmax = 0;           // per-byte max of the code magnitudes
#pragma unroll 1
  for (int64_t base = begin; base < end; base += kNormTile) {
    if (vec && base + kNormTile <= end) {
      uint2 c[kNormGroups];
#pragma unroll
      for (int q = 0; q < kNormGroups; ++q)
        c[q] = ld_once2(g + base + q * (kThreads * kGroup) + tid * kGroup);
#pragma unroll
      for (int q = 0; q < kNormGroups; ++q) {
        const uint32_t x = c[q].x & 0x7F7F7F7Fu, y = c[q].y & 0x7F7F7F7Fu;
        vmax = __vmaxu4(vmax, __vmaxu4(x, y));
        if (GF == kE4M3) {
          sq_e4m3(x, s4);
          sq_e4m3(y, s4);
        } else {
          s5 = sq_e5m2(y, sq_e5m2(x, s5));
        }
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < kNormGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        for (int e = 0; e < kGroup; ++e) {
          const int64_t i = i0 + e;
          if (i >= end) break;
          const uint32_t x = g[i] & 0x7Fu;
          vmax = __vmaxu4(vmax, x);
          if (GF == kE4M3)
            sq_e4m3(x, s4);
          else
            s5 = sq_e5m2(x, s5);
        }
      }
    }
  }
  if (GF == kE4M3) {
    sum.lo = s4 << 14;           // s4 < 2^43 here, so no bits are lost
    sum.hi = s4 >> 50;
  } else {
    sum = s5;
  }
  cmax = max(max(vmax & 0xFFu, (vmax >> 8) & 0xFFu),
             max((vmax >> 16) & 0xFFu, vmax >> 24));
}

__global__ void __launch_bounds__(kThreads, 4)
grad_norm_kernel(const StepDesc* __restrict__ descs,
                 const Chunk* __restrict__ chunks, uint32_t nchunks, float ils,
                 unsigned long long* __restrict__ sums,
                 unsigned long long* __restrict__ found, uint32_t epoch) {
  __shared__ unsigned long long red[2 * (kThreads / 32)];
  __shared__ uint32_t redm[kThreads / 32];
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const StepDesc d = descs[ch.tensor];
    const int64_t begin = (int64_t)ch.index * kChunkElems;
    const int64_t end = min(begin + kChunkElems, d.numel);
    const bool vec = d.vec_ok != 0;
    U128 s = {0ull, 0ull};
    uint32_t cmax = 0;
    if (d.g_fmt == kE4M3)
      thread_norm<kE4M3>(d.g, begin, end, vec, s, cmax);
    else
      thread_norm<kE5M2>(d.g, begin, end, vec, s, cmax);
    s = block_sum128(s, red);
    cmax = block_max_u32(cmax, redm);
    if (threadIdx.x == 0 && end > begin) {
      const bool any_bad = d.g_fmt == kE4M3 ? cmax == 0x7Fu : cmax >= 0x7Cu;
      if (s.lo | s.hi) {
        const unsigned long long old = atomicAdd(&sums[2 * ch.tensor], s.lo);
        const unsigned long long carry = old + s.lo < old ? 1ull : 0ull;
        if (s.hi + carry) atomicAdd(&sums[2 * ch.tensor + 1], s.hi + carry);
      }
      // the step's test: decode(code) * k not finite for some code
      const float k = __fdiv_rn(ils, *d.g_scale);
      const float vmax = d.g_fmt == kE4M3 ? dec2<kE4M3>(cmax).x : dec2<kE5M2>(cmax).x;
      if (any_bad || nonfinite(__fmul_rn(vmax, k)))
        atomicMax(found, slot_tag(epoch, 1u));
    }
  }
}

// Correctly rounded conversion of a 128-bit unsigned integer to double: the
// top 64 bits after normalisation, with every lower bit folded into the
// lowest one (a sticky bit, eleven places below the rounding position), then
// an exact power-of-two scaling.
__device__ double u128_to_double(U128 v) {
  if (v.hi == 0) return __ull2double_rn(v.lo);
  const int lz = __clzll((long long)v.hi);
  const unsigned long long top = lz ? (v.hi << lz) | (v.lo >> (64 - lz)) : v.hi;
  const unsigned long long rest = v.lo << lz;
  const double d = __ull2double_rn(top | (rest != 0 ? 1ull : 0ull));
  return __dmul_rn(d, __longlong_as_double((long long)(1023 + 64 - lz) << 52));
}

// Per-record terms fl64(k^2 * fl64(S) * 2^-32) (k^2 is exact in double), one
// thread per record; block 0 also exports this call's found_inf.
__global__ void __launch_bounds__(kThreads)
grad_norm_terms_kernel(const StepDesc* __restrict__ descs, int n, float ils,
                       const unsigned long long* __restrict__ sums,
                       const unsigned long long* __restrict__ found,
                       uint32_t epoch, double* __restrict__ terms,
                       uint32_t* __restrict__ found_out) {
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t < n) {
    const U128 s = {sums[2 * t], sums[2 * t + 1]};
    const double k = (double)__fdiv_rn(ils, *descs[t].g_scale);
    terms[t] = __dmul_rn(__dmul_rn(k, k), __dmul_rn(u128_to_double(s), 0x1p-32));
  }
  if (found_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *found_out = slot_value(*found, epoch) != 0 ? 1u : 0u;
}

// One CTA: total = sum of the terms in order, norm = sqrt(total) (+inf when
// found_inf is set in the slot or in found_flag), clip coefficient.
__global__ void __launch_bounds__(kThreads)
clip_coef_kernel(const double* __restrict__ terms, int n,
                 const unsigned long long* __restrict__ found_slot,
                 uint32_t epoch, const uint32_t* __restrict__ found_flag,
                 float max_norm, double* __restrict__ norm_out,
                 float* __restrict__ clip_out, float* __restrict__ user_norm) {
  __shared__ double term[kThreads];
  const bool inf = (found_slot != nullptr && slot_value(*found_slot, epoch) != 0) ||
                   (found_flag != nullptr && *found_flag != 0);
  double total = 0.0;
  for (int t0 = 0; t0 < n; t0 += kThreads) {
    const int t = t0 + threadIdx.x;
    if (t < n) term[threadIdx.x] = terms[t];
    __syncthreads();
    if (threadIdx.x == 0)
      for (int i = 0; i < kThreads && t0 + i < n; ++i) total = __dadd_rn(total, term[i]);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double norm = inf ? __longlong_as_double(0x7FF0000000000000ll)
                            : __dsqrt_rn(total);
    float clip = 1.0f;
    if (!inf && max_norm > 0.0f) {
      const double c = __ddiv_rn((double)max_norm, __dadd_rn(norm, 1e-6));
      if (c < 1.0) clip = __double2float_rn(c);
    }
    if (norm_out != nullptr) *norm_out = norm;
    if (clip_out != nullptr) *clip_out = clip;
    if (user_norm != nullptr) *user_norm = __double2float_rn(norm);
  }
}

// Writes a call's found_inf slot as 0 / 1 (out), after merging in an outside
// flag (in, may be NULL: e.g. found_inf reduced over ranks).
__global__ void found_kernel(unsigned long long* __restrict__ slot, uint32_t epoch,
                             const uint32_t* __restrict__ in,
                             uint32_t* __restrict__ out) {
  bool f = slot_value(*slot, epoch) != 0;
  if (in != nullptr && *in != 0 && !f) {
    *slot = slot_tag(epoch, 1u);
    f = true;
  }
  if (out != nullptr) *out = f ? 1u : 0u;
}

}  // namespace

// The norm pass and the per-record terms on `stream`.  sums: 2n zeroed words;
// found: the call's found_inf slot; terms: n doubles out; found_out: the
// call's found_inf as 0 / 1, or NULL.
cudaError_t launch_grad_norm_terms(const StepDesc* descs, const Chunk* chunks,
                                   uint32_t nchunks, int n, float ils,
                                   unsigned long long* sums,
                                   unsigned long long* found, uint32_t epoch,
                                   double* terms, uint32_t* found_out, int grid,
                                   cudaStream_t stream, LaunchMark mark) {
  if (nchunks != 0) {
    if (mark) mark(kGradNormK, 0, stream);
    grad_norm_kernel<<<grid_min((uint32_t)grid, nchunks), kThreads, 0, stream>>>(
        descs, chunks, nchunks, ils, sums, found, epoch);
    if (mark) mark(kGradNormK, 1, stream);
  }
  if (n > 0) {
    if (mark) mark(kGradNormTermsK, 0, stream);
    grad_norm_terms_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
        descs, n, ils, sums, found, epoch, terms, found_out);
    if (mark) mark(kGradNormTermsK, 1, stream);
  }
  return cudaGetLastError();
}

// The norm and clip coefficient from n terms (see clip_coef_kernel).
cudaError_t launch_clip_coef(const double* terms, int n,
                             const unsigned long long* found_slot, uint32_t epoch,
                             const uint32_t* found_flag, float max_norm,
                             double* norm_out, float* clip_out, float* user_norm,
                             cudaStream_t stream, LaunchMark mark) {
  if (mark) mark(kClipCoefK, 0, stream);
  clip_coef_kernel<<<1, kThreads, 0, stream>>>(terms, n, found_slot, epoch,
                                               found_flag, max_norm, norm_out,
                                               clip_out, user_norm);
  if (mark) mark(kClipCoefK, 1, stream);
  return cudaGetLastError();
}

// found_kernel on `stream`.
cudaError_t launch_found(unsigned long long* slot, uint32_t epoch,
                         const uint32_t* in, uint32_t* out, cudaStream_t stream,
                         LaunchMark mark) {
  if (mark) mark(kFoundK, 0, stream);
  found_kernel<<<1, 1, 0, stream>>>(slot, epoch, in, out);
  if (mark) mark(kFoundK, 1, stream);
  return cudaGetLastError();
}

cudaError_t grad_norm_occupancy(int* per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, grad_norm_kernel,
                                                       kThreads, 0);
}

}  // namespace fp8opt
