// Global L2 norm of the unscaled gradient of a step call, and the clip
// coefficient that follows from it (torch.nn.utils.clip_grad_norm_, the run
// script's --clip-grad).
//
// grad_norm_kernel: a persistent grid over the step's chunk table; each
// chunk's exact sum of squared code values (SqAcc, fp8opt_internal.cuh) goes
// to its tensor's 128-bit slot, and found_inf is decided exactly as the
// step's first pass does (sq_commit).
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

// 8-code groups per thread per tile, and resident CTAs per SM of the norm
// pass.  Measured on the 350M list: 0.152 to 0.156 ms with eight groups at 5
// CTAs/SM, 0.165 with four, 0.156 with sixteen (which spill at 5 CTAs/SM).
#ifndef FP8OPT_NORM_GROUPS
#define FP8OPT_NORM_GROUPS 8
#endif
#ifndef FP8OPT_NORM_MIN_BLOCKS
#define FP8OPT_NORM_MIN_BLOCKS 5
#endif
constexpr int kNormGroups = FP8OPT_NORM_GROUPS;
constexpr int64_t kNormTile = (int64_t)kThreads * kGroup * kNormGroups;

// This thread's share of [begin, end) into acc.
template <int GF>
__device__ void thread_norm(const uint8_t* g, int64_t begin, int64_t end,
                            bool vec, SqAcc<GF>& acc) {
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int64_t base = begin; base < end; base += kNormTile) {
    if (vec && base + kNormTile <= end) {
      uint2 c[kNormGroups];
#pragma unroll
      for (int q = 0; q < kNormGroups; ++q)
        c[q] = ld_once2(g + base + q * (kThreads * kGroup) + tid * kGroup);
#pragma unroll
      for (int q = 0; q < kNormGroups; ++q) {
        acc.add_word(c[q].x);
        acc.add_word(c[q].y);
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < kNormGroups; ++q) {
        const int64_t i0 = base + q * (kThreads * kGroup) + tid * kGroup;
        for (int e = 0; e < kGroup; ++e) {
          const int64_t i = i0 + e;
          if (i >= end) break;
          acc.add_word(g[i]);
        }
      }
    }
  }
}

template <int GF>
__device__ __forceinline__ void norm_chunk(const StepDesc& d, const Chunk& ch,
                                           int64_t begin, int64_t end, float ils,
                                           unsigned long long* sums,
                                           unsigned long long* found,
                                           uint32_t epoch,
                                           unsigned long long* red64,
                                           uint32_t* red32) {
  SqAcc<GF> acc;
  thread_norm<GF>(d.g, begin, end, d.vec_ok != 0, acc);
  const float k = __fdiv_rn(ils, *d.g_scale);
  sq_commit<GF>(acc, ch.tensor, end > begin, k, sums, found, epoch, red64, red32);
}

__global__ void __launch_bounds__(kThreads, FP8OPT_NORM_MIN_BLOCKS)
grad_norm_kernel(const StepDesc* __restrict__ descs,
                 const Chunk* __restrict__ chunks, uint32_t nchunks, float ils_h,
                 const float* __restrict__ ils_dev,
                 unsigned long long* __restrict__ sums,
                 unsigned long long* __restrict__ found, uint32_t epoch) {
  const float ils = ils_dev != nullptr ? *ils_dev : ils_h;
  __shared__ unsigned long long red64[2 * (kThreads / 32)];
  __shared__ uint32_t red32[kThreads / 32];
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const StepDesc d = descs[ch.tensor];
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    if (d.g_fmt == kE4M3)
      norm_chunk<kE4M3>(d, ch, begin, end, ils, sums, found, epoch, red64, red32);
    else
      norm_chunk<kE5M2>(d, ch, begin, end, ils, sums, found, epoch, red64, red32);
  }
}

// Per-record terms fl64(k^2 * fl64(S) * 2^-32) (k^2 is exact in double), one
// thread per record; block 0 also exports this call's found_inf.
__global__ void __launch_bounds__(kThreads)
grad_norm_terms_kernel(const StepDesc* __restrict__ descs, int n, float ils,
                       const float* __restrict__ ils_dev,
                       const unsigned long long* __restrict__ sums,
                       const unsigned long long* __restrict__ found,
                       uint32_t epoch, double* __restrict__ terms,
                       uint32_t* __restrict__ found_out) {
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t < n) {
    const U128 s = {sums[2 * t], sums[2 * t + 1]};
    const float k = __fdiv_rn(ils_dev != nullptr ? *ils_dev : ils,
                              *descs[t].g_scale);
    terms[t] = norm_term(s, k);
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
// call's found_inf as 0 / 1, or NULL.  ils_dev: inv_loss_scale in device
// memory instead of ils, or NULL.
cudaError_t launch_grad_norm_terms(const StepDesc* descs, const Chunk* chunks,
                                   uint32_t nchunks, int n, float ils,
                                   const float* ils_dev,
                                   unsigned long long* sums,
                                   unsigned long long* found, uint32_t epoch,
                                   double* terms, uint32_t* found_out, int grid,
                                   cudaStream_t stream, LaunchMark mark) {
  if (nchunks != 0) {
    if (mark) mark(kGradNormK, 0, stream);
    grad_norm_kernel<<<grid_min((uint32_t)grid, nchunks), kThreads, 0, stream>>>(
        descs, chunks, nchunks, ils, ils_dev, sums, found, epoch);
    if (mark) mark(kGradNormK, 1, stream);
  }
  if (n > 0) {
    if (mark) mark(kGradNormTermsK, 0, stream);
    grad_norm_terms_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
        descs, n, ils, ils_dev, sums, found, epoch, terms, found_out);
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
