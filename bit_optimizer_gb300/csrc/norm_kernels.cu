// Global L2 norm of the unscaled gradient of a step call, and the clip
// coefficient that follows from it (torch.nn.utils.clip_grad_norm_, the run
// script's --clip-grad).
//
// grad_norm_kernel: a persistent grid over the step's chunk table, each CTA
// walking one contiguous range of it; the exact sum of squared code values
// of each run of one tensor's chunks (read from a shared-memory table of the
// integer square roots: SqTable and SqTab, or for an all-E5M2 list Sq5Table
// and SqSum, fp8opt_internal.cuh) goes to the tensor's 128-bit slot, and
// found_inf is decided exactly as the step's first pass does (the tensor's
// overflow threshold).
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

// Resident CTAs per SM of the norm pass (each CTA holds the 32 KB table of
// the exact squares).
#ifndef FP8OPT_NORM_MIN_BLOCKS
#define FP8OPT_NORM_MIN_BLOCKS 4
#endif
// A chunk is read as two half tiles of eight 8-code groups per thread.  The
// pass is bound by memory latency, so each half's loads go out one half tile
// ahead of its arithmetic: a chunk's second half is requested before its
// first is summed, and the next chunk's first half before the second is
// summed, so a thread always has a half tile in flight.
constexpr int kHalfGroups = 8;
constexpr int64_t kHalfTile = (int64_t)kThreads * kGroup * kHalfGroups;
static_assert(2 * kHalfTile == kChunkElems, "a full chunk is two half tiles");

struct HalfTile {
  uint2 c[kHalfGroups];
};

// Issues the loads of the half tile at p (8-byte aligned, kHalfTile codes).
__device__ __forceinline__ void load_half(HalfTile& h, const uint8_t* p) {
#pragma unroll
  for (int q = 0; q < kHalfGroups; ++q)
    h.c[q] = ld_once2(p + q * (kThreads * kGroup) + threadIdx.x * kGroup);
}

// A thread's exact sums in the norm pass.  kNormAny: a list of either code
// format, per tensor, through SqTable (E5M2 squares in 128 bits).
// kNormE5M2: every tensor has E5M2 codes, through SqSum<kE5M2> (two 64-bit
// sums, a 64-bit table entry per code).
constexpr int kNormAny = 0;
constexpr int kNormE5M2 = 1;

template <int MODE>
struct NormAcc;

template <>
struct NormAcc<kNormAny> {
  using Table = SqTable;
  const SqTable* tab;
  SqTab s;
  __device__ __forceinline__ explicit NormAcc(const SqTable* t) : tab(t) {}
  template <int GF>
  __device__ __forceinline__ void add(uint32_t wm) {
    s.add_word<GF>(wm, sq_lane_byte<GF>(), *tab);
  }
  __device__ __forceinline__ U128 sum() const { return s.sum(); }
  __device__ __forceinline__ void clear() { s = SqTab(); }
};

template <>
struct NormAcc<kNormE5M2> {
  using Table = Sq5Table;
  SqSum<kE5M2> s;
  __device__ __forceinline__ explicit NormAcc(const Sq5Table* t) : s(t) {}
  template <int GF>
  __device__ __forceinline__ void add(uint32_t wm) { s.add_word(wm); }
  __device__ __forceinline__ U128 sum() const { return s.sum(); }
  __device__ __forceinline__ void clear() { s.clear(); }
};

// Adds a loaded half tile to acc; bad collects the codes at or above the
// tensor's overflow threshold (addend tadd).
template <int GF, class Acc>
__device__ __forceinline__ void sum_half(const HalfTile& h, uint32_t tadd,
                                         Acc& acc, uint32_t& bad) {
#pragma unroll
  for (int q = 0; q < kHalfGroups; ++q) {
    const uint32_t a = h.c[q].x & 0x7F7F7F7Fu, b = h.c[q].y & 0x7F7F7F7Fu;
    bad |= ((a + tadd) | (b + tadd)) & 0x80808080u;
    acc.template add<GF>(a);
    acc.template add<GF>(b);
  }
}

template <int MODE>
__device__ __forceinline__ void sum_half_fmt(const HalfTile& h, int fmt,
                                             uint32_t tadd, NormAcc<MODE>& acc,
                                             uint32_t& bad) {
  if (MODE == kNormAny && fmt == kE4M3)
    sum_half<kE4M3>(h, tadd, acc, bad);
  else
    sum_half<kE5M2>(h, tadd, acc, bad);
}

// This thread's share of a chunk that is not full ([begin, end) shorter than
// kChunkElems, or codes without vector loads): whole 8-code groups as
// vectors where they can be, the rest by code.
template <int GF, class Acc>
__device__ void thread_norm_part(const uint8_t* g, int64_t begin, int64_t end,
                                 bool vec, uint32_t tadd, Acc& acc,
                                 uint32_t& bad) {
#pragma unroll 1
  for (int64_t i0 = begin + threadIdx.x * kGroup; i0 < end;
       i0 += kThreads * kGroup) {
    if (vec && i0 + kGroup <= end) {
      const uint2 c = ld_once2(g + i0);
      const uint32_t a = c.x & 0x7F7F7F7Fu, b = c.y & 0x7F7F7F7Fu;
      bad |= ((a + tadd) | (b + tadd)) & 0x80808080u;
      acc.template add<GF>(a);
      acc.template add<GF>(b);
      continue;
    }
    for (int e = 0; e < kGroup && i0 + e < end; ++e) {
      const uint32_t a = g[i0 + e] & 0x7Fu;
      bad |= (a + tadd) & 0x80u;
      acc.template add<GF>(a);    // bytes 1..3 are zero: magnitude 0
    }
  }
}

// What the pass needs of a chunk and its tensor.
struct NormChunk {
  const uint8_t* g;
  const float* g_scale;
  int64_t begin;
  uint32_t len, tensor;
  int fmt;
  bool vec;

  __device__ __forceinline__ bool full() const {
    return vec && len == (uint32_t)kChunkElems;
  }
};

__device__ __forceinline__ NormChunk norm_chunk(const StepDesc* descs,
                                                const Chunk* chunks, uint32_t c) {
  const Chunk ch = chunks[c];
  const StepDesc& d = descs[ch.tensor];
  NormChunk r;
  r.g = d.g;
  r.g_scale = d.g_scale;
  r.begin = ch.begin;
  r.len = ch.len;
  r.tensor = ch.tensor;
  r.fmt = d.g_fmt;
  r.vec = d.vec_ok != 0;
  return r;
}

// Each CTA takes one contiguous range of the chunk table (an equal share),
// so a large tensor's chunks reach it as one run; a run adds to one
// accumulator, which goes to the tensor's slot when the tensor changes: one
// CTA reduction per run instead of one per chunk.  The next chunk's record
// is read while the current one is summed.  MODE: kNormAny, or kNormE5M2
// when every tensor of the call has E5M2 codes.
template <int MODE>
__global__ void __launch_bounds__(kThreads, FP8OPT_NORM_MIN_BLOCKS)
grad_norm_kernel(const StepDesc* __restrict__ descs,
                 const Chunk* __restrict__ chunks, uint32_t nchunks, float ils_h,
                 const float* __restrict__ ils_dev,
                 unsigned long long* __restrict__ sums,
                 unsigned long long* __restrict__ found, uint32_t epoch) {
  const float ils = ils_dev != nullptr ? *ils_dev : ils_h;
  __shared__ typename NormAcc<MODE>::Table tab;
  __shared__ SqRed red;
  const uint32_t c0 = (uint32_t)((uint64_t)blockIdx.x * nchunks / gridDim.x);
  const uint32_t c1 = (uint32_t)((uint64_t)(blockIdx.x + 1) * nchunks / gridDim.x);
  if (c0 >= c1) return;   // uniform over the CTA
  NormChunk cur = norm_chunk(descs, chunks, c0);
  HalfTile a, b;          // a holds the current chunk's first half if full
  if (cur.full()) load_half(a, cur.g + cur.begin);
  if constexpr (MODE == kNormAny)
    sq_table_fill(tab);
  else
    sq5_table_fill(tab);
  NormAcc<MODE> acc(&tab);
  uint32_t bad = 0, tadd = 0, tensor = 0xFFFFFFFFu, turn = 0;
  bool nonempty = false;
  for (uint32_t c = c0; c < c1; ++c) {
    const bool more = c + 1 < c1;
    NormChunk nxt = cur;
    if (more) nxt = norm_chunk(descs, chunks, c + 1);
    if (cur.tensor != tensor) {   // uniform over the CTA
      if (tensor != 0xFFFFFFFFu) {
        sq_commit(acc.sum(), bad, tensor, nonempty, sums, found, epoch, red, turn);
        acc.clear();
        bad = 0;
        nonempty = false;
      }
      tensor = cur.tensor;
      // found_inf exactly as the step's first pass decides it: some code at
      // or above the overflow threshold of k = inv_loss_scale / g_scale
      const float k = __fdiv_rn(ils, *cur.g_scale);
      tadd = threshold_addend(MODE == kNormAny && cur.fmt == kE4M3
                                  ? overflow_threshold<kE4M3>(k)
                                  : overflow_threshold<kE5M2>(k));
    }
    nonempty |= cur.len > 0;
    const bool next_full = more && nxt.full();
    if (cur.full()) {
      load_half(b, cur.g + cur.begin + kHalfTile);
      sum_half_fmt<MODE>(a, cur.fmt, tadd, acc, bad);
      if (next_full) load_half(a, nxt.g + nxt.begin);
      sum_half_fmt<MODE>(b, cur.fmt, tadd, acc, bad);
    } else {
      if (next_full) load_half(a, nxt.g + nxt.begin);
      const int64_t end = cur.begin + cur.len;
      if (MODE == kNormAny && cur.fmt == kE4M3)
        thread_norm_part<kE4M3>(cur.g, cur.begin, end, cur.vec, tadd, acc, bad);
      else
        thread_norm_part<kE5M2>(cur.g, cur.begin, end, cur.vec, tadd, acc, bad);
    }
    cur = nxt;
  }
  sq_commit(acc.sum(), bad, tensor, nonempty, sums, found, epoch, red, turn);
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

// total = the terms summed in record order in double (one thread; the
// additions are a dependent chain, so the terms are read eight at a time
// ahead of it), norm = sqrt(total) (+inf when found_inf is set in the slot
// or in found_flag), clip coefficient.  Thread 0 only.
__device__ __forceinline__ void finish_norm(const double* terms, int n, bool inf,
                                            float max_norm, double* norm_out,
                                            float* clip_out, float* user_norm) {
  double total = 0.0;
  int i = 0;
  for (; i + 8 <= n; i += 8) {
    double x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = terms[i + j];
#pragma unroll
    for (int j = 0; j < 8; ++j) total = __dadd_rn(total, x[j]);
  }
  for (; i < n; ++i) total = __dadd_rn(total, terms[i]);
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

// One CTA: the norm and clip coefficient from n given terms (finish_norm).
__global__ void __launch_bounds__(kThreads)
clip_coef_kernel(const double* __restrict__ terms, int n,
                 const unsigned long long* __restrict__ found_slot,
                 uint32_t epoch, const uint32_t* __restrict__ found_flag,
                 float max_norm, double* __restrict__ norm_out,
                 float* __restrict__ clip_out, float* __restrict__ user_norm) {
  if (threadIdx.x != 0) return;
  const bool inf = (found_slot != nullptr && slot_value(*found_slot, epoch) != 0) ||
                   (found_flag != nullptr && *found_flag != 0);
  finish_norm(terms, n, inf, max_norm, norm_out, clip_out, user_norm);
}

// One CTA: the records' terms as grad_norm_terms_kernel writes them (every
// thread a share of the records), then, after the CTA barrier that makes
// them visible, the norm and clip coefficient from them (finish_norm).
// terms is written and read here, so it is neither const nor restrict.
__global__ void __launch_bounds__(kThreads)
norm_finish_kernel(const StepDesc* __restrict__ descs, int n, float ils,
                   const float* __restrict__ ils_dev,
                   const unsigned long long* __restrict__ sums,
                   const unsigned long long* __restrict__ found_slot,
                   uint32_t epoch, double* terms, float max_norm,
                   double* __restrict__ norm_out, float* __restrict__ clip_out,
                   float* __restrict__ user_norm) {
  const float k_ils = ils_dev != nullptr ? *ils_dev : ils;
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    const U128 s = {sums[2 * t], sums[2 * t + 1]};
    terms[t] = norm_term(s, __fdiv_rn(k_ils, *descs[t].g_scale));
  }
  __syncthreads();
  if (threadIdx.x == 0)
    finish_norm(terms, n, slot_value(*found_slot, epoch) != 0, max_norm, norm_out,
                clip_out, user_norm);
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

// ---------------------------------------------- exchanges between ranks
//
// A tensor cut into pieces on several ranks has per-tensor quantities that
// are maxima (an amax, max |g|) or exact sums over its pieces.  The calls
// split at those quantities export each piece's value and import the
// combined one: maxima as the fp32 bits of a non-negative value (their
// unsigned order is the amax order: NaN 0x7FC00000 above +inf above every
// finite value, so a MAX over ranks combines them), exact sums as four
// 32-bit limbs held in int64 (a SUM over fewer than 2^31 ranks stays exact).

// out[i] = this call's value in slot i (0 if the slot holds none).
__global__ void slots_export_kernel(const unsigned long long* __restrict__ slots,
                                    uint32_t epoch, int n,
                                    uint32_t* __restrict__ out) {
  const int i = blockIdx.x * kThreads + threadIdx.x;
  if (i < n) out[i] = slot_value(slots[i], epoch);
}

// Slot i takes the given value as this call's.
__global__ void slots_import_kernel(unsigned long long* __restrict__ slots,
                                    uint32_t epoch, int n,
                                    const uint32_t* __restrict__ in) {
  const int i = blockIdx.x * kThreads + threadIdx.x;
  if (i < n) slots[i] = slot_tag(epoch, in[i]);
}

// The exact 128-bit sums (sums[2i], sums[2i + 1]) as limbs[4i .. 4i + 3],
// low limb first; block 0 also exports the call's found_inf.
__global__ void sums_to_limbs_kernel(const unsigned long long* __restrict__ sums,
                                     int n,
                                     const unsigned long long* __restrict__ found,
                                     uint32_t epoch, long long* __restrict__ limbs,
                                     uint32_t* __restrict__ found_out) {
  const int i = blockIdx.x * kThreads + threadIdx.x;
  if (i < n) {
    const unsigned long long lo = sums[2 * i], hi = sums[2 * i + 1];
    limbs[4 * i] = (long long)(lo & 0xFFFFFFFFull);
    limbs[4 * i + 1] = (long long)(lo >> 32);
    limbs[4 * i + 2] = (long long)(hi & 0xFFFFFFFFull);
    limbs[4 * i + 3] = (long long)(hi >> 32);
  }
  if (found_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *found_out = slot_value(*found, epoch) != 0 ? 1u : 0u;
}

// terms[t] = the norm term of tensor t from its limbs summed over ranks (each
// below 2^63; the top limb below 2^32) and the factor k = inv_loss_scale /
// scale, scale = fp8_max / amax with the cast's guards (amax_bits[t]).
__global__ void limbs_terms_kernel(const long long* __restrict__ limbs,
                                   const uint32_t* __restrict__ amax_bits, int n,
                                   float fp8_max, float ils,
                                   double* __restrict__ terms) {
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t >= n) return;
  const unsigned long long l0 = (unsigned long long)limbs[4 * t];
  const unsigned long long l1 = (unsigned long long)limbs[4 * t + 1];
  const unsigned long long l2 = (unsigned long long)limbs[4 * t + 2];
  const unsigned long long l3 = (unsigned long long)limbs[4 * t + 3];
  U128 s = {l0, 0ull};
  s = add128(s, U128{l1 << 32, l1 >> 32});
  s = add128(s, U128{0ull, l2});
  s = add128(s, U128{0ull, l3 << 32});
  const float scale = scale_from_amax_bits(amax_bits[t], fp8_max);
  terms[t] = norm_term(s, __fdiv_rn(ils, scale));
}

}  // namespace

// Slot values of this call out to a device array, and back in.
cudaError_t launch_slots_export(const unsigned long long* slots, uint32_t epoch,
                                int n, uint32_t* out, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  slots_export_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
      slots, epoch, n, out);
  return cudaGetLastError();
}

cudaError_t launch_slots_import(unsigned long long* slots, uint32_t epoch, int n,
                                const uint32_t* in, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  slots_import_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
      slots, epoch, n, in);
  return cudaGetLastError();
}

// The exact sums of n records as limbs, and the call's found_inf (found_out,
// may be NULL).
cudaError_t launch_sums_to_limbs(const unsigned long long* sums, int n,
                                 const unsigned long long* found, uint32_t epoch,
                                 long long* limbs, uint32_t* found_out,
                                 cudaStream_t stream) {
  const int blocks = n > 0 ? (n + kThreads - 1) / kThreads : 1;
  sums_to_limbs_kernel<<<blocks, kThreads, 0, stream>>>(sums, n, found, epoch,
                                                        limbs, found_out);
  return cudaGetLastError();
}

cudaError_t launch_limbs_terms(const long long* limbs, const uint32_t* amax_bits,
                               int n, int fmt, float ils, double* terms,
                               cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  limbs_terms_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
      limbs, amax_bits, n, fmt == kE4M3 ? 448.0f : 57344.0f, ils, terms);
  return cudaGetLastError();
}

// The norm pass and the per-record terms on `stream`.  sums: 2n zeroed words;
// found: the call's found_inf slot; terms: n doubles out; found_out: the
// call's found_inf as 0 / 1, or NULL.  ils_dev: inv_loss_scale in device
// memory instead of ils, or NULL.  fmts: bit f set when some record has
// codes of format f.
cudaError_t launch_grad_norm_terms(const StepDesc* descs, const Chunk* chunks,
                                   uint32_t nchunks, int n, float ils,
                                   const float* ils_dev,
                                   unsigned long long* sums,
                                   unsigned long long* found, uint32_t epoch,
                                   double* terms, uint32_t* found_out, int grid,
                                   int fmts, cudaStream_t stream, LaunchMark mark) {
  if (nchunks != 0) {
    if (mark) mark(kGradNormK, 0, stream);
    const uint32_t g = grid_min((uint32_t)grid, nchunks);
    if (fmts == (1 << kE5M2))
      grad_norm_kernel<kNormE5M2><<<g, kThreads, 0, stream>>>(
          descs, chunks, nchunks, ils, ils_dev, sums, found, epoch);
    else
      grad_norm_kernel<kNormAny><<<g, kThreads, 0, stream>>>(
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

// The records' terms, the norm and the clip coefficient in one launch (see
// norm_finish_kernel): after the norm pass, in place of the terms kernel and
// launch_clip_coef.
cudaError_t launch_norm_finish(const StepDesc* descs, int n, float ils,
                               const float* ils_dev,
                               const unsigned long long* sums,
                               const unsigned long long* found_slot,
                               uint32_t epoch, double* terms, float max_norm,
                               double* norm_out, float* clip_out,
                               float* user_norm, cudaStream_t stream,
                               LaunchMark mark) {
  if (mark) mark(kClipCoefK, 0, stream);
  norm_finish_kernel<<<1, kThreads, 0, stream>>>(descs, n, ils, ils_dev, sums,
                                                 found_slot, epoch, terms, max_norm,
                                                 norm_out, clip_out, user_norm);
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
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      per_sm, grad_norm_kernel<kNormAny>, kThreads, 0);
}

}  // namespace fp8opt
