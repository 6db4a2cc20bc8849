// Internal definitions shared by the libfp8opt kernels and the host layer.
//
// Work decomposition (multi-tensor chunk table): every tensor of a call is cut
// into chunks of 2^shift elements (the last chunk of a tensor may be shorter;
// an empty tensor gets one empty chunk so that its per-tensor outputs are
// still written).  The shift is kChunkShift (32768 elements); the host picks
// a smaller one for the cast's tables of short lists and for every table of
// a tiny list, and each chunk carries its first element and length.  The host
// builds the chunk table once per tensor list and caches it on the device.
// Each kernel is a persistent grid (a multiple of the SM count) whose CTAs
// stride over the chunk table; a CTA handles one chunk at a time in tiles:
// thread t of an N-thread CTA takes the groups of G elements starting at
// tile + k * (N * G) + t * G, so every load and store instruction of a warp
// touches one contiguous span.  Each pass sets its own N, G and groups per
// tile.
//
// Per-tensor reductions (amax) and the found_inf flag live in 64-bit slots
// tagged with a per-call epoch in the high word: a slot is current only when
// its tag equals this call's epoch, and atomicMax on (epoch << 32 | bits)
// both starts a new call's maximum and ignores stale values, so the slots need
// no clearing between calls.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8opt {

constexpr int kThreads = 256;                    // threads per CTA
constexpr int kGroup = 8;                        // elements per vector group
constexpr int kChunkShift = 15;                  // 32768 elements per chunk
constexpr int64_t kChunkElems = (int64_t)1 << kChunkShift;

constexpr int kE4M3 = 0;
constexpr int kE5M2 = 1;
constexpr int kF32 = 0;
constexpr int kBF16 = 1;
constexpr int kF16 = 2;

struct Chunk {
  uint32_t tensor;  // index into the tensor table
  uint32_t len;     // elements in the chunk (0 for an empty tensor's chunk)
  int64_t begin;    // first element; 0 marks a tensor's first chunk
};

// Most tensors one call takes.
constexpr uint32_t kMaxListTensors = 1u << 30;

// Chunk `index` of 2^shift elements of a tensor with numel elements.
inline Chunk make_chunk(uint32_t tensor, uint32_t index, int shift,
                        int64_t numel) {
  Chunk c;
  c.tensor = tensor;
  c.begin = (int64_t)index << shift;
  const int64_t rest = numel - c.begin;
  const int64_t size = (int64_t)1 << shift;
  c.len = (uint32_t)(rest < size ? (rest > 0 ? rest : 0) : size);
  return c;
}

struct CastDesc {
  const void* src;
  uint8_t* codes;
  float* amax_out;
  float* scale_out;
  int64_t numel;
  int32_t dtype;
  int32_t vec_ok;   // all buffers aligned for the vector path
};

struct StepDesc {
  const uint8_t* g;
  uint8_t* m;
  uint16_t* v;
  uint16_t* w;
  uint8_t* w8;
  const float* g_scale;
  float* m_scale;
  float* w8_scale;
  float* w8_amax;
  float* v_bound;   // scaled second moment: its bound (in/out), else NULL
  int64_t numel;
  int32_t g_fmt;
  int16_t vec_ok;
  int16_t o3;       // emits the E4M3 weight copy (w8 is NULL if numel is 0)
};

// One tensor of a local FP8 reduction: k shards of numel codes, shard j at
// src + j * stride, encoded with scale src_scale[j].
struct ReduceDesc {
  const uint8_t* src;
  const float* src_scale;
  uint8_t* codes;
  float* amax_out;
  float* scale_out;
  int64_t numel;
  int64_t stride;
  int32_t vec_ok;   // src, stride and codes aligned for 16-byte accesses
  int32_t pad;
};

// Most shards one reduction call takes.
constexpr int kMaxShards = 64;

// The gradient norm of a reduction's outputs: 2n zeroed words of exact sums,
// the call's found_inf slot, the inverse loss scale, n terms out (or, when
// limbs is set, the exact sums as 4n limbs instead) and the found flag out
// (may be NULL).
struct ReduceNorm {
  unsigned long long* sums;
  unsigned long long* found;
  float ils;
  int n;
  double* terms;
  uint32_t* found_out;
  long long* limbs;
};

// Passes of a reduction call: the amax pass, the encode pass, or both.
enum ReducePhase { kReduceAmaxPass = 1, kReduceEncodePass = 2,
                   kReduceBothPasses = 3 };

// Kernels, for the optional per-launch event timing.
enum KernelId { kCastAmaxK = 0, kCastEncodeK, kStepAmaxK, kStepUpdateK,
                kStepW8K, kCastStepAmaxK, kReduceAmaxK, kReduceEncodeK,
                kGradNormK, kGradNormTermsK, kClipCoefK, kFoundK,
                kNumKernels };

// Called before (end = 0) and after (end = 1) each kernel launch when timing
// is on; nullptr otherwise.
typedef void (*LaunchMark)(int kernel, int end, cudaStream_t stream);

struct DevScalars;

// Per-call scalars of the AdamW step (computed on the host): the bias
// corrections enter only through step_size = lr / (1 - beta1^t) and
// inv_sbc2 = 1 / sqrt(1 - beta2^t), each evaluated in double and rounded once.
struct StepScalars {
  float beta1, beta2, eps, omb1, omb2, step_size, inv_sbc2, decay, ils;
  float wd;       // the L2 coefficient (used when l2)
  int32_t l2;     // Adam with L2 decay: g = fma(wd, w, g); decay is then 1
  const float* clip;  // device clip coefficient (k becomes k * clip), or NULL
  // Device-resident step (the *_dev calls): step_size, inv_sbc2, decay and
  // ils come from *dev instead, and the update kernel stores dev->t into
  // *step_out when the step is taken.  NULL otherwise.
  const DevScalars* dev;
  long long* step_out;
};

// The caller's device-resident step values (fp8opt_step_state, same layout).
struct DevState {
  float lr;
  float inv_loss_scale;
  long long step;   // steps taken so far
};

// The per-step scalars of a *_dev call, made on the device from a DevState
// by step_scalars_kernel with the same arithmetic as the host's, and the
// step t they belong to.
struct DevScalars {
  float step_size, inv_sbc2, decay, ils;
  long long t;
};

// inv_loss_scale of the call: from the host, or (DEVS) from the device.
template <bool DEVS>
__device__ __forceinline__ float step_ils(const StepScalars& s) {
  if constexpr (DEVS) return __ldg(&s.dev->ils);
  else return s.ils;
}

// A scaled second moment is stored as FP16 of v * kVTarget / bound.
constexpr float kVTarget = 16384.0f;

// Scratch of one step call: per-tensor slots and the old first-moment scales.
struct StepScratch {
  unsigned long long* amax_m;   // [n] amax of this step's fp32 first moment
  unsigned long long* amax_w;   // [n] amax of the FP16 master (O3)
  unsigned long long* amax_g;   // [n] max |g| (scaled second moment)
  unsigned long long* found;    // [1] found_inf
  float* old_m_scale;           // [n] m_scale before this step
  float* old_v_bound;           // [n] v_bound before this step
};

// ------------------------------------------------------------------ helpers

inline uint32_t grid_min(uint32_t a, uint32_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint32_t canon_amax_bits(uint32_t b) {
  return b > 0x7F800000u ? 0x7FC00000u : b;   // any NaN -> one quiet NaN
}

__device__ __forceinline__ uint32_t slot_value(unsigned long long s,
                                               uint32_t epoch) {
  return (uint32_t)(s >> 32) == epoch ? (uint32_t)s : 0u;
}

__device__ __forceinline__ unsigned long long slot_tag(uint32_t epoch,
                                                       uint32_t bits) {
  return ((unsigned long long)epoch << 32) | bits;
}

// fp8_max / amax with the guards: 1.0 when amax is zero or not finite, or
// when the IEEE quotient is not finite.
__device__ __forceinline__ float scale_from_amax_bits(uint32_t bits,
                                                      float fp8_max) {
  float amax = __uint_as_float(bits);
  if (!(amax > 0.0f) || bits >= 0x7F800000u) return 1.0f;
  float q = __fdiv_rn(fp8_max, amax);
  return (__float_as_uint(q) & 0x7FFFFFFFu) >= 0x7F800000u ? 1.0f : q;
}

// Scale of a scaled second moment from its bound: kVTarget / bound, with
// the same guards as scale_from_amax_bits.
__device__ __forceinline__ float v_scale_from_bound(float b) {
  if (!(b > 0.0f) || (__float_as_uint(b) & 0x7FFFFFFFu) >= 0x7F800000u) return 1.0f;
  const float q = __fdiv_rn(kVTarget, b);
  return (__float_as_uint(q) & 0x7FFFFFFFu) >= 0x7F800000u ? 1.0f : q;
}

template <int FMT>
__device__ __forceinline__ float fp8_max_of() {
  return FMT == kE4M3 ? 448.0f : 57344.0f;
}

// Two FP8 codes (low byte first) -> two floats, exactly (through FP16).
template <int FMT>
__device__ __forceinline__ float2 dec2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
      (__nv_fp8x2_storage_t)two, FMT == kE4M3 ? __NV_E4M3 : __NV_E5M2);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Two floats -> two FP8 codes (x in the low byte), nearest-even, finite
// overflow saturated.  Only for finite inputs.
template <int FMT>
__device__ __forceinline__ uint32_t enc2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(
      make_float2(a, b), __NV_SATFINITE, FMT == kE4M3 ? __NV_E4M3 : __NV_E5M2);
}

// One float -> code, with the non-finite cases selected explicitly (the
// saturating conversion would map an infinity to the maximum).
template <int FMT>
__device__ __forceinline__ uint32_t enc1_checked(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0x7Fu;
  if ((b & 0x7FFFFFFFu) == 0x7F800000u)
    return FMT == kE4M3 ? 0x7Fu : ((b >> 31) ? 0xFCu : 0x7Cu);
  return (uint32_t)__nv_cvt_float_to_fp8(
      x, __NV_SATFINITE, FMT == kE4M3 ? __NV_E4M3 : __NV_E5M2);
}

// Eight floats -> eight codes packed in a uint2 (element 0 in the low byte).
template <int FMT, bool CHECKED>
__device__ __forceinline__ uint2 enc8(const float (&x)[8]) {
  uint32_t p[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (CHECKED)
      p[j] = enc1_checked<FMT>(x[2 * j]) | (enc1_checked<FMT>(x[2 * j + 1]) << 8);
    else
      p[j] = enc2<FMT>(x[2 * j], x[2 * j + 1]);
  }
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// Eight codes in a uint2 -> eight floats.
template <int FMT>
__device__ __forceinline__ void dec8(uint2 c, float (&x)[8]) {
  float2 a = dec2<FMT>(c.x & 0xFFFFu), b = dec2<FMT>(c.x >> 16);
  float2 d = dec2<FMT>(c.y & 0xFFFFu), e = dec2<FMT>(c.y >> 16);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  x[4] = d.x; x[5] = d.y; x[6] = e.x; x[7] = e.y;
}

// Eight FP16 in a uint4 -> eight floats, and back (nearest-even).
__device__ __forceinline__ void h8_to_f(uint4 h, float (&x)[8]) {
  const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
    x[2 * j] = f.x;
    x[2 * j + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 f_to_h8(const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __half2 h = __floats2half2_rn(x[2 * j], x[2 * j + 1]);
    w[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint16_t f_to_h(float x) {
  __half h = __float2half_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float h_to_f(uint16_t b) {
  return __half2float(*reinterpret_cast<const __half*>(&b));
}

// Paired fp32 arithmetic (one instruction for two lanes of a float2).  Each
// lane is rounded exactly like the scalar operation (round to nearest even,
// denormals kept).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// a * b + c with one rounding per lane.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

// Loads.  ld_keep: read-only data that a later pass reads again (normal
// caching, through the non-coherent path).  ld_once: data read for the last
// time in this call, including buffers this kernel overwrites in place
// (cache-streaming, evict-first; coherent path).
__device__ __forceinline__ uint2 ld_keep2(const void* p) {
  return __ldg(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ uint4 ld_keep4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint2 ld_once2(const void* p) {
  return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ uint4 ld_once4(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// ------------------------------------------- shared by several kernels

__device__ __forceinline__ uint32_t nonfinite(float x) {
  return (__float_as_uint(x) & 0x7FFFFFFFu) >= 0x7F800000u;
}

__device__ __forceinline__ uint32_t abs_bits(float x) {
  return __float_as_uint(x) & 0x7FFFFFFFu;
}

// The GradScaler test of a chunk of gradient codes as one comparison per
// code.  |decode(code) * k| depends only on the code's magnitude (code &
// 0x7F), and rounds monotonically in it; the non-finite codes (E4M3 0x7F,
// E5M2 0x7C and above) are the format's largest magnitudes and never give a
// finite product.  The magnitudes whose unscaled value is not finite are
// therefore one upper range [T, 0x7F] (T is 0 when k is not finite: 0 * inf
// is NaN), and overflow_threshold returns T: lane l of the warp tests
// magnitudes l, l + 32, l + 64 and l + 96, and the lowest failing one is T
// (0x7F always fails).  Every lane of the warp must call it; all get T.
template <int FMT>
__device__ __forceinline__ uint32_t overflow_threshold(float k) {
  const uint32_t lane = threadIdx.x & 31u;
  const float2 a = dec2<FMT>(lane | ((lane + 32u) << 8));
  const float2 b = dec2<FMT>((lane + 64u) | ((lane + 96u) << 8));
  const uint32_t m0 = __ballot_sync(0xFFFFFFFFu, nonfinite(__fmul_rn(a.x, k)));
  const uint32_t m1 = __ballot_sync(0xFFFFFFFFu, nonfinite(__fmul_rn(a.y, k)));
  const uint32_t m2 = __ballot_sync(0xFFFFFFFFu, nonfinite(__fmul_rn(b.x, k)));
  const uint32_t m3 = __ballot_sync(0xFFFFFFFFu, nonfinite(__fmul_rn(b.y, k)));
  return m0 ? __ffs(m0) - 1u : m1 ? 31u + __ffs(m1)
       : m2 ? 63u + __ffs(m2) : 95u + __ffs(m3);
}

// The per-byte addend of codes_at_least for threshold T (0 <= T <= 0x80).
__device__ __forceinline__ uint32_t threshold_addend(uint32_t t) {
  return (0x80u - t) * 0x01010101u;
}

// Bit 7 of each byte of w (four codes) whose magnitude is at least T, given
// add = threshold_addend(T): a magnitude m <= 0x7F plus 0x80 - T reaches 0x80
// exactly when m >= T, and never carries into the next byte.
__device__ __forceinline__ uint32_t codes_at_least(uint32_t w, uint32_t add) {
  return ((w & 0x7F7F7F7Fu) + add) & 0x80808080u;
}

// Two FP16 (one 32-bit word) <-> float2.
__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ uint32_t f2_to_h2(float2 f) {
  __half2 h = __float22half2_rn(f);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Code pair j (0..3) of eight codes held in a uint2.
__device__ __forceinline__ uint32_t code_pair(uint2 c, int j) {
  const uint32_t w = j < 2 ? c.x : c.y;
  return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}

__device__ __forceinline__ uint32_t half_pair(uint4 h, int j) {
  return j == 0 ? h.x : j == 1 ? h.y : j == 2 ? h.z : h.w;
}

// Eight source elements of type DT from element i0 (vector path, last use),
// and one element (scalar path), widened exactly to fp32.
template <int DT>
__device__ __forceinline__ void load8(const void* src, int64_t i0,
                                      float (&x)[8]) {
  if (DT == kF32) {
    const float* f = static_cast<const float*>(src) + i0;
    const uint4 a = ld_once4(f), b = ld_once4(f + 4);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  } else {
    const uint4 a = ld_once4(static_cast<const uint16_t*>(src) + i0);
    if (DT == kF16) {
      h8_to_f(a, x);
    } else {
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
}

template <int DT>
__device__ __forceinline__ float load1(const void* src, int64_t i) {
  if (DT == kF32) return static_cast<const float*>(src)[i];
  const uint16_t b = static_cast<const uint16_t*>(src)[i];
  if (DT == kF16) return h_to_f(b);
  return __uint_as_float((uint32_t)b << 16);
}

// Asynchronous bulk prefetch of [p, p + bytes) into L2 (no shared memory, no
// completion to wait for).  p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
               :: "l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Max over the CTA (NT threads) of a per-thread uint32; the result is valid
// in thread 0.  Every thread of the CTA must call it.
template <int NT = kThreads>
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* smem) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();                 // smem may still be read by a prior call
  if (lane == 0) smem[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < (NT / 32) ? smem[lane] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
  }
  return v;
}

// ------------------------------------- exact sums of squared FP8 code values
//
// Every E4M3 or E5M2 code's value is a multiple of 2^-16, so its square is an
// integer count of 2^-32 and a tensor's sum of squares can be taken exactly:
//   E4M3: r = |value| * 2^9 is an integer below 2^18, r^2 below 2^36 in
//         units of 2^-18, summed in 64 bits per thread;
//   E5M2: r = |value| * 2^16 is an integer below 2^32, r^2 below 2^64 in
//         units of 2^-32, summed in 128 bits per thread (or, where a pass
//         has one code format, as two 64-bit sums: SqSum<kE5M2>).
// Integer sums are exact and order-free, so a norm built on them does not
// depend on the kernel schedule.

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

// The exact sums go through a shared-memory table of the integers r (r =
// |value| * 2^9 for E4M3, |value| * 2^16 for E5M2; 0 for the non-finite
// codes, which set found_inf instead), so that a code costs one byte
// permutation, one shared load and one multiply-add.  Entry [mag][fmt * 32 +
// lane] holds r of magnitude `mag` in format `fmt` for lane `lane`: the
// lanes of a warp always read 32 different banks, whatever their codes.
// __byte_perm(magnitudes, sq_lane_byte(), 0x5504 + 16 * j) is the byte
// offset of code j's entry: magnitude j in byte 1 (mag * 256), the format
// and lane in byte 0 (fmt * 128 + lane * 4).
struct SqTable {
  uint32_t r[128][64];   // 32 KB
};

// Fills the table (every thread of the CTA calls it; it ends with a CTA
// barrier).
__device__ __forceinline__ void sq_table_fill(SqTable& t) {
  for (int i = threadIdx.x; i < 128 * 64; i += blockDim.x) {
    const uint32_t mag = (uint32_t)i >> 6, e5 = ((uint32_t)i >> 5) & 1u;
    const float v = e5 ? dec2<kE5M2>(mag).x * 65536.0f : dec2<kE4M3>(mag).x * 512.0f;
    t.r[mag][i & 63] = (__float_as_uint(v) & 0x7FFFFFFFu) >= 0x7F800000u
                           ? 0u : __float2uint_rn(v);
  }
  __syncthreads();
}

// Byte 0 of an entry's offset: the format's column block and this lane's
// word within it.
template <int FMT>
__device__ __forceinline__ uint32_t sq_lane_byte() {
  return (FMT == kE4M3 ? 0u : 128u) + 4u * (threadIdx.x & 31u);
}

// A thread's exact sums through the table, for either format (a CTA may
// accumulate several chunks of one tensor before it commits).  E4M3 squares
// are below 2^36, so the 64-bit sum holds 2^28 codes a thread.
struct SqTab {
  unsigned long long s4 = 0;   // E4M3: units of 2^-18
  U128 s5 = {0ull, 0ull};      // E5M2: units of 2^-32

  // wm: four code magnitudes (sign bits cleared); lb: sq_lane_byte<FMT>().
  template <int FMT>
  __device__ __forceinline__ void add_word(uint32_t wm, uint32_t lb,
                                           const SqTable& t) {
    const char* base = reinterpret_cast<const char*>(&t);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t r = *reinterpret_cast<const uint32_t*>(
          base + __byte_perm(wm, lb, 0x5504u + 16u * j));
      if (FMT == kE4M3)
        s4 += (unsigned long long)r * r;
      else
        s5 = add64(s5, (unsigned long long)r * r);
    }
  }
  // the sum in units of 2^-32 (both formats' parts)
  __device__ __forceinline__ U128 sum() const {
    return add128(U128{s4 << 14, s4 >> 50}, s5);
  }
};

// Shared memory of sq_commit: each warp's partial sum and flag, in two
// buffers used in turn.
struct SqRed {
  unsigned long long w[2][3 * (kThreads / 32)];
};

// End of a run of chunks of tensor t for a table-summing pass: the CTA's
// exact sum (each thread's `sum`, in units of 2^-32) goes to the tensor's
// 128-bit slot (sums[2t], sums[2t + 1]; the low word's carry goes to the
// high word), and found_inf is set when any thread saw a non-finite value
// (`bad`, from the codes and the tensor's overflow threshold).  Warps reduce
// by shuffles; one CTA barrier then lets thread 0 add the warps' parts.  The
// buffers alternate (turn), so a warp writing the next commit's part cannot
// overtake thread 0's reading of this one: it first passes the barrier of
// the commit in between, which thread 0 reaches only after its reads.
// Every thread calls it, with the same nonempty and turn.
__device__ __forceinline__ void sq_commit(U128 v, uint32_t bad, uint32_t t,
                                          bool nonempty, unsigned long long* sums,
                                          unsigned long long* found,
                                          uint32_t epoch, SqRed& red,
                                          uint32_t& turn) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    U128 w;
    w.lo = __shfl_xor_sync(0xFFFFFFFFu, v.lo, o);
    w.hi = __shfl_xor_sync(0xFFFFFFFFu, v.hi, o);
    v = add128(v, w);
  }
  const bool wbad = __any_sync(0xFFFFFFFFu, bad != 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long* buf = red.w[turn];
  if (lane == 0) {
    buf[3 * warp] = v.lo;
    buf[3 * warp + 1] = v.hi;
    buf[3 * warp + 2] = wbad ? 1ull : 0ull;
  }
  __syncthreads();
  if (threadIdx.x == 0 && nonempty) {
    U128 s = {0ull, 0ull};
    unsigned long long any_bad = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      s = add128(s, U128{buf[3 * i], buf[3 * i + 1]});
      any_bad |= buf[3 * i + 2];
    }
    if (s.lo | s.hi) {
      const unsigned long long old = atomicAdd(&sums[2 * t], s.lo);
      const unsigned long long carry = old + s.lo < old ? 1ull : 0ull;
      if (s.hi + carry) atomicAdd(&sums[2 * t + 1], s.hi + carry);
    }
    if (any_bad) atomicMax(found, slot_tag(epoch, 1u));
  }
  turn ^= 1u;
}

// A thread's exact sum of squared code values for one code format (the
// passes whose codes all have one format), read through a shared-memory
// table of integer roots (one byte permutation gives each code's entry).
//   E4M3: SqTable's E4M3 columns, r = |value| * 2^9 below 2^18; r^2 summed
//         in 64 bits in units of 2^-18.
//   E5M2: Sq5Table, r = |value| * 2^16 below 2^32 split by the exponent field
//         e: for e <= 16, r is below 2^18 and r^2 goes to `lo` (units of
//         2^-32); for e >= 17, r is a multiple of 2^16 and (r / 2^16)^2,
//         below 2^32, goes to `hi` (units of 1).  Each entry holds {r, 0} or
//         {0, r / 2^16} for the lane reading it, so a code costs one 64-bit
//         shared load and two multiply-adds instead of a 128-bit addition.
// Both 64-bit sums hold at least 2^28 codes a thread.
struct Sq5Table {
  uint2 t[128][32];   // [magnitude][lane], 32 KB; rows of 256 bytes
};

__device__ __forceinline__ void sq5_table_fill(Sq5Table& t) {
  for (int i = threadIdx.x; i < 128 * 32; i += blockDim.x) {
    const uint32_t mag = (uint32_t)i >> 5, e = mag >> 2;
    const float v = dec2<kE5M2>(mag).x * 65536.0f;
    const uint32_t r = e == 31 ? 0u : __float2uint_rn(v);   // e == 31: inf, NaN
    t.t[mag][i & 31] = e <= 16 ? make_uint2(r, 0u) : make_uint2(0u, r >> 16);
  }
  __syncthreads();
}

template <int FMT>
struct SqSum;

template <>
struct SqSum<kE4M3> {
  using Table = SqTable;
  const SqTable* tab;
  SqTab s;
  __device__ __forceinline__ explicit SqSum(const SqTable* t) : tab(t) {}
  // wm: four code magnitudes (sign bits cleared)
  __device__ __forceinline__ void add_word(uint32_t wm) {
    s.add_word<kE4M3>(wm, sq_lane_byte<kE4M3>(), *tab);
  }
  __device__ __forceinline__ U128 sum() const { return s.sum(); }
  __device__ __forceinline__ void clear() { s = SqTab(); }
};

template <>
struct SqSum<kE5M2> {
  using Table = Sq5Table;
  const Sq5Table* tab;
  unsigned long long lo = 0, hi = 0;
  __device__ __forceinline__ explicit SqSum(const Sq5Table* t) : tab(t) {}
  __device__ __forceinline__ void add_word(uint32_t wm) {
    const char* base = reinterpret_cast<const char*>(tab);
    const uint32_t lb = 8u * (threadIdx.x & 31u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // byte 1: code j's magnitude (its row), byte 0: this lane's entry
      const uint2 e = *reinterpret_cast<const uint2*>(
          base + __byte_perm(wm, lb, 0x5504u + 16u * j));
      lo += (unsigned long long)e.x * e.x;
      hi += (unsigned long long)e.y * e.y;
    }
  }
  // lo + hi * 2^32, in units of 2^-32
  __device__ __forceinline__ U128 sum() const {
    return add128(U128{lo, 0ull}, U128{hi << 32, hi >> 32});
  }
  __device__ __forceinline__ void clear() { lo = hi = 0; }
};

template <int FMT>
__device__ __forceinline__ void sq_table_fill_fmt(typename SqSum<FMT>::Table& t) {
  if constexpr (FMT == kE4M3)
    sq_table_fill(t);
  else
    sq5_table_fill(t);
}

// Correctly rounded conversion of a 128-bit unsigned integer to double: the
// top 64 bits after normalisation, with every lower bit folded into the
// lowest one (a sticky bit, eleven places below the rounding position), then
// an exact power-of-two scaling.
__device__ __forceinline__ double u128_to_double(U128 v) {
  if (v.hi == 0) return __ull2double_rn(v.lo);
  const int lz = __clzll((long long)v.hi);
  const unsigned long long top = lz ? (v.hi << lz) | (v.lo >> (64 - lz)) : v.hi;
  const unsigned long long rest = v.lo << lz;
  const double d = __ull2double_rn(top | (rest != 0 ? 1ull : 0ull));
  return __dmul_rn(d, __longlong_as_double((long long)(1023 + 64 - lz) << 52));
}

// A record's norm term from its exact sum S (units of 2^-32) and factor k:
// fl64(k^2 * fl64(S * 2^-32)), where k^2 and the power-of-two scaling are
// exact in double.
__device__ __forceinline__ double norm_term(U128 s, float k) {
  const double kd = (double)k;
  return __dmul_rn(__dmul_rn(kd, kd), __dmul_rn(u128_to_double(s), 0x1p-32));
}

}  // namespace fp8opt
