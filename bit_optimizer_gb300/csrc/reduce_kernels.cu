// Local reduction of FP8 shards: the arithmetic half of an FP8 all-reduce
// (MS-AMP O1 keeps weight gradients and their AllReduce communication in FP8).
//
// k shards of one tensor, shard j encoded with its own scale s_j, are summed
// per element as y = post * (((x_0 + x_1) + x_2) + ...), x_j = decode(c_j) *
// (1 / s_j), in fp32 with every product and sum rounded on its own, and y is
// cast back to FP8 with a just-in-time per-tensor scale.  Two persistent
// kernels over the chunk table, like the cast:
//   reduce_amax_kernel    y per element, per-tensor max |y| (NaN above +inf
//                         above every finite value) into the tagged slots.
//   reduce_encode_kernel  scale = fp8_max / amax in each chunk's prologue, y
//                         again, code = encode(y * scale).  It walks the
//                         chunk table backwards so the chunks the first pass
//                         read last are still in L2.
// Bytes per element: k (first pass) + k + 1 (encode).  With 1, 2, 4 or 8
// shards both passes run in forms specialised on k (reduce_amax_small_kernel,
// reduce_encode_small_kernel).
//
// Vector path: thread t of a CTA takes the 16-code groups at tile + g *
// (kThreads * 16) + t * 16 (g = 0, 1): one 16-byte load per shard and group,
// issued for kShardBatch shards at a time before their sums, so a warp's
// every access is one contiguous 512-byte span and a thread keeps four loads
// in flight.  A
// tensor whose sum has a non-finite element (amax not finite) is encoded on
// the scalar path, which selects the NaN / infinity codes explicitly.
#include "fp8opt_internal.cuh"

namespace fp8opt {

cudaError_t launch_sums_to_limbs(const unsigned long long* sums, int n,
                                 const unsigned long long* found, uint32_t epoch,
                                 long long* limbs, uint32_t* found_out,
                                 cudaStream_t stream);

namespace {

// Tunables: 16-code groups per thread per tile, shards whose loads are issued
// before their sums, resident CTAs per SM both kernels are compiled for (caps
// their registers), and tiles ahead of the current one that one thread per
// CTA prefetches into L2 (0: none).
#ifndef FP8OPT_REDUCE_GROUPS
#define FP8OPT_REDUCE_GROUPS 2
#endif
#ifndef FP8OPT_REDUCE_BATCH
#define FP8OPT_REDUCE_BATCH 2
#endif
#ifndef FP8OPT_REDUCE_MIN_BLOCKS
#define FP8OPT_REDUCE_MIN_BLOCKS 3
#endif
#ifndef FP8OPT_REDUCE_PREFETCH
#define FP8OPT_REDUCE_PREFETCH 1
#endif
// Resident CTAs per SM of the general encode pass with exact squares.
#ifndef FP8OPT_REDUCE_SQ_MIN_BLOCKS
#define FP8OPT_REDUCE_SQ_MIN_BLOCKS 2
#endif
// The passes specialised on k (1, 2, 4 or 8 shards): 16-code groups per
// thread per tile and resident CTAs per SM for each k.  Measured on the 124M
// list (the whole reduction):
//   k = 2: 0.111 ms with two groups and 4 CTAs/SM, 0.113 with four groups,
//          0.119 on the general kernel;
//   k = 4: 0.175 ms with two groups at 4 CTAs/SM, 0.176 with one group,
//          0.193 on the general kernel;
//   k = 8: 0.316 ms with one group at 3 CTAs/SM, 0.321 at 4, 0.351 on the
//          general kernel.
#ifndef FP8OPT_RSMALL_GROUPS
#define FP8OPT_RSMALL_GROUPS 2
#endif
#ifndef FP8OPT_RSMALL_MIN_BLOCKS
#define FP8OPT_RSMALL_MIN_BLOCKS 4
#endif
#ifndef FP8OPT_RSMALL_G4
#define FP8OPT_RSMALL_G4 2
#endif
#ifndef FP8OPT_RSMALL_MIN_BLOCKS_K4
#define FP8OPT_RSMALL_MIN_BLOCKS_K4 4
#endif
#ifndef FP8OPT_RSMALL_G8
#define FP8OPT_RSMALL_G8 1
#endif
#ifndef FP8OPT_RSMALL_MIN_BLOCKS_K8
#define FP8OPT_RSMALL_MIN_BLOCKS_K8 3
#endif

constexpr int kRGroup = 16;    // codes per vector group (one 16-byte access)
constexpr int kRGroups = FP8OPT_REDUCE_GROUPS;
constexpr int kShardBatch = FP8OPT_REDUCE_BATCH;
constexpr int64_t kRTile = (int64_t)kThreads * kRGroup * kRGroups;

// L2 prefetch of the tile FP8OPT_REDUCE_PREFETCH tiles after `base`, every
// shard (thread 0 only; vector path, so the rows are 16-byte aligned).
__device__ __forceinline__ void prefetch_tiles(const uint8_t* src, int64_t stride,
                                               int k, int64_t base, int64_t end) {
  if (FP8OPT_REDUCE_PREFETCH == 0 || threadIdx.x != 0) return;
  const int64_t ahead = base + FP8OPT_REDUCE_PREFETCH * kRTile;
  if (ahead + kRTile > end) return;
  for (int j = 0; j < k; ++j)
    prefetch_l2(src + (int64_t)j * stride + ahead, (uint32_t)kRTile);
}

// acc (+)= decode(16 codes) * r.  The product and the sum are the scalar
// round-to-nearest intrinsics, which are never merged into a fused
// multiply-add: the sum must round twice, as written.
__device__ __forceinline__ float2 mul_add2(float2 acc, float2 x, float r) {
  return make_float2(__fadd_rn(acc.x, __fmul_rn(x.x, r)),
                     __fadd_rn(acc.y, __fmul_rn(x.y, r)));
}

template <int IN, bool FIRST>
__device__ __forceinline__ void accum16(uint4 c, float r, float2 (&acc)[8]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 a = dec2<IN>(w[q] & 0xFFFFu), b = dec2<IN>(w[q] >> 16);
    if (FIRST) {
      acc[2 * q] = make_float2(__fmul_rn(a.x, r), __fmul_rn(a.y, r));
      acc[2 * q + 1] = make_float2(__fmul_rn(b.x, r), __fmul_rn(b.y, r));
    } else {
      acc[2 * q] = mul_add2(acc[2 * q], a, r);
      acc[2 * q + 1] = mul_add2(acc[2 * q + 1], b, r);
    }
  }
}

// y for this thread's kRGroups full 16-code groups at i0[g]: the shard-order
// sum times post.  LAST: the codes are read for the last time (encode pass).
template <int IN, bool LAST>
__device__ __forceinline__ void reduce_groups(const uint8_t* src, int64_t stride,
                                              int k, const float* r_s,
                                              float post, const int64_t (&i0)[kRGroups],
                                              float2 (&y)[kRGroups][8]) {
#pragma unroll 1
  for (int j0 = 0; j0 < k; j0 += kShardBatch) {
    uint4 c[kShardBatch][kRGroups];
#pragma unroll
    for (int b = 0; b < kShardBatch; ++b) {
      if (j0 + b < k) {
        const uint8_t* p = src + (int64_t)(j0 + b) * stride;
#pragma unroll
        for (int g = 0; g < kRGroups; ++g)
          c[b][g] = LAST ? ld_once4(p + i0[g]) : ld_keep4(p + i0[g]);
      }
    }
#pragma unroll
    for (int b = 0; b < kShardBatch; ++b) {
      if (j0 + b < k) {
        const float r = r_s[j0 + b];
#pragma unroll
        for (int g = 0; g < kRGroups; ++g) {
          if (j0 + b == 0)
            accum16<IN, true>(c[b][g], r, y[g]);
          else
            accum16<IN, false>(c[b][g], r, y[g]);
        }
      }
    }
  }
  const float2 pp = splat2(post);
#pragma unroll
  for (int g = 0; g < kRGroups; ++g)
#pragma unroll
    for (int q = 0; q < 8; ++q) y[g][q] = mul2(y[g][q], pp);
}

// y of one element (scalar path: unaligned buffers and ragged tails).
template <int IN>
__device__ __forceinline__ float reduce_one(const uint8_t* src, int64_t stride,
                                            int k, const float* r_s, float post,
                                            int64_t i) {
  float acc = __fmul_rn(dec2<IN>(src[i]).x, r_s[0]);
  for (int j = 1; j < k; ++j)
    acc = __fadd_rn(acc, __fmul_rn(dec2<IN>(src[(int64_t)j * stride + i]).x, r_s[j]));
  return __fmul_rn(acc, post);
}

// r_s[j] = 1 / s_j for this chunk's tensor (one IEEE division per shard).
__device__ __forceinline__ void load_reciprocals(const ReduceDesc& d, int k,
                                                 float* r_s) {
  __syncthreads();   // the previous chunk may still be reading r_s
  if (threadIdx.x < k && d.numel > 0)
    r_s[threadIdx.x] = __fdiv_rn(1.0f, d.src_scale[threadIdx.x]);
  __syncthreads();
}

// ---------------------------------------------------------------- amax pass

template <int IN>
__device__ uint32_t thread_reduce_amax(const ReduceDesc& d, int k,
                                       const float* r_s, float post,
                                       int64_t begin, int64_t end) {
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  uint32_t mx = 0;
#pragma unroll 1
  for (int64_t base = begin; base < end; base += kRTile) {
    if (vec && base + kRTile <= end) {
      prefetch_tiles(d.src, d.stride, k, base, end);
      int64_t i0[kRGroups];
#pragma unroll
      for (int g = 0; g < kRGroups; ++g)
        i0[g] = base + g * (kThreads * kRGroup) + tid * kRGroup;
      float2 y[kRGroups][8];
      reduce_groups<IN, false>(d.src, d.stride, k, r_s, post, i0, y);
#pragma unroll
      for (int g = 0; g < kRGroups; ++g)
#pragma unroll
        for (int q = 0; q < 8; ++q)
          mx = max(mx, max(abs_bits(y[g][q].x), abs_bits(y[g][q].y)));
    } else {
#pragma unroll 1
      for (int g = 0; g < kRGroups; ++g) {
        const int64_t i0 = base + g * (kThreads * kRGroup) + tid * kRGroup;
        for (int e = 0; e < kRGroup; ++e) {
          const int64_t i = i0 + e;
          if (i >= end) break;
          mx = max(mx, abs_bits(reduce_one<IN>(d.src, d.stride, k, r_s, post, i)));
        }
      }
    }
  }
  return mx;
}

template <int IN>
__global__ void __launch_bounds__(kThreads, FP8OPT_REDUCE_MIN_BLOCKS)
reduce_amax_kernel(const ReduceDesc* __restrict__ descs,
                   const Chunk* __restrict__ chunks, uint32_t nchunks, int k,
                   float post, unsigned long long* __restrict__ slots,
                   uint32_t epoch) {
  __shared__ uint32_t red[kThreads / 32];
  __shared__ float r_s[kMaxShards];
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const ReduceDesc d = descs[ch.tensor];
    load_reciprocals(d, k, r_s);
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    uint32_t mx = thread_reduce_amax<IN>(d, k, r_s, post, begin, end);
    mx = block_max_u32(mx, red);
    if (threadIdx.x == 0 && mx != 0)
      atomicMax(&slots[ch.tensor], slot_tag(epoch, canon_amax_bits(mx)));
  }
}

// Groups per thread per tile and CTAs per SM of the k-specialised passes.
template <int K>
__host__ __device__ constexpr int small_groups() {
  return K <= 2 ? FP8OPT_RSMALL_GROUPS : K == 4 ? FP8OPT_RSMALL_G4 : FP8OPT_RSMALL_G8;
}
template <int K>
__host__ __device__ constexpr int small_min_blocks() {
  return K <= 2   ? FP8OPT_RSMALL_MIN_BLOCKS
         : K == 4 ? FP8OPT_RSMALL_MIN_BLOCKS_K4
                  : FP8OPT_RSMALL_MIN_BLOCKS_K8;
}

// The first pass for K = 1, 2, 4 or 8 shards.  Every shard's loads for all
// the tile's groups are issued first.  Each group's sum is then reduced to
// its max at once, not kept for the encode.  A thread thus keeps
// K * small_groups<K>() 16-byte loads in flight in few registers, so more
// CTAs fit on an SM than the general kernel's three.  The sum is the same
// expression as in reduce_groups, so y and its max are identical.
template <int IN, int K>
__global__ void __launch_bounds__(kThreads, small_min_blocks<K>())
reduce_amax_small_kernel(const ReduceDesc* __restrict__ descs,
                         const Chunk* __restrict__ chunks, uint32_t nchunks,
                         float post, unsigned long long* __restrict__ slots,
                         uint32_t epoch) {
  __shared__ uint32_t red[kThreads / 32];
  __shared__ float r_s[kMaxShards];
  constexpr int kSGroups = small_groups<K>();
  constexpr int64_t kSTile = (int64_t)kThreads * kRGroup * kSGroups;
  const int tid = threadIdx.x;
  const float2 pp = splat2(post);
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const ReduceDesc d = descs[ch.tensor];
    load_reciprocals(d, K, r_s);
    float r[K];
#pragma unroll
    for (int j = 0; j < K; ++j) r[j] = r_s[j];
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    const bool vec = d.vec_ok != 0;
    uint32_t mx = 0;
#pragma unroll 1
    for (int64_t base = begin; base < end; base += kSTile) {
      if (vec && base + kSTile <= end) {
        if (FP8OPT_REDUCE_PREFETCH > 0 && tid == 0) {
          const int64_t ahead = base + FP8OPT_REDUCE_PREFETCH * kSTile;
          if (ahead + kSTile <= end)
            for (int j = 0; j < K; ++j)
              prefetch_l2(d.src + (int64_t)j * d.stride + ahead, (uint32_t)kSTile);
        }
        uint4 cv[K][kSGroups];
#pragma unroll
        for (int j = 0; j < K; ++j)
#pragma unroll
          for (int g = 0; g < kSGroups; ++g)
            cv[j][g] = ld_keep4(d.src + (int64_t)j * d.stride + base +
                                g * (kThreads * kRGroup) + tid * kRGroup);
#pragma unroll
        for (int g = 0; g < kSGroups; ++g) {
          float2 y[8];
          accum16<IN, true>(cv[0][g], r[0], y);
#pragma unroll
          for (int j = 1; j < K; ++j) accum16<IN, false>(cv[j][g], r[j], y);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float2 t = mul2(y[q], pp);
            mx = max(mx, max(abs_bits(t.x), abs_bits(t.y)));
          }
        }
      } else {
#pragma unroll 1
        for (int g = 0; g < kSGroups; ++g) {
          const int64_t i0 = base + g * (kThreads * kRGroup) + tid * kRGroup;
          for (int e = 0; e < kRGroup; ++e) {
            const int64_t i = i0 + e;
            if (i >= end) break;
            mx = max(mx, abs_bits(reduce_one<IN>(d.src, d.stride, K, r_s, post, i)));
          }
        }
      }
    }
    mx = block_max_u32(mx, red);
    if (threadIdx.x == 0 && mx != 0)
      atomicMax(&slots[ch.tensor], slot_tag(epoch, canon_amax_bits(mx)));
  }
}

template <int IN>
void launch_amax(uint32_t grid, const ReduceDesc* descs, const Chunk* chunks,
                 uint32_t nchunks, int k, float post, unsigned long long* slots,
                 uint32_t epoch, cudaStream_t stream) {
  if (k == 1)
    reduce_amax_small_kernel<IN, 1><<<grid, kThreads, 0, stream>>>(
        descs, chunks, nchunks, post, slots, epoch);
  else if (k == 2)
    reduce_amax_small_kernel<IN, 2><<<grid, kThreads, 0, stream>>>(
        descs, chunks, nchunks, post, slots, epoch);
  else if (k == 4)
    reduce_amax_small_kernel<IN, 4><<<grid, kThreads, 0, stream>>>(
        descs, chunks, nchunks, post, slots, epoch);
  else if (k == 8)
    reduce_amax_small_kernel<IN, 8><<<grid, kThreads, 0, stream>>>(
        descs, chunks, nchunks, post, slots, epoch);
  else
    reduce_amax_kernel<IN><<<grid, kThreads, 0, stream>>>(descs, chunks, nchunks,
                                                          k, post, slots, epoch);
}

// -------------------------------------------------------------- encode pass

// Sixteen finite y -> sixteen codes of format OUT in a uint4.
template <int OUT>
__device__ __forceinline__ uint4 encode16(const float2 (&y)[8], float scale) {
  const float2 ss = splat2(scale);
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 a = mul2(y[2 * q], ss), b = mul2(y[2 * q + 1], ss);
    w[q] = enc2<OUT>(a.x, a.y) | (enc2<OUT>(b.x, b.y) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sixteen codes written by an encode pass: their exact squares into acc, and
// into bad the codes at or above the overflow threshold whose addend is tadd.
template <int OUT>
__device__ __forceinline__ void sq_add16(uint4 c, uint32_t tadd, SqSum<OUT>& acc,
                                         uint32_t& bad) {
  bad |= codes_at_least(c.x, tadd) | codes_at_least(c.y, tadd) |
         codes_at_least(c.z, tadd) | codes_at_least(c.w, tadd);
  acc.add_word(c.x & 0x7F7F7F7Fu);
  acc.add_word(c.y & 0x7F7F7F7Fu);
  acc.add_word(c.z & 0x7F7F7F7Fu);
  acc.add_word(c.w & 0x7F7F7F7Fu);
}

// SQ: also add the exact squares of the codes written to acc and collect in
// bad the codes at or above the overflow threshold whose addend is tadd.
template <int IN, int OUT, bool CHECKED, bool SQ>
__device__ void thread_reduce_encode(const ReduceDesc& d, int k,
                                     const float* r_s, float post, float scale,
                                     int64_t begin, int64_t end,
                                     SqSum<OUT>& acc, uint32_t tadd,
                                     uint32_t& bad) {
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0 && !CHECKED;
#pragma unroll 1
  for (int64_t base = begin; base < end; base += kRTile) {
    if (vec && base + kRTile <= end) {
      prefetch_tiles(d.src, d.stride, k, base, end);
      int64_t i0[kRGroups];
#pragma unroll
      for (int g = 0; g < kRGroups; ++g)
        i0[g] = base + g * (kThreads * kRGroup) + tid * kRGroup;
      float2 y[kRGroups][8];
      reduce_groups<IN, true>(d.src, d.stride, k, r_s, post, i0, y);
#pragma unroll
      for (int g = 0; g < kRGroups; ++g) {
        const uint4 c = encode16<OUT>(y[g], scale);
        *reinterpret_cast<uint4*>(d.codes + i0[g]) = c;
        if (SQ) sq_add16(c, tadd, acc, bad);
      }
    } else {
#pragma unroll 1
      for (int g = 0; g < kRGroups; ++g) {
        const int64_t i0 = base + g * (kThreads * kRGroup) + tid * kRGroup;
        for (int e = 0; e < kRGroup; ++e) {
          const int64_t i = i0 + e;
          if (i >= end) break;
          const float t =
              __fmul_rn(reduce_one<IN>(d.src, d.stride, k, r_s, post, i), scale);
          const uint32_t c = CHECKED ? enc1_checked<OUT>(t)
                                     : (enc2<OUT>(t, 0.0f) & 0xFFu);
          d.codes[i] = (uint8_t)c;
          if (SQ) {
            bad |= ((c & 0x7Fu) + tadd) & 0x80u;
            acc.add_word(c & 0x7Fu);
          }
        }
      }
    }
  }
}

// The encode pass's vector path for K = 1, 2, 4 or 8 shards (finite amax):
// like reduce_amax_small_kernel, all loads of the tile first, then each
// group is summed, encoded and stored at once.
template <int IN, int OUT, int K, bool SQ>
__device__ void thread_reduce_encode_small(const ReduceDesc& d, const float* r_s,
                                           float post, float scale,
                                           int64_t begin, int64_t end,
                                           SqSum<OUT>& acc, uint32_t tadd,
                                           uint32_t& bad) {
  constexpr int kSGroups = small_groups<K>();
  constexpr int64_t kSTile = (int64_t)kThreads * kRGroup * kSGroups;
  const int tid = threadIdx.x;
  const bool vec = d.vec_ok != 0;
  const float2 pp = splat2(post);
  float r[K];
#pragma unroll
  for (int j = 0; j < K; ++j) r[j] = r_s[j];
#pragma unroll 1
  for (int64_t base = begin; base < end; base += kSTile) {
    if (vec && base + kSTile <= end) {
      if (FP8OPT_REDUCE_PREFETCH > 0 && tid == 0) {
        const int64_t ahead = base + FP8OPT_REDUCE_PREFETCH * kSTile;
        if (ahead + kSTile <= end)
          for (int j = 0; j < K; ++j)
            prefetch_l2(d.src + (int64_t)j * d.stride + ahead, (uint32_t)kSTile);
      }
      uint4 cv[K][kSGroups];
#pragma unroll
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int g = 0; g < kSGroups; ++g)
          cv[j][g] = ld_once4(d.src + (int64_t)j * d.stride + base +
                              g * (kThreads * kRGroup) + tid * kRGroup);
#pragma unroll
      for (int g = 0; g < kSGroups; ++g) {
        float2 y[8];
        accum16<IN, true>(cv[0][g], r[0], y);
#pragma unroll
        for (int j = 1; j < K; ++j) accum16<IN, false>(cv[j][g], r[j], y);
#pragma unroll
        for (int q = 0; q < 8; ++q) y[q] = mul2(y[q], pp);
        const uint4 c = encode16<OUT>(y, scale);
        *reinterpret_cast<uint4*>(d.codes + base + g * (kThreads * kRGroup) +
                                  tid * kRGroup) = c;
        if (SQ) sq_add16(c, tadd, acc, bad);
      }
    } else {
#pragma unroll 1
      for (int g = 0; g < kSGroups; ++g) {
        const int64_t i0 = base + g * (kThreads * kRGroup) + tid * kRGroup;
        for (int e = 0; e < kRGroup; ++e) {
          const int64_t i = i0 + e;
          if (i >= end) break;
          const float t =
              __fmul_rn(reduce_one<IN>(d.src, d.stride, K, r_s, post, i), scale);
          const uint32_t c = enc2<OUT>(t, 0.0f) & 0xFFu;
          d.codes[i] = (uint8_t)c;
          if (SQ) {
            bad |= ((c & 0x7Fu) + tadd) & 0x80u;
            acc.add_word(c & 0x7Fu);
          }
        }
      }
    }
  }
}

// Where an encode pass also sums the exact squares of the codes it writes
// (the gradient norm of the reduced tensors): the 128-bit slots, the
// found_inf slot and the inverse loss scale.
struct RedSq {
  unsigned long long* sums;
  unsigned long long* found;
  float ils;
};

// KS: 0, or the number of shards (1, 2, 4 or 8) the vector path is
// specialised on.  SQ: with the exact squares of the codes through the table
// tab, committed to the tensor's slot per chunk, and found_inf from the
// overflow threshold of k = inv_loss_scale / the output scale.
template <int IN, int OUT, bool SQ, int KS>
__device__ __forceinline__ void encode_pass(const ReduceDesc* __restrict__ descs,
                                            const Chunk* __restrict__ chunks,
                                            uint32_t nchunks, int k, float post,
                                            const unsigned long long* __restrict__ slots,
                                            uint32_t epoch, const RedSq& sq,
                                            float* r_s,
                                            const typename SqSum<OUT>::Table* tab,
                                            SqRed* red) {
  SqSum<OUT> acc(tab);
  uint32_t turn = 0;
  for (uint32_t r = blockIdx.x; r < nchunks; r += gridDim.x) {
    const Chunk ch = chunks[nchunks - 1 - r];
    const ReduceDesc d = descs[ch.tensor];
    load_reciprocals(d, k, r_s);
    const uint32_t ab = slot_value(slots[ch.tensor], epoch);
    const float scale = scale_from_amax_bits(ab, fp8_max_of<OUT>());
    if (ch.begin == 0 && threadIdx.x == 0) {
      *d.amax_out = __uint_as_float(ab);
      *d.scale_out = scale;
    }
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    uint32_t tadd = 0, bad = 0;
    if (SQ)
      tadd = threshold_addend(overflow_threshold<OUT>(__fdiv_rn(sq.ils, scale)));
    if (ab >= 0x7F800000u)
      thread_reduce_encode<IN, OUT, true, SQ>(d, k, r_s, post, scale, begin, end,
                                              acc, tadd, bad);
    else if (KS > 0)
      thread_reduce_encode_small<IN, OUT, (KS > 0 ? KS : 1), SQ>(
          d, r_s, post, scale, begin, end, acc, tadd, bad);
    else
      thread_reduce_encode<IN, OUT, false, SQ>(d, k, r_s, post, scale, begin, end,
                                               acc, tadd, bad);
    if (SQ) {
      sq_commit(acc.sum(), bad, ch.tensor, end > begin, sq.sums, sq.found, epoch,
                *red, turn);
      acc.clear();
    }
  }
}

template <int IN, int OUT>
__global__ void __launch_bounds__(kThreads, FP8OPT_REDUCE_MIN_BLOCKS)
reduce_encode_kernel(const ReduceDesc* __restrict__ descs,
                     const Chunk* __restrict__ chunks, uint32_t nchunks, int k,
                     float post, const unsigned long long* __restrict__ slots,
                     uint32_t epoch) {
  __shared__ float r_s[kMaxShards];
  const RedSq none = {nullptr, nullptr, 0.0f};
  encode_pass<IN, OUT, false, 0>(descs, chunks, nchunks, k, post, slots, epoch,
                                 none, r_s, nullptr, nullptr);
}

template <int IN, int OUT, int K>
__global__ void __launch_bounds__(kThreads, small_min_blocks<K>())
reduce_encode_small_kernel(const ReduceDesc* __restrict__ descs,
                           const Chunk* __restrict__ chunks, uint32_t nchunks,
                           float post, const unsigned long long* __restrict__ slots,
                           uint32_t epoch) {
  __shared__ float r_s[kMaxShards];
  const RedSq none = {nullptr, nullptr, 0.0f};
  encode_pass<IN, OUT, false, K>(descs, chunks, nchunks, K, post, slots, epoch,
                                 none, r_s, nullptr, nullptr);
}

// The encode pass with the exact squares (table roots: SqSum), in the
// general form and specialised on k = 1, 2, 4 or 8 (KS; 0: general).
template <int KS>
constexpr int reduce_sq_min_blocks() {
  return KS > 0 ? small_min_blocks<KS>() : FP8OPT_REDUCE_SQ_MIN_BLOCKS;
}

template <int IN, int OUT, int KS>
__global__ void __launch_bounds__(kThreads, reduce_sq_min_blocks<KS>())
reduce_encode_sq_kernel(const ReduceDesc* __restrict__ descs,
                        const Chunk* __restrict__ chunks, uint32_t nchunks, int k,
                        float post, const unsigned long long* __restrict__ slots,
                        uint32_t epoch, RedSq sq) {
  __shared__ float r_s[kMaxShards];
  __shared__ typename SqSum<OUT>::Table tab;
  __shared__ SqRed red;
  sq_table_fill_fmt<OUT>(tab);
  encode_pass<IN, OUT, true, KS>(descs, chunks, nchunks, KS > 0 ? KS : k, post,
                                 slots, epoch, sq, r_s, &tab, &red);
}

// Per-item norm terms of the reduced tensors (k = ils / the output scale);
// block 0 also exports found_inf.
__global__ void __launch_bounds__(kThreads)
reduce_terms_kernel(const ReduceDesc* __restrict__ descs, int n, float ils,
                    const unsigned long long* __restrict__ sums,
                    const unsigned long long* __restrict__ found, uint32_t epoch,
                    double* __restrict__ terms, uint32_t* __restrict__ found_out) {
  const int t = blockIdx.x * kThreads + threadIdx.x;
  if (t < n) {
    const U128 s = {sums[2 * t], sums[2 * t + 1]};
    terms[t] = norm_term(s, __fdiv_rn(ils, *descs[t].scale_out));
  }
  if (found_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *found_out = slot_value(*found, epoch) != 0 ? 1u : 0u;
}

template <int IN>
void launch_encode(uint32_t grid, const ReduceDesc* descs, const Chunk* chunks,
                   uint32_t nchunks, int k, float post,
                   const unsigned long long* slots, uint32_t epoch, int out_fmt,
                   const RedSq* sq, cudaStream_t stream) {
  if (sq == nullptr && (k == 1 || k == 2 || k == 4 || k == 8)) {
    const int v = (out_fmt == kE4M3 ? 0 : 4) | (k == 1 ? 0 : k == 2 ? 1 : k == 4 ? 2 : 3);
    switch (v) {
#define FP8OPT_ENCODE_SMALL_CASE(OUT, KI, K)                                 \
  case (OUT == kE4M3 ? 0 : 4) | KI:                                          \
    reduce_encode_small_kernel<IN, OUT, K><<<grid, kThreads, 0, stream>>>(   \
        descs, chunks, nchunks, post, slots, epoch);                         \
    break;
      FP8OPT_ENCODE_SMALL_CASE(kE4M3, 0, 1)
      FP8OPT_ENCODE_SMALL_CASE(kE4M3, 1, 2)
      FP8OPT_ENCODE_SMALL_CASE(kE4M3, 2, 4)
      FP8OPT_ENCODE_SMALL_CASE(kE4M3, 3, 8)
      FP8OPT_ENCODE_SMALL_CASE(kE5M2, 0, 1)
      FP8OPT_ENCODE_SMALL_CASE(kE5M2, 1, 2)
      FP8OPT_ENCODE_SMALL_CASE(kE5M2, 2, 4)
      FP8OPT_ENCODE_SMALL_CASE(kE5M2, 3, 8)
#undef FP8OPT_ENCODE_SMALL_CASE
    }
  } else if (sq == nullptr) {
    if (out_fmt == kE4M3)
      reduce_encode_kernel<IN, kE4M3><<<grid, kThreads, 0, stream>>>(
          descs, chunks, nchunks, k, post, slots, epoch);
    else
      reduce_encode_kernel<IN, kE5M2><<<grid, kThreads, 0, stream>>>(
          descs, chunks, nchunks, k, post, slots, epoch);
  } else {
    const int ki = k == 1 ? 1 : k == 2 ? 2 : k == 4 ? 3 : k == 8 ? 4 : 0;
    const int v = (out_fmt == kE4M3 ? 0 : 8) | ki;
    switch (v) {
#define FP8OPT_ENCODE_SQ_CASE(OUT, KI, KS)                                   \
  case (OUT == kE4M3 ? 0 : 8) | KI:                                          \
    reduce_encode_sq_kernel<IN, OUT, KS><<<grid, kThreads, 0, stream>>>(     \
        descs, chunks, nchunks, k, post, slots, epoch, *sq);                 \
    break;
      FP8OPT_ENCODE_SQ_CASE(kE4M3, 0, 0)
      FP8OPT_ENCODE_SQ_CASE(kE4M3, 1, 1)
      FP8OPT_ENCODE_SQ_CASE(kE4M3, 2, 2)
      FP8OPT_ENCODE_SQ_CASE(kE4M3, 3, 4)
      FP8OPT_ENCODE_SQ_CASE(kE4M3, 4, 8)
      FP8OPT_ENCODE_SQ_CASE(kE5M2, 0, 0)
      FP8OPT_ENCODE_SQ_CASE(kE5M2, 1, 1)
      FP8OPT_ENCODE_SQ_CASE(kE5M2, 2, 2)
      FP8OPT_ENCODE_SQ_CASE(kE5M2, 3, 4)
      FP8OPT_ENCODE_SQ_CASE(kE5M2, 4, 8)
#undef FP8OPT_ENCODE_SQ_CASE
    }
  }
}

}  // namespace

// Launches both passes on `stream`; 1 <= k <= kMaxShards.  With k in {1, 2,
// 4, 8} the grids are sized for the k-specialised kernels.  With norm set,
// the encode pass also sums the exact squares of the codes it writes into
// norm->sums (2n zeroed words; found_inf into norm->found), and a last kernel
// writes each item's norm term and the found flag.
cudaError_t launch_reduce(const ReduceDesc* descs, const Chunk* chunks,
                          uint32_t nchunks, unsigned long long* slots,
                          uint32_t epoch, int k, int in_fmt, int out_fmt,
                          float post, int grid_amax, int grid_encode,
                          const ReduceNorm* norm, cudaStream_t stream,
                          LaunchMark mark, int phase) {
  if (nchunks == 0) return cudaSuccess;
  const uint32_t ga = grid_min((uint32_t)grid_amax, nchunks);
  const uint32_t ge = grid_min((uint32_t)grid_encode, nchunks);
  if (phase & kReduceAmaxPass) {
    if (mark) mark(kReduceAmaxK, 0, stream);
    if (in_fmt == kE4M3)
      launch_amax<kE4M3>(ga, descs, chunks, nchunks, k, post, slots, epoch, stream);
    else
      launch_amax<kE5M2>(ga, descs, chunks, nchunks, k, post, slots, epoch, stream);
    if (mark) mark(kReduceAmaxK, 1, stream);
  }
  if (!(phase & kReduceEncodePass)) return cudaGetLastError();
  if (mark) mark(kReduceEncodeK, 0, stream);
  RedSq sq;
  if (norm != nullptr) sq = RedSq{norm->sums, norm->found, norm->ils};
  const RedSq* sqp = norm != nullptr ? &sq : nullptr;
  if (in_fmt == kE4M3)
    launch_encode<kE4M3>(ge, descs, chunks, nchunks, k, post, slots, epoch,
                         out_fmt, sqp, stream);
  else
    launch_encode<kE5M2>(ge, descs, chunks, nchunks, k, post, slots, epoch,
                         out_fmt, sqp, stream);
  if (mark) mark(kReduceEncodeK, 1, stream);
  if (norm != nullptr && norm->n > 0 && norm->limbs != nullptr) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_sums_to_limbs(norm->sums, norm->n, norm->found, epoch,
                                norm->limbs, norm->found_out, stream);
  }
  if (norm != nullptr && norm->n > 0) {
    if (mark) mark(kGradNormTermsK, 0, stream);
    reduce_terms_kernel<<<(norm->n + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
        descs, norm->n, norm->ils, norm->sums, norm->found, epoch, norm->terms,
        norm->found_out);
    if (mark) mark(kGradNormTermsK, 1, stream);
  }
  return cudaGetLastError();
}

// Resident CTAs per SM of the encode pass with squares: general (per_sm)
// and specialised on k for k <= 2, k = 4 and k = 8 (small_per_sm[3]).
cudaError_t reduce_encode_sq_occupancy(int* per_sm, int* small_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      per_sm, reduce_encode_sq_kernel<kE4M3, kE4M3, 0>, kThreads, 0);
  if (e != cudaSuccess) return e;
  const void* k[3] = {(const void*)reduce_encode_sq_kernel<kE4M3, kE4M3, 2>,
                      (const void*)reduce_encode_sq_kernel<kE4M3, kE4M3, 4>,
                      (const void*)reduce_encode_sq_kernel<kE4M3, kE4M3, 8>};
  for (int i = 0; i < 3; ++i) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&small_per_sm[i], k[i],
                                                      kThreads, 0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Resident CTAs per SM of the reduction kernels: the first and the encode
// pass in their general form, and in the forms specialised on k for k <= 2,
// k = 4 and k = 8 (amax_small and encode_small: three entries each).
cudaError_t reduce_occupancy(int* amax_per_sm, int* amax_small_per_sm,
                             int* encode_per_sm, int* encode_small_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      amax_per_sm, reduce_amax_kernel<kE4M3>, kThreads, 0);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      encode_per_sm, reduce_encode_kernel<kE4M3, kE4M3>, kThreads, 0);
  if (e != cudaSuccess) return e;
  const void* amax_k[3] = {(const void*)reduce_amax_small_kernel<kE4M3, 2>,
                           (const void*)reduce_amax_small_kernel<kE4M3, 4>,
                           (const void*)reduce_amax_small_kernel<kE4M3, 8>};
  const void* encode_k[3] = {(const void*)reduce_encode_small_kernel<kE4M3, kE4M3, 2>,
                             (const void*)reduce_encode_small_kernel<kE4M3, kE4M3, 4>,
                             (const void*)reduce_encode_small_kernel<kE4M3, kE4M3, 8>};
  for (int i = 0; i < 3; ++i) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&amax_small_per_sm[i],
                                                      amax_k[i], kThreads, 0);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&encode_small_per_sm[i],
                                                      encode_k[i], kThreads, 0);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace fp8opt
