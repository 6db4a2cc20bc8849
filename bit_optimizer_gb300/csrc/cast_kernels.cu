// Scaled FP8 cast of a tensor list (MS-AMP O1: weight gradients kept in FP8).
//
// Two persistent kernels over the chunk table:
//   cast_amax_kernel    per-tensor max |x| (on the fp32 bit patterns, so NaN
//                       orders above +inf above every finite value), reduced
//                       with warp max-reductions, a shared-memory CTA step,
//                       and one 64-bit atomicMax per (chunk, tensor).
//   cast_encode_kernel  scale = fp8_max / amax in each CTA's chunk prologue,
//                       then code = RNE-saturating encode of x * scale.  It
//                       walks the chunk table backwards, so the chunks the
//                       amax pass read last are still in L2 when it starts.
// Bytes per element: BF16/FP16 in: 2 (amax) + 2 + 1 (encode); FP32: 4 + 4 + 1.
#include "fp8opt_internal.cuh"

namespace fp8opt {

namespace {

// 8-element groups per thread per tile in the amax and encode passes (the
// latter without and with exact squares), and the resident CTAs per SM the
// encode pass with exact squares is compiled for.  Measured on the clipped
// 6.7B step: the encode pass with squares takes 3.47 ms with four groups at
// 4 CTAs/SM, against 3.95 with two.
#ifndef FP8OPT_ENC_GROUPS
#define FP8OPT_ENC_GROUPS 2
#endif
#ifndef FP8OPT_ENCSQ_GROUPS
#define FP8OPT_ENCSQ_GROUPS 4
#endif
#ifndef FP8OPT_ENCSQ_MIN_BLOCKS
#define FP8OPT_ENCSQ_MIN_BLOCKS 4
#endif
// The same for E5M2 codes, whose 128-bit sums take more registers, and
// whether their chunks go through the tile pipeline (1) or one tile at a
// time (0).
#ifndef FP8OPT_ENCSQ5_MIN_BLOCKS
#define FP8OPT_ENCSQ5_MIN_BLOCKS 3
#endif
#ifndef FP8OPT_ENCSQ5_TILES
#define FP8OPT_ENCSQ5_TILES 1
#endif
constexpr int kAmaxGroups = 4;

// Tiles ahead of the current one the encode pass prefetches into L2 (0:
// none).  Measured: no gain for this pass or for the read-only amax pass.
#ifndef FP8OPT_ENC_PREFETCH
#define FP8OPT_ENC_PREFETCH 0
#endif

// ---------------------------------------------------------------- amax pass

// Max of |x| bit patterns over the four words of a uint4 of 16-bit values,
// accumulated per 16-bit lane.
__device__ __forceinline__ uint32_t vmax16x8(uint32_t acc, uint4 a) {
  acc = __vmaxu2(acc, a.x & 0x7FFF7FFFu);
  acc = __vmaxu2(acc, a.y & 0x7FFF7FFFu);
  acc = __vmaxu2(acc, a.z & 0x7FFF7FFFu);
  return __vmaxu2(acc, a.w & 0x7FFF7FFFu);
}

__device__ __forceinline__ uint32_t vmax32x4(uint32_t acc, uint4 a) {
  acc = max(acc, a.x & 0x7FFFFFFFu);
  acc = max(acc, a.y & 0x7FFFFFFFu);
  acc = max(acc, a.z & 0x7FFFFFFFu);
  return max(acc, a.w & 0x7FFFFFFFu);
}

// This thread's share of max |x| over [begin, end), as an fp32 bit pattern
// (not yet NaN-canonical).  For 16-bit types the running maximum is kept per
// 16-bit lane of a 32-bit word and widened at the end; the order of
// non-negative bit patterns is the order of their values in all three types.
template <int DT>
__device__ uint32_t thread_amax(const void* src, int64_t begin, int64_t end,
                                bool vec) {
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kAmaxGroups;
  const int tid = threadIdx.x;
  uint32_t acc = 0;
  for (int64_t base = begin; base < end; base += kTile) {
    if (vec && base + kTile <= end) {
      if (DT == kF32) {
        const float* f = static_cast<const float*>(src);
        uint4 a[kAmaxGroups][2];
#pragma unroll
        for (int k = 0; k < kAmaxGroups; ++k) {
          const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
          a[k][0] = ld_keep4(f + i0);
          a[k][1] = ld_keep4(f + i0 + 4);
        }
#pragma unroll
        for (int k = 0; k < kAmaxGroups; ++k)
          acc = vmax32x4(vmax32x4(acc, a[k][0]), a[k][1]);
      } else {
        const uint16_t* h = static_cast<const uint16_t*>(src);
        uint4 a[kAmaxGroups];
#pragma unroll
        for (int k = 0; k < kAmaxGroups; ++k)
          a[k] = ld_keep4(h + base + k * (kThreads * kGroup) + tid * kGroup);
#pragma unroll
        for (int k = 0; k < kAmaxGroups; ++k) acc = vmax16x8(acc, a[k]);
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < kAmaxGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        for (int j = 0; j < kGroup; ++j) {
          const int64_t i = i0 + j;
          if (i >= end) break;
          if (DT == kF32) {
            acc = max(acc, __float_as_uint(static_cast<const float*>(src)[i]) &
                               0x7FFFFFFFu);
          } else {
            const uint32_t b = static_cast<const uint16_t*>(src)[i] & 0x7FFFu;
            acc = __vmaxu2(acc, b);
          }
        }
      }
    }
  }
  if (DT == kF32) return acc;
  const uint32_t h = max(acc & 0xFFFFu, acc >> 16);
  if (DT == kBF16) return h << 16;
  if (h > 0x7C00u) return 0x7FC00000u;                 // FP16 NaN
  return __float_as_uint(h_to_f((uint16_t)h));          // exact widening
}

__global__ void __launch_bounds__(kThreads)
cast_amax_kernel(const CastDesc* __restrict__ descs,
                 const Chunk* __restrict__ chunks, uint32_t nchunks,
                 unsigned long long* __restrict__ slots, uint32_t epoch) {
  __shared__ uint32_t red[kThreads / 32];
  for (uint32_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const CastDesc d = descs[ch.tensor];
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    const bool vec = d.vec_ok != 0;
    uint32_t mx;
    if (d.dtype == kF32)
      mx = thread_amax<kF32>(d.src, begin, end, vec);
    else if (d.dtype == kBF16)
      mx = thread_amax<kBF16>(d.src, begin, end, vec);
    else
      mx = thread_amax<kF16>(d.src, begin, end, vec);
    mx = block_max_u32(mx, red);
    if (threadIdx.x == 0 && mx != 0)
      atomicMax(&slots[ch.tensor], slot_tag(epoch, canon_amax_bits(mx)));
  }
}

// -------------------------------------------------------------- encode pass

// Where an encode pass also sums the exact squares of the codes it writes
// (the gradient norm of a clipped step): the tensors' 128-bit slots, the
// found_inf slot, and the step's inverse loss scale.
struct SqOut {
  unsigned long long* sums;
  unsigned long long* found;
  float ils;
  const float* ils_dev;   // inv_loss_scale in device memory instead, or NULL
};

// Encode this thread's share of [begin, end).  CHECKED when the tensor holds a
// non-finite element (its amax is not finite): those take the explicit
// NaN / infinity codes; otherwise every product is finite.  SQ: also add the
// exact squares of the codes written to acc (through the table tab) and
// collect in bad the codes at or above the overflow threshold whose addend
// is tadd (found_inf of a step with factor inv_loss_scale / scale).
template <int DT, int FMT, bool CHECKED, bool SQ>
__device__ void thread_encode(const void* src, uint8_t* codes, int64_t begin,
                              int64_t end, bool vec, float scale,
                              uint32_t tadd, SqSum<FMT>& acc,
                              uint32_t& bad) {
  constexpr int kEncGroups = SQ ? FP8OPT_ENCSQ_GROUPS : FP8OPT_ENC_GROUPS;
  constexpr int64_t kTile = (int64_t)kThreads * kGroup * kEncGroups;
  constexpr uint32_t kSrcBytes = DT == kF32 ? 4 : 2;
  const int tid = threadIdx.x;
  const bool pf = FP8OPT_ENC_PREFETCH > 0 && tid == 0 && vec && aligned16(src);
  for (int64_t base = begin; base < end; base += kTile) {
    if (pf) {
      const int64_t ahead = base + FP8OPT_ENC_PREFETCH * kTile;
      if (ahead + kTile <= end)
        prefetch_l2(static_cast<const char*>(src) + ahead * kSrcBytes,
                    (uint32_t)(kSrcBytes * kTile));
    }
    if (vec && base + kTile <= end) {
      float x[kEncGroups][8];
#pragma unroll
      for (int k = 0; k < kEncGroups; ++k)
        load8<DT>(src, base + k * (kThreads * kGroup) + tid * kGroup, x[k]);
#pragma unroll
      for (int k = 0; k < kEncGroups; ++k) {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[k][j] = __fmul_rn(x[k][j], scale);
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        const uint2 c = enc8<FMT, CHECKED>(x[k]);
        *reinterpret_cast<uint2*>(codes + i0) = c;
        if (SQ) {
          const uint32_t a = c.x & 0x7F7F7F7Fu, b = c.y & 0x7F7F7F7Fu;
          bad |= ((a + tadd) | (b + tadd)) & 0x80808080u;
          acc.add_word(a);
          acc.add_word(b);
        }
      }
    } else {
#pragma unroll 1
      for (int k = 0; k < kEncGroups; ++k) {
        const int64_t i0 = base + k * (kThreads * kGroup) + tid * kGroup;
        if (vec && i0 + kGroup <= end) {
          float x[8];
          load8<DT>(src, i0, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(x[j], scale);
          const uint2 c = enc8<FMT, CHECKED>(x);
          *reinterpret_cast<uint2*>(codes + i0) = c;
          if (SQ) {
            const uint32_t a = c.x & 0x7F7F7F7Fu, b = c.y & 0x7F7F7F7Fu;
            bad |= ((a + tadd) | (b + tadd)) & 0x80808080u;
            acc.add_word(a);
            acc.add_word(b);
          }
        } else {
          for (int j = 0; j < kGroup; ++j) {
            const int64_t i = i0 + j;
            if (i >= end) break;
            const float t = __fmul_rn(load1<DT>(src, i), scale);
            const uint32_t c = CHECKED ? enc1_checked<FMT>(t)
                                       : (enc2<FMT>(t, 0.0f) & 0xFFu);
            codes[i] = (uint8_t)c;
            if (SQ) {
              bad |= ((c & 0x7Fu) + tadd) & 0x80u;
              acc.add_word(c & 0x7Fu);
            }
          }
        }
      }
    }
  }
}

template <int DT, int FMT, bool SQ>
__device__ __forceinline__ void encode_dispatch(const CastDesc& d,
                                                int64_t begin, int64_t end,
                                                float scale, bool checked,
                                                uint32_t tadd, SqSum<FMT>& acc,
                                                uint32_t& bad) {
  const bool vec = d.vec_ok != 0;
  if (checked)
    thread_encode<DT, FMT, true, SQ>(d.src, d.codes, begin, end, vec, scale,
                                     tadd, acc, bad);
  else
    thread_encode<DT, FMT, false, SQ>(d.src, d.codes, begin, end, vec, scale,
                                      tadd, acc, bad);
}

// One chunk-strided encode pass.
template <int FMT>
__device__ __forceinline__ void encode_pass(const CastDesc* __restrict__ descs,
                                            const Chunk* __restrict__ chunks,
                                            uint32_t nchunks,
                                            const unsigned long long* __restrict__ slots,
                                            uint32_t epoch) {
  SqSum<FMT> acc(nullptr);   // unused without squares
  uint32_t bad = 0;
  for (uint32_t r = blockIdx.x; r < nchunks; r += gridDim.x) {
    const Chunk ch = chunks[nchunks - 1 - r];
    const CastDesc d = descs[ch.tensor];
    const uint32_t ab = slot_value(slots[ch.tensor], epoch);
    const float scale = scale_from_amax_bits(ab, fp8_max_of<FMT>());
    if (ch.begin == 0 && threadIdx.x == 0) {
      *d.amax_out = __uint_as_float(ab);
      *d.scale_out = scale;
    }
    const int64_t begin = ch.begin;
    const int64_t end = begin + ch.len;
    const bool checked = ab >= 0x7F800000u;
    if (d.dtype == kF32)
      encode_dispatch<kF32, FMT, false>(d, begin, end, scale, checked, 0, acc, bad);
    else if (d.dtype == kBF16)
      encode_dispatch<kBF16, FMT, false>(d, begin, end, scale, checked, 0, acc, bad);
    else
      encode_dispatch<kF16, FMT, false>(d, begin, end, scale, checked, 0, acc, bad);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads)
cast_encode_kernel(const CastDesc* __restrict__ descs,
                   const Chunk* __restrict__ chunks, uint32_t nchunks,
                   const unsigned long long* __restrict__ slots,
                   uint32_t epoch) {
  encode_pass<FMT>(descs, chunks, nchunks, slots, epoch);
}

// ------------------------------------ encode pass with the exact squares
//
// A full chunk of 16-bit elements (kChunkElems of them, vector loads, a
// finite amax) is encoded as four tiles of kEncSqGroups 8-element groups per
// thread, each tile's loads issued one tile ahead of its arithmetic (the
// next chunk's first tile while this chunk's last is encoded), so that a
// thread always has a tile in flight.  Other chunks take thread_encode.  The
// E5M2 instance runs fewer CTAs per SM: its 128-bit sums leave too few
// registers for two tiles in flight at four.  A CTA's exact sum goes to its
// tensor's slot when the next chunk it takes belongs to another tensor.
constexpr int kEncSqGroups = FP8OPT_ENCSQ_GROUPS;
constexpr int64_t kEncSqTile = (int64_t)kThreads * kGroup * kEncSqGroups;
static_assert(kChunkElems % kEncSqTile == 0 && kChunkElems / kEncSqTile == 4,
              "a full chunk is four tiles");

struct EncTile {
  uint4 h[kEncSqGroups];   // 8 16-bit elements per group
};

__device__ __forceinline__ void load_enc_tile(EncTile& t, const uint16_t* p) {
#pragma unroll
  for (int q = 0; q < kEncSqGroups; ++q)
    t.h[q] = ld_once4(p + q * (kThreads * kGroup) + threadIdx.x * kGroup);
}

// Encodes a loaded tile (16-bit type DT, finite scale products) to codes at
// c (the tile's first code), adding the exact squares to acc and the codes
// at or above the overflow threshold (addend tadd) to bad.
template <int DT, int FMT>
__device__ __forceinline__ void enc_tile(const EncTile& t, uint8_t* c,
                                         float scale, uint32_t tadd,
                                         SqSum<FMT>& acc,
                                         uint32_t& bad) {
#pragma unroll
  for (int q = 0; q < kEncSqGroups; ++q) {
    float x[8];
    if (DT == kF16) {
      h8_to_f(t.h[q], x);
    } else {
      const uint32_t w[4] = {t.h[q].x, t.h[q].y, t.h[q].z, t.h[q].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[2 * j] = __uint_as_float(w[j] << 16);
        x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = __fmul_rn(x[j], scale);
    const uint2 code = enc8<FMT, false>(x);
    *reinterpret_cast<uint2*>(c + q * (kThreads * kGroup) + threadIdx.x * kGroup) = code;
    const uint32_t a = code.x & 0x7F7F7F7Fu, b = code.y & 0x7F7F7F7Fu;
    bad |= ((a + tadd) | (b + tadd)) & 0x80808080u;
    acc.add_word(a);
    acc.add_word(b);
  }
}

template <int FMT>
__device__ __forceinline__ void enc_tile_dt(const EncTile& t, int dtype,
                                            uint8_t* c, float scale,
                                            uint32_t tadd, SqSum<FMT>& acc,
                                            uint32_t& bad) {
  if (dtype == kF16)
    enc_tile<kF16, FMT>(t, c, scale, tadd, acc, bad);
  else
    enc_tile<kBF16, FMT>(t, c, scale, tadd, acc, bad);
}

// What the pass needs of a chunk, its tensor and the tensor's amax.
struct EncChunk {
  const void* src;
  uint8_t* codes;
  float* amax_out;
  float* scale_out;
  int64_t begin;
  uint32_t len, tensor, ab;
  int dtype;
  bool vec;

  // encoded by the tile pipeline
  __device__ __forceinline__ bool tiled() const {
    return vec && dtype != kF32 && len == (uint32_t)kChunkElems &&
           ab < 0x7F800000u;
  }
  __device__ __forceinline__ const uint16_t* tile(int i) const {
    return static_cast<const uint16_t*>(src) + begin + i * kEncSqTile;
  }
};

__device__ __forceinline__ EncChunk enc_chunk(const CastDesc* descs,
                                              const Chunk* chunks, uint32_t c,
                                              const unsigned long long* slots,
                                              uint32_t epoch) {
  const Chunk ch = chunks[c];
  const CastDesc& d = descs[ch.tensor];
  EncChunk r;
  r.src = d.src;
  r.codes = d.codes;
  r.amax_out = d.amax_out;
  r.scale_out = d.scale_out;
  r.begin = ch.begin;
  r.len = ch.len;
  r.tensor = ch.tensor;
  r.ab = slot_value(slots[ch.tensor], epoch);
  r.dtype = d.dtype;
  r.vec = d.vec_ok != 0;
  return r;
}

// The encode pass with the exact squares through the shared-memory table of
// the integer square roots (SqSum<FMT>: SqTable for E4M3, Sq5Table for
// E5M2).  It walks the chunk table backwards in CTA strides, as the plain
// encode pass does; chunks of one tensor are adjacent in the table, so a
// tensor's chunks reach a CTA as one run.
template <int FMT>
constexpr int encsq_min_blocks() {
  return FMT == kE4M3 ? FP8OPT_ENCSQ_MIN_BLOCKS : FP8OPT_ENCSQ5_MIN_BLOCKS;
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, encsq_min_blocks<FMT>())
cast_encode_sq_kernel(const CastDesc* __restrict__ descs,
                      const Chunk* __restrict__ chunks, uint32_t nchunks,
                      const unsigned long long* __restrict__ slots,
                      uint32_t epoch, SqOut sq) {
  __shared__ typename SqSum<FMT>::Table tab;
  __shared__ SqRed red;
  if (blockIdx.x >= nchunks) return;   // uniform over the CTA
  const float ils = sq.ils_dev != nullptr ? *sq.ils_dev : sq.ils;
  constexpr bool kTiles = FMT == kE4M3 || FP8OPT_ENCSQ5_TILES != 0;
  uint32_t r = blockIdx.x;
  EncChunk cur = enc_chunk(descs, chunks, nchunks - 1 - r, slots, epoch);
  EncTile ta, tb;   // ta holds the current chunk's first tile if tiled
  if (kTiles && cur.tiled()) load_enc_tile(ta, cur.tile(0));
  sq_table_fill_fmt<FMT>(tab);
  SqSum<FMT> acc(&tab);
  uint32_t bad = 0, tadd = 0, tensor = 0xFFFFFFFFu, turn = 0;
  bool nonempty = false;
  float scale = 1.0f;
  for (; r < nchunks; r += gridDim.x) {
    const bool more = r + gridDim.x < nchunks;
    EncChunk nxt = cur;
    if (more) nxt = enc_chunk(descs, chunks, nchunks - 1 - (r + gridDim.x), slots, epoch);
    if (cur.tensor != tensor) {   // uniform over the CTA
      if (tensor != 0xFFFFFFFFu) {
        sq_commit(acc.sum(), bad, tensor, nonempty, sq.sums, sq.found, epoch, red,
                  turn);
        acc.clear();
        bad = 0;
        nonempty = false;
      }
      tensor = cur.tensor;
      scale = scale_from_amax_bits(cur.ab, fp8_max_of<FMT>());
      // found_inf as the step decides it, from its factor
      tadd = threshold_addend(overflow_threshold<FMT>(__fdiv_rn(ils, scale)));
    }
    if (cur.begin == 0 && threadIdx.x == 0) {
      *cur.amax_out = __uint_as_float(cur.ab);
      *cur.scale_out = scale;
    }
    nonempty |= cur.len > 0;
    const bool next_tiled = kTiles && more && nxt.tiled();
    if (kTiles && cur.tiled()) {
      uint8_t* c = cur.codes + cur.begin;
      load_enc_tile(tb, cur.tile(1));
      enc_tile_dt<FMT>(ta, cur.dtype, c, scale, tadd, acc, bad);
      load_enc_tile(ta, cur.tile(2));
      enc_tile_dt<FMT>(tb, cur.dtype, c + kEncSqTile, scale, tadd, acc, bad);
      load_enc_tile(tb, cur.tile(3));
      enc_tile_dt<FMT>(ta, cur.dtype, c + 2 * kEncSqTile, scale, tadd, acc, bad);
      if (next_tiled) load_enc_tile(ta, nxt.tile(0));
      enc_tile_dt<FMT>(tb, cur.dtype, c + 3 * kEncSqTile, scale, tadd, acc, bad);
    } else {
      if (next_tiled) load_enc_tile(ta, nxt.tile(0));
      const CastDesc d = descs[cur.tensor];
      const int64_t end = cur.begin + cur.len;
      const bool checked = cur.ab >= 0x7F800000u;
      if (d.dtype == kF32)
        encode_dispatch<kF32, FMT, true>(d, cur.begin, end, scale, checked,
                                         tadd, acc, bad);
      else if (d.dtype == kBF16)
        encode_dispatch<kBF16, FMT, true>(d, cur.begin, end, scale, checked,
                                          tadd, acc, bad);
      else
        encode_dispatch<kF16, FMT, true>(d, cur.begin, end, scale, checked,
                                         tadd, acc, bad);
    }
    cur = nxt;
  }
  sq_commit(acc.sum(), bad, tensor, nonempty, sq.sums, sq.found, epoch, red, turn);
}

}  // namespace

// Launches both passes on `stream`; grid is the persistent CTA count.
cudaError_t launch_cast(const CastDesc* descs, const Chunk* chunks,
                        uint32_t nchunks, unsigned long long* slots,
                        uint32_t epoch, int fmt, int grid_amax,
                        int grid_encode, cudaStream_t stream, LaunchMark mark) {
  if (nchunks == 0) return cudaSuccess;
  const uint32_t ga = grid_min((uint32_t)grid_amax, nchunks);
  const uint32_t ge = grid_min((uint32_t)grid_encode, nchunks);
  if (mark) mark(kCastAmaxK, 0, stream);
  cast_amax_kernel<<<ga, kThreads, 0, stream>>>(descs, chunks, nchunks, slots,
                                                epoch);
  if (mark) mark(kCastAmaxK, 1, stream);
  if (mark) mark(kCastEncodeK, 0, stream);
  if (fmt == kE4M3)
    cast_encode_kernel<kE4M3><<<ge, kThreads, 0, stream>>>(descs, chunks,
                                                           nchunks, slots, epoch);
  else
    cast_encode_kernel<kE5M2><<<ge, kThreads, 0, stream>>>(descs, chunks,
                                                           nchunks, slots, epoch);
  if (mark) mark(kCastEncodeK, 1, stream);
  return cudaGetLastError();
}

// The encode pass alone (after launch_cast_amax).
cudaError_t launch_cast_encode(const CastDesc* descs, const Chunk* chunks,
                               uint32_t nchunks, const unsigned long long* slots,
                               uint32_t epoch, int fmt, int grid_encode,
                               cudaStream_t stream, LaunchMark mark) {
  if (nchunks == 0) return cudaSuccess;
  const uint32_t ge = grid_min((uint32_t)grid_encode, nchunks);
  if (mark) mark(kCastEncodeK, 0, stream);
  if (fmt == kE4M3)
    cast_encode_kernel<kE4M3><<<ge, kThreads, 0, stream>>>(descs, chunks,
                                                           nchunks, slots, epoch);
  else
    cast_encode_kernel<kE5M2><<<ge, kThreads, 0, stream>>>(descs, chunks,
                                                           nchunks, slots, epoch);
  if (mark) mark(kCastEncodeK, 1, stream);
  return cudaGetLastError();
}

// The encode pass alone (after launch_cast_amax), also summing the exact
// squares of the codes it writes into sums (2n zeroed words) and setting the
// found_inf slot `found` as a step with factor inv_loss_scale / scale would
// (inv_loss_scale read from ils_dev on the device when that is set).
cudaError_t launch_cast_encode_sq(const CastDesc* descs, const Chunk* chunks,
                                  uint32_t nchunks, const unsigned long long* slots,
                                  uint32_t epoch, int fmt, int grid_encode,
                                  unsigned long long* sums,
                                  unsigned long long* found, float ils,
                                  const float* ils_dev, cudaStream_t stream,
                                  LaunchMark mark) {
  if (nchunks == 0) return cudaSuccess;
  const uint32_t ge = grid_min((uint32_t)grid_encode, nchunks);
  const SqOut sq = {sums, found, ils, ils_dev};
  if (mark) mark(kCastEncodeK, 0, stream);
  if (fmt == kE4M3)
    cast_encode_sq_kernel<kE4M3><<<ge, kThreads, 0, stream>>>(
        descs, chunks, nchunks, slots, epoch, sq);
  else
    cast_encode_sq_kernel<kE5M2><<<ge, kThreads, 0, stream>>>(
        descs, chunks, nchunks, slots, epoch, sq);
  if (mark) mark(kCastEncodeK, 1, stream);
  return cudaGetLastError();
}

// The amax pass alone (the fused cast + step path runs its own encode pass).
cudaError_t launch_cast_amax(const CastDesc* descs, const Chunk* chunks,
                             uint32_t nchunks, unsigned long long* slots,
                             uint32_t epoch, int grid_amax, cudaStream_t stream,
                             LaunchMark mark) {
  if (nchunks == 0) return cudaSuccess;
  if (mark) mark(kCastAmaxK, 0, stream);
  cast_amax_kernel<<<grid_min((uint32_t)grid_amax, nchunks), kThreads, 0,
                     stream>>>(descs, chunks, nchunks, slots, epoch);
  if (mark) mark(kCastAmaxK, 1, stream);
  return cudaGetLastError();
}

// Resident CTAs per SM of each cast kernel (for persistent grid sizing).
cudaError_t cast_occupancy(int* amax_per_sm, int* encode_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      amax_per_sm, cast_amax_kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      encode_per_sm, cast_encode_kernel<kE4M3>, kThreads, 0);
}

// per_sm[f]: for codes of format f.
cudaError_t cast_encode_sq_occupancy(int* per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm[kE4M3], cast_encode_sq_kernel<kE4M3>, kThreads, 0);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm[kE5M2], cast_encode_sq_kernel<kE5M2>, kThreads, 0);
}

}  // namespace fp8opt
