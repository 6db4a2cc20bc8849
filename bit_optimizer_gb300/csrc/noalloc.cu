// fp8_cast_scaled_noalloc: the scaled FP8 cast for callers that must not
// allocate device memory.
//
// fp8_cast_scaled keeps its tensor table, chunk table and per-tensor amax
// slots in a workspace it allocates with cudaMalloc on first use.  Some
// callers cannot let a library do that: runtimes that hand all device memory
// to their own pool allocator at start-up and forbid other allocations, and
// services that must never stall on, or fail from, an allocation in the
// middle of a step.  For them this entry point runs the same two cast kernels
// with all of that scratch in one fixed-size array compiled into the library
// (`g_noalloc_scratch` below), so a call allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine, and no host heap either (the
// tables are staged in fixed host arrays).
//
// What that costs the caller:
//   * fixed limits: at most kMaxTensors tensors and kMaxChunks chunks of
//     32768 elements per call (2^31 elements in all); a call beyond either
//     limit returns FP8OPT_ERR_LIMIT and launches nothing;
//   * one copy of the array per device, held from the moment the library's
//     device code is loaded on that device until the process exits
//     (kScratchBytes, about 1.1 MB);
//   * every call, on every stream of a device, uses the same array, and it
//     keeps what the last call left there.  Each call clears the amax slots it
//     needs before its kernels run, but calls whose GPU work overlaps (two
//     streams, or two host threads) race on the array and can corrupt each
//     other's results: order such calls on one stream, or with events;
//   * each call copies its tables from host arrays that the next call
//     refills, so a stream that is capturing work into a CUDA graph is
//     refused (FP8OPT_ERR_ARG, nothing enqueued): a recorded copy would read
//     whatever a later call left in those arrays;
//   * the first call on each device does the set-up for that device (it asks
//     the runtime for the array's device address and the kernels' occupancy).
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fp8opt.h"
#include "fp8opt_internal.cuh"

namespace fp8opt {

cudaError_t launch_cast(const CastDesc* descs, const Chunk* chunks,
                        uint32_t nchunks, unsigned long long* slots,
                        uint32_t epoch, int fmt, int grid_amax,
                        int grid_encode, cudaStream_t stream, LaunchMark mark);
cudaError_t cast_occupancy(int* amax_per_sm, int* encode_per_sm);
int record_error(int status, const char* what);

namespace {

constexpr int kMaxTensors = FP8OPT_NOALLOC_MAX_TENSORS;
constexpr uint32_t kMaxChunks = FP8OPT_NOALLOC_MAX_CHUNKS;
constexpr int kMaxDevices = 64;

// Layout of the array: amax slots, then the tensor table, then the chunk table.
constexpr size_t kSlotsOffset = 0;
constexpr size_t kDescOffset = kMaxTensors * sizeof(unsigned long long);
constexpr size_t kChunkOffset = kDescOffset + kMaxTensors * sizeof(CastDesc);
constexpr size_t kScratchBytes = kChunkOffset + kMaxChunks * sizeof(Chunk);
static_assert(kDescOffset % 16 == 0 && kChunkOffset % 16 == 0, "layout");

// The whole scratch of the entry point.  In host code this name is only a
// handle for the runtime: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host staging of the tables (fixed arrays: no heap), guarded by g_mu.
CastDesc h_descs[kMaxTensors];
Chunk h_chunks[kMaxChunks];

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int grid_amax = 0, grid_encode = 0;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_mu;

int setup_device(int dev, DeviceSetup** out) {
  char msg[160];
  if (dev < 0 || dev >= kMaxDevices) {
    std::snprintf(msg, sizeof msg,
                  "fp8_cast_scaled_noalloc: device %d is beyond the %d this "
                  "entry point supports", dev, kMaxDevices);
    return record_error(FP8OPT_ERR_LIMIT, msg);
  }
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    int sms = 0, a = 0, b = 0;
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cast_occupancy(&a, &b);
    if (e != cudaSuccess) {
      std::snprintf(msg, sizeof msg, "fp8_cast_scaled_noalloc: set-up: %s: %s",
                    cudaGetErrorName(e), cudaGetErrorString(e));
      return record_error(FP8OPT_ERR_CUDA, msg);
    }
    s.scratch = static_cast<unsigned char*>(p);
    s.grid_amax = sms * (a > 0 ? a : 1);
    s.grid_encode = sms * (b > 0 ? b : 1);
    s.ready = true;
  }
  *out = &s;
  return FP8OPT_OK;
}

bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace
}  // namespace fp8opt

using namespace fp8opt;

extern "C" int fp8_cast_scaled_noalloc(const fp8opt_cast_item* items, int n,
                                       int fmt, void* stream_ptr) {
  char msg[200];
  if (n < 0 || (n > 0 && items == nullptr))
    return record_error(FP8OPT_ERR_ARG,
                        "fp8_cast_scaled_noalloc: n < 0 or items is NULL");
  if (fmt != FP8OPT_E4M3 && fmt != FP8OPT_E5M2)
    return record_error(FP8OPT_ERR_UNSUPPORTED,
                        "fp8_cast_scaled_noalloc: unknown format");
  if (n > kMaxTensors) {
    std::snprintf(msg, sizeof msg,
                  "fp8_cast_scaled_noalloc: %d tensors, above the maximum of %d",
                  n, kMaxTensors);
    return record_error(FP8OPT_ERR_LIMIT, msg);
  }
  uint64_t total_chunks = 0;
  for (int i = 0; i < n; ++i) {
    const fp8opt_cast_item& it = items[i];
    if (it.dtype != FP8OPT_F32 && it.dtype != FP8OPT_BF16 && it.dtype != FP8OPT_F16) {
      std::snprintf(msg, sizeof msg,
                    "fp8_cast_scaled_noalloc: item %d: unknown dtype", i);
      return record_error(FP8OPT_ERR_UNSUPPORTED, msg);
    }
    if (it.numel < 0 || it.reserved != 0 || it.amax == nullptr ||
        it.scale == nullptr ||
        (it.numel > 0 && (it.src == nullptr || it.codes == nullptr))) {
      std::snprintf(msg, sizeof msg,
                    "fp8_cast_scaled_noalloc: item %d: bad numel, reserved "
                    "field or NULL pointer", i);
      return record_error(FP8OPT_ERR_ARG, msg);
    }
    total_chunks += it.numel == 0 ? 1 : (uint64_t)((it.numel + kChunkElems - 1) / kChunkElems);
  }
  if (total_chunks > kMaxChunks) {
    std::snprintf(msg, sizeof msg,
                  "fp8_cast_scaled_noalloc: %llu chunks of %lld elements, above "
                  "the maximum of %u", (unsigned long long)total_chunks,
                  (long long)kChunkElems, kMaxChunks);
    return record_error(FP8OPT_ERR_LIMIT, msg);
  }
  if (n == 0) return FP8OPT_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess ||
      cap != cudaStreamCaptureStatusNone)
    return record_error(FP8OPT_ERR_ARG,
                        "fp8_cast_scaled_noalloc: the stream is capturing a "
                        "CUDA graph (or its capture state is unknown); the "
                        "call copies its tables from host arrays that the "
                        "next call refills, so it runs only uncaptured");

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return record_error(FP8OPT_ERR_CUDA, "fp8_cast_scaled_noalloc: cudaGetDevice failed");
  DeviceSetup* ds = nullptr;
  int st = setup_device(dev, &ds);
  if (st != FP8OPT_OK) return st;

  uint32_t nc = 0;
  for (int i = 0; i < n; ++i) {
    const fp8opt_cast_item& it = items[i];
    CastDesc& d = h_descs[i];
    d.src = it.src;
    d.codes = it.codes;
    d.amax_out = it.amax;
    d.scale_out = it.scale;
    d.numel = it.numel;
    d.dtype = it.dtype;
    d.vec_ok = aligned_to(it.src, 16) && aligned_to(it.codes, 8);
    const uint32_t chunks = it.numel == 0 ? 1u : (uint32_t)((it.numel + kChunkElems - 1) / kChunkElems);
    for (uint32_t c = 0; c < chunks; ++c)
      h_chunks[nc++] = make_chunk((uint32_t)i, c, kChunkShift, it.numel);
  }
  unsigned char* base = ds->scratch;
  unsigned long long* slots = reinterpret_cast<unsigned long long*>(base + kSlotsOffset);
  CastDesc* descs = reinterpret_cast<CastDesc*>(base + kDescOffset);
  Chunk* chunks = reinterpret_cast<Chunk*>(base + kChunkOffset);
  // The copies come from pageable host arrays, so each returns once its data
  // is staged and the arrays may be refilled by the next call.
  e = cudaMemcpyAsync(descs, h_descs, sizeof(CastDesc) * (size_t)n,
                      cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(chunks, h_chunks, sizeof(Chunk) * (size_t)nc,
                        cudaMemcpyHostToDevice, stream);
  // The slots must start at zero: the last call left its amax values there.
  if (e == cudaSuccess)
    e = cudaMemsetAsync(slots, 0, sizeof(unsigned long long) * (size_t)n, stream);
  if (e == cudaSuccess)
    e = launch_cast(descs, chunks, nc, slots, 1u, fmt, ds->grid_amax,
                    ds->grid_encode, stream, nullptr);
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof msg, "fp8_cast_scaled_noalloc: %s: %s",
                  cudaGetErrorName(e), cudaGetErrorString(e));
    return record_error(FP8OPT_ERR_CUDA, msg);
  }
  return FP8OPT_OK;
}
