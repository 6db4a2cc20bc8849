// The libfp8opt C ABI (include/fp8opt.h): argument checks, the per-(device,
// stream) workspace with its cached tensor and chunk tables, the per-call
// scalars, and the kernel launches.
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fp8opt.h"
#include "fp8opt_internal.cuh"

namespace fp8opt {

cudaError_t launch_cast(const CastDesc* descs, const Chunk* chunks,
                        uint32_t nchunks, unsigned long long* slots,
                        uint32_t epoch, int fmt, int grid_amax,
                        int grid_encode, cudaStream_t stream, LaunchMark mark);
cudaError_t cast_occupancy(int* amax_per_sm, int* encode_per_sm);
cudaError_t launch_step(const StepDesc* descs, const Chunk* chunks,
                        uint32_t nchunks, const Chunk* chunks_o3,
                        uint32_t nchunks_o3, const StepScratch& sc,
                        const StepScalars& s, uint32_t epoch,
                        uint32_t* found_dev, int grid_amax, int grid_update,
                        int grid_update_var, int grid_w8, bool any_vs,
                        cudaStream_t stream, LaunchMark mark);
cudaError_t step_occupancy(int* amax_per_sm, int* update_per_sm,
                           int* update_var_per_sm, int* w8_per_sm);
cudaError_t launch_step_scalars(DevState* state, float beta1, float beta2,
                                float wd, bool l2, DevScalars* out, bool commit,
                                cudaStream_t stream);
cudaError_t launch_cast_amax(const CastDesc* descs, const Chunk* chunks,
                             uint32_t nchunks, unsigned long long* slots,
                             uint32_t epoch, int grid_amax, cudaStream_t stream,
                             LaunchMark mark);
cudaError_t launch_cast_encode_sq(const CastDesc* descs, const Chunk* chunks,
                                  uint32_t nchunks, const unsigned long long* slots,
                                  uint32_t epoch, int fmt, int grid_encode,
                                  unsigned long long* sums,
                                  unsigned long long* found, float ils,
                                  const float* ils_dev, cudaStream_t stream,
                                  LaunchMark mark);
cudaError_t cast_encode_sq_occupancy(int* per_sm);   // per_sm[2], per format
cudaError_t launch_cast_encode(const CastDesc* descs, const Chunk* chunks,
                               uint32_t nchunks, const unsigned long long* slots,
                               uint32_t epoch, int fmt, int grid_encode,
                               cudaStream_t stream, LaunchMark mark);
cudaError_t launch_cast_step(const CastDesc* cdescs, const StepDesc* sdescs,
                             const Chunk* chunks, uint32_t nchunks,
                             const Chunk* chunks_o3, uint32_t nchunks_o3,
                             unsigned long long* gslots, const StepScratch& sc,
                             const StepScalars& s, uint32_t epoch, int fmt,
                             uint32_t* found_dev, int grid_amax, int grid_fused,
                             int grid_update, int grid_update_var, int grid_w8,
                             bool any_vs, cudaStream_t stream, LaunchMark mark);
cudaError_t cast_step_occupancy(int* per_sm);
cudaError_t launch_reduce(const ReduceDesc* descs, const Chunk* chunks,
                          uint32_t nchunks, unsigned long long* slots,
                          uint32_t epoch, int k, int in_fmt, int out_fmt,
                          float post, int grid_amax, int grid_encode,
                          const ReduceNorm* norm, cudaStream_t stream,
                          LaunchMark mark, int phase);
cudaError_t launch_slots_export(const unsigned long long* slots, uint32_t epoch,
                                int n, uint32_t* out, cudaStream_t stream);
cudaError_t launch_slots_import(unsigned long long* slots, uint32_t epoch, int n,
                                const uint32_t* in, cudaStream_t stream);
cudaError_t launch_limbs_terms(const long long* limbs, const uint32_t* amax_bits,
                               int n, int fmt, float ils, double* terms,
                               cudaStream_t stream);
cudaError_t launch_step_w8(const StepDesc* descs, const Chunk* chunks_o3,
                           uint32_t nchunks_o3, const StepScratch& sc,
                           uint32_t epoch, int grid_w8, cudaStream_t stream,
                           LaunchMark mark);
cudaError_t reduce_occupancy(int* amax_per_sm, int* amax_small_per_sm,
                             int* encode_per_sm, int* encode_small_per_sm);
cudaError_t reduce_encode_sq_occupancy(int* per_sm, int* small_per_sm);
cudaError_t launch_grad_norm_terms(const StepDesc* descs, const Chunk* chunks,
                                   uint32_t nchunks, int n, float ils,
                                   const float* ils_dev,
                                   unsigned long long* sums,
                                   unsigned long long* found, uint32_t epoch,
                                   double* terms, uint32_t* found_out, int grid,
                                   int fmts, cudaStream_t stream, LaunchMark mark);
cudaError_t launch_norm_finish(const StepDesc* descs, int n, float ils,
                               const float* ils_dev,
                               const unsigned long long* sums,
                               const unsigned long long* found_slot,
                               uint32_t epoch, double* terms, float max_norm,
                               double* norm_out, float* clip_out,
                               float* user_norm, cudaStream_t stream,
                               LaunchMark mark);
cudaError_t launch_clip_coef(const double* terms, int n,
                             const unsigned long long* found_slot, uint32_t epoch,
                             const uint32_t* found_flag, float max_norm,
                             double* norm_out, float* clip_out, float* user_norm,
                             cudaStream_t stream, LaunchMark mark);
cudaError_t launch_found(unsigned long long* slot, uint32_t epoch,
                         const uint32_t* in, uint32_t* out, cudaStream_t stream,
                         LaunchMark mark);
cudaError_t launch_step_amax(const StepDesc* descs, const Chunk* chunks,
                             uint32_t nchunks, const StepScratch& sc,
                             const StepScalars& s, uint32_t epoch, int grid_amax,
                             cudaStream_t stream, LaunchMark mark);
cudaError_t launch_step_update(const StepDesc* descs, const Chunk* chunks,
                               uint32_t nchunks, const Chunk* chunks_o3,
                               uint32_t nchunks_o3, const StepScratch& sc,
                               const StepScalars& s, uint32_t epoch,
                               uint32_t* found_dev, int grid_update,
                               int grid_update_var, int grid_w8, bool any_vs,
                               cudaStream_t stream, LaunchMark mark);
cudaError_t grad_norm_occupancy(int* per_sm);

namespace {

thread_local std::string t_last_error;

int fail(int status, const std::string& what) {
  t_last_error = what;
  return status;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(FP8OPT_ERR_CUDA,
              std::string(where) + ": " + cudaGetErrorName(e) + ": " +
                  cudaGetErrorString(e));
}

// A device buffer that only grows, and not at all once frozen (a captured
// CUDA graph holds its address).
struct DevBuf {
  void* ptr = nullptr;
  size_t cap = 0;
  bool frozen = false;
  cudaError_t reserve(size_t bytes) {
    if (bytes <= cap) return cudaSuccess;
    if (frozen) return cudaErrorNotPermitted;
    if (ptr != nullptr) {
      cudaError_t e = cudaFree(ptr);
      if (e != cudaSuccess) return e;
      ptr = nullptr;
      cap = 0;
    }
    size_t want = bytes < 4096 ? 4096 : bytes + bytes / 4;
    cudaError_t e = cudaMalloc(&ptr, want);
    if (e != cudaSuccess) return e;
    cap = want;
    return cudaSuccess;
  }
  void release() {
    if (ptr != nullptr) cudaFree(ptr);
    ptr = nullptr;
    cap = 0;
  }
};

struct DeviceInfo {
  int sms = 0;
  int cast_amax = 0, cast_encode = 0;          // persistent grid sizes
  int step_amax = 0, step_update = 0, step_update_var = 0, step_w8 = 0;
  int cast_step = 0;
  int reduce_amax = 0, reduce_encode = 0;
  // the k-specialised passes, for k <= 2, k = 4 and k = 8
  int reduce_amax_small[3] = {0, 0, 0}, reduce_encode_small[3] = {0, 0, 0};
  int grad_norm = 0;
  int cast_encode_sq[2] = {0, 0};   // per code format
  int reduce_encode_sq = 0, reduce_encode_sq_small[3] = {0, 0, 0};
};

// Per-(device, stream) state.  The slot region holds only epoch-tagged
// uint64 words: [0, n) per-tensor amax A, [n, 2n) per-tensor amax B, [2n]
// found_inf (a call with another n lays them out differently, which is safe
// because every word carries an older epoch).  Untagged scratch (the saved
// first-moment scales) lives in its own buffer, so it can never be read as a
// tag.
struct Workspace {
  int device = 0;
  uint32_t epoch = 0;
  DevBuf slots;
  DevBuf saved_scales;       // n floats: m_scale before the step
  DevBuf norm_buf;           // gradient norm: 2n sum words, norm, clip
  DevBuf dev_scalars;        // the *_dev calls' DevScalars
  // cast tables
  std::vector<fp8opt_cast_item> cast_key;
  DevBuf cast_descs, cast_chunks;
  uint32_t cast_nchunks = 0;
  // step tables
  std::vector<fp8opt_param> step_key;
  DevBuf step_descs, step_chunks;
  uint32_t step_nchunks = 0, step_nchunks_o3 = 0;
  bool step_any_vs = false;   // some record has a scaled second moment
  int step_fmts = 0;          // bit f: some record has gradient codes of format f
  uint32_t begin_epoch = 0;   // epoch of an fp8_adam_step_begin awaiting its finish
  uint32_t copy_epoch = 0;    // epoch of a finish awaiting its fp8_adam_step_copy
  // reduction tables
  std::vector<fp8opt_reduce_item> reduce_key;
  DevBuf reduce_descs, reduce_chunks;
  uint32_t reduce_nchunks = 0;
  bool have_cast = false, have_step = false, have_reduce = false;
  // A CUDA graph captured on this stream refers to these buffers and tables:
  // from then on they neither move nor change to another list.
  bool frozen = false;

  void freeze() {
    frozen = true;
    for (DevBuf* b : {&slots, &saved_scales, &norm_buf, &dev_scalars, &cast_descs,
                      &cast_chunks, &step_descs, &step_chunks, &reduce_descs,
                      &reduce_chunks})
      b->frozen = true;
  }

  void release() {
    slots.release();
    saved_scales.release();
    norm_buf.release();
    dev_scalars.release();
    cast_descs.release();
    cast_chunks.release();
    step_descs.release();
    step_chunks.release();
    reduce_descs.release();
    reduce_chunks.release();
    cast_key.clear();
    step_key.clear();
    reduce_key.clear();
    have_cast = have_step = have_reduce = false;
  }
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Workspace*> g_ws;
std::map<int, DeviceInfo> g_dev;

cudaError_t device_info(int dev, DeviceInfo** out) {
  auto it = g_dev.find(dev);
  if (it != g_dev.end()) {
    *out = &it->second;
    return cudaSuccess;
  }
  DeviceInfo info;
  cudaError_t e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int a = 0, b = 0, c = 0;
  if ((e = cast_occupancy(&a, &b)) != cudaSuccess) return e;
  info.cast_amax = info.sms * (a > 0 ? a : 1);
  info.cast_encode = info.sms * (b > 0 ? b : 1);
  int v = 0;
  if ((e = step_occupancy(&a, &b, &v, &c)) != cudaSuccess) return e;
  info.step_amax = info.sms * (a > 0 ? a : 1);
  info.step_update = info.sms * (b > 0 ? b : 1);
  info.step_update_var = info.sms * (v > 0 ? v : 1);
  info.step_w8 = info.sms * (c > 0 ? c : 1);
  if ((e = cast_step_occupancy(&a)) != cudaSuccess) return e;
  info.cast_step = info.sms * (a > 0 ? a : 1);
  int as[3] = {0, 0, 0}, es[3] = {0, 0, 0};
  if ((e = reduce_occupancy(&a, as, &b, es)) != cudaSuccess) return e;
  info.reduce_amax = info.sms * (a > 0 ? a : 1);
  info.reduce_encode = info.sms * (b > 0 ? b : 1);
  for (int i = 0; i < 3; ++i) {
    info.reduce_amax_small[i] = info.sms * (as[i] > 0 ? as[i] : 1);
    info.reduce_encode_small[i] = info.sms * (es[i] > 0 ? es[i] : 1);
  }
  if ((e = grad_norm_occupancy(&a)) != cudaSuccess) return e;
  info.grad_norm = info.sms * (a > 0 ? a : 1);
  int sq[2] = {0, 0};
  if ((e = cast_encode_sq_occupancy(sq)) != cudaSuccess) return e;
  for (int f = 0; f < 2; ++f)
    info.cast_encode_sq[f] = info.sms * (sq[f] > 0 ? sq[f] : 1);
  if ((e = reduce_encode_sq_occupancy(&a, es)) != cudaSuccess) return e;
  info.reduce_encode_sq = info.sms * (a > 0 ? a : 1);
  for (int i = 0; i < 3; ++i)
    info.reduce_encode_sq_small[i] = info.sms * (es[i] > 0 ? es[i] : 1);
  *out = &(g_dev[dev] = info);
  return cudaSuccess;
}

Workspace* workspace(int dev, cudaStream_t s) {
  auto key = std::make_pair(dev, s);
  auto it = g_ws.find(key);
  if (it != g_ws.end()) return it->second;
  Workspace* w = new Workspace();
  w->device = dev;
  g_ws[key] = w;
  return w;
}

// Whether work on `stream` is being captured into a CUDA graph.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(stream, &st) == cudaSuccess &&
         st != cudaStreamCaptureStatusNone;
}

// `words` tagged slots for this call, zeroed when (re)allocated or when the
// epoch wraps; returns the call's epoch.  Under stream capture the epoch is
// fixed into the graph, so the slots are zeroed as part of the captured
// work: every replay then starts from clean slots (and a capture may not
// grow the workspace: run the same list once before capturing).
cudaError_t prepare_slots(Workspace* ws, size_t words, cudaStream_t stream,
                          uint32_t* epoch_out) {
  const size_t bytes = words * sizeof(unsigned long long);
  const bool graph = capturing(stream);
  if (graph && bytes > ws->slots.cap) return cudaErrorStreamCaptureUnsupported;
  if (graph) ws->freeze();
  bool fresh = graph;
  if (bytes > ws->slots.cap) {
    cudaError_t e = ws->slots.reserve(bytes);
    if (e != cudaSuccess) return e;
    fresh = true;
  }
  ws->epoch += 1;
  if (ws->epoch == 0) {   // 2^32 calls: tags would repeat
    fresh = true;
    ws->epoch = 1;
  }
  if (fresh) {
    cudaError_t e = cudaMemsetAsync(ws->slots.ptr, 0, graph ? bytes : ws->slots.cap,
                                    stream);
    if (e != cudaSuccess) return e;
  }
  *epoch_out = ws->epoch;
  return cudaSuccess;
}

// ------------------------------------------------------- per-kernel timing

const char* const kKernelNames[kNumKernels] = {
    "cast_amax", "cast_encode", "step_amax", "step_update", "step_w8",
    "cast_step_amax", "reduce_amax", "reduce_encode", "grad_norm",
    "grad_norm_terms", "clip_coef", "found"};

struct Timing {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  struct Open { int kernel; cudaEvent_t a, b; };
  std::vector<Open> pending;
  cudaEvent_t open_start[kNumKernels] = {};
  int launches[kNumKernels] = {};
  double ms[kNumKernels] = {};
};
Timing g_timing;   // guarded by g_mu

cudaEvent_t timing_event() {
  if (!g_timing.pool.empty()) {
    cudaEvent_t e = g_timing.pool.back();
    g_timing.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void timing_mark(int kernel, int end, cudaStream_t stream) {
  if (capturing(stream)) return;   // graph replays are not timed per kernel
  cudaEvent_t e = timing_event();
  cudaEventRecord(e, stream);
  if (!end) {
    g_timing.open_start[kernel] = e;
  } else {
    g_timing.pending.push_back({kernel, g_timing.open_start[kernel], e});
    g_timing.open_start[kernel] = nullptr;
  }
}

// Every launch sits in an NVTX range named for its pass, so a profiler's
// timeline (Nsight Systems, Nsight Compute's range filters) shows the passes
// by name; without an attached tool a range costs one indirect call.  While
// per-kernel timing is on, the range also holds the two events.
void nvtx_mark(int kernel, int end, cudaStream_t) {
  if (!end)
    nvtxRangePushA(kKernelNames[kernel]);
  else
    nvtxRangePop();
}

void nvtx_timing_mark(int kernel, int end, cudaStream_t stream) {
  if (!end) nvtx_mark(kernel, end, stream);
  timing_mark(kernel, end, stream);
  if (end) nvtx_mark(kernel, end, stream);
}

LaunchMark launch_mark() { return g_timing.on ? nvtx_timing_mark : nvtx_mark; }

// Folds finished event pairs into the totals.
cudaError_t timing_collect() {
  for (const Timing::Open& o : g_timing.pending) {
    cudaError_t e = cudaEventSynchronize(o.b);
    if (e != cudaSuccess) return e;
    float ms = 0.0f;
    e = cudaEventElapsedTime(&ms, o.a, o.b);
    if (e != cudaSuccess) return e;
    g_timing.launches[o.kernel] += 1;
    g_timing.ms[o.kernel] += ms;
    g_timing.pool.push_back(o.a);
    g_timing.pool.push_back(o.b);
  }
  g_timing.pending.clear();
  return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

uint64_t chunks_of(int64_t numel, int shift) {
  return numel == 0 ? 1u : (uint64_t)((numel + ((int64_t)1 << shift) - 1) >> shift);
}

// Chunk size of a list (as a shift): kChunkShift, halved down to min_shift
// while the list has fewer than FP8OPT_CHUNKS_PER_SM chunks per SM.  A
// persistent pass then runs several rounds of chunks on every SM, and its
// last, partly filled round is a small part of it.  min_shift keeps a chunk
// at least one full tile of the passes over the table.  numel(i) gives
// tensor i's element count.  Only the cast's tables use it.  Measured on the
// 124M list: the cast takes 0.0986 ms at 48 or 96 chunks per SM, and 0.1020
// ms with 32768-element chunks.  The reduction (k = 8: 0.408 against 0.352
// ms), the norm and the clipped step were slower with smaller chunks, whose
// per-chunk prologue and CTA reduction then weigh more.  The O2 350M step
// gained under 1 %, so the step's tables keep 32768-element chunks.
#ifndef FP8OPT_CHUNKS_PER_SM
#define FP8OPT_CHUNKS_PER_SM 48
#endif
template <class F>
int halve_chunks(int n, F numel, uint64_t target, int shift, int min_shift) {
  while (shift > min_shift) {
    uint64_t total = 0;
    for (int i = 0; i < n && total < target; ++i) total += chunks_of(numel(i), shift);
    if (total >= target) break;
    --shift;
  }
  return shift;
}

// Smallest chunk shift of the cast's tables: a chunk holds at least one full
// tile of the cast passes (8192 elements).
constexpr int kMinShiftCast = 13;
// A tiny list (at most kTinyElems elements, any table) gets chunks of 2048
// elements, the update pass's tile, so that its few thousand elements spread
// over several SMs instead of one CTA per tensor walking its tiles in turn.
// Passes whose tiles are larger take their scalar path there, which at a
// few elements a thread costs little.  (Larger lists keep chunks of at least
// one full tile of every pass, so their vector paths run.)
constexpr int kMinShiftTiny = 11;
constexpr int64_t kTinyElems = 65536;

// The chunk shift of a table: tiny lists spread over the SMs; the cast's
// tables (cast = true) also follow FP8OPT_CHUNKS_PER_SM; the others keep
// kChunkShift.
template <class F>
int chunk_shift_for(int n, F numel, int sms, bool cast) {
  int64_t elems = 0;
  for (int i = 0; i < n && elems <= kTinyElems; ++i) elems += numel(i);
  if (elems <= kTinyElems)
    return halve_chunks(n, numel, (uint64_t)sms, kChunkShift, kMinShiftTiny);
  if (!cast) return kChunkShift;
  return halve_chunks(n, numel, (uint64_t)FP8OPT_CHUNKS_PER_SM * (uint64_t)sms,
                      kChunkShift, kMinShiftCast);
}

template <class T>
bool same_list(const std::vector<T>& key, const T* items, int n) {
  return key.size() == (size_t)n &&
         (n == 0 || std::memcmp(key.data(), items, sizeof(T) * (size_t)n) == 0);
}

cudaError_t upload(DevBuf& buf, const void* host, size_t bytes,
                   cudaStream_t stream) {
  cudaError_t e = buf.reserve(bytes);
  if (e != cudaSuccess) return e;
  return cudaMemcpyAsync(buf.ptr, host, bytes, cudaMemcpyHostToDevice, stream);
}

int current_device_and_info(int* dev, DeviceInfo** info) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = device_info(*dev, info);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  return FP8OPT_OK;
}

}  // namespace

// Records the detail fp8opt_last_error() returns, for entry points defined
// in other translation units.
int record_error(int status, const char* what) { return fail(status, what); }

}  // namespace fp8opt

using namespace fp8opt;

namespace fp8opt {
namespace {

// A new tensor list is refused under stream capture (the table upload
// would record a copy from host memory the library frees after the call)
// and on a stream whose workspace a captured graph holds.
int refuse_capture(const char* fn) {
  return fail(FP8OPT_ERR_ARG, std::string(fn) +
                                  ": a new tensor list under stream capture, or "
                                  "on a stream a captured CUDA graph uses; run "
                                  "the list once on this stream before capturing, "
                                  "and other lists on other streams");
}

int check_cast_args(const char* fn, const fp8opt_cast_item* items, int n,
                    int fmt) {
  if (n < 0 || (n > 0 && items == nullptr))
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": n < 0 or items is NULL");
  if (fmt != FP8OPT_E4M3 && fmt != FP8OPT_E5M2)
    return fail(FP8OPT_ERR_UNSUPPORTED, std::string(fn) + ": unknown format");
  for (int i = 0; i < n; ++i) {
    const fp8opt_cast_item& it = items[i];
    const std::string at = std::string(fn) + ": item " + std::to_string(i);
    if (it.dtype != FP8OPT_F32 && it.dtype != FP8OPT_BF16 && it.dtype != FP8OPT_F16)
      return fail(FP8OPT_ERR_UNSUPPORTED, at + ": unknown dtype");
    if (it.numel < 0 || it.reserved != 0 || it.amax == nullptr ||
        it.scale == nullptr ||
        (it.numel > 0 && (it.src == nullptr || it.codes == nullptr)))
      return fail(FP8OPT_ERR_ARG, at + ": bad numel, reserved field or NULL pointer");
  }
  return FP8OPT_OK;
}

int check_step_args(const char* fn, const fp8opt_param* params, int n,
                    int64_t step) {
  if (n < 0 || (n > 0 && params == nullptr))
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": n < 0 or params is NULL");
  if (step < 1) return fail(FP8OPT_ERR_ARG, std::string(fn) + ": step < 1");
  for (int i = 0; i < n; ++i) {
    const fp8opt_param& p = params[i];
    const std::string at = std::string(fn) + ": param " + std::to_string(i);
    if (p.g_fmt != FP8OPT_E4M3 && p.g_fmt != FP8OPT_E5M2)
      return fail(FP8OPT_ERR_UNSUPPORTED, at + ": unknown gradient format");
    if (p.numel < 0 || p.reserved != 0 || p.g_scale == nullptr ||
        p.m_scale == nullptr ||
        (p.numel > 0 && (p.g == nullptr || p.m == nullptr || p.v == nullptr ||
                         p.w == nullptr)))
      return fail(FP8OPT_ERR_ARG, at + ": bad numel, reserved field or NULL pointer");
    const bool o3 = p.w8_scale != nullptr || p.w8_amax != nullptr;
    if (o3 && (p.w8_scale == nullptr || p.w8_amax == nullptr ||
               (p.numel > 0 && p.w8 == nullptr)))
      return fail(FP8OPT_ERR_ARG, at + ": O3 needs w8, w8_scale and w8_amax together");
    if (!o3 && p.w8 != nullptr)
      return fail(FP8OPT_ERR_ARG, at + ": w8 given without w8_scale and w8_amax");
  }
  return FP8OPT_OK;
}

// beta^t in double by binary exponentiation (each product rounded to
// double): the same bits on every platform, and the same as a device kernel
// computing it with the same products.
double bias_power(double b, int64_t t) {
  double r = 1.0;
  while (t > 0) {
    if (t & 1) r = r * b;
    b = b * b;
    t >>= 1;
  }
  return r;
}

// Per-call scalars: the bias corrections 1 - beta^t in double, entering only
// through lr / bc1 and 1 / sqrt(bc2), each rounded to fp32 once.
StepScalars make_scalars(float lr, float beta1, float beta2, float eps, float wd,
                         int64_t step, float inv_loss_scale, bool l2) {
  StepScalars s;
  const double bc1 = 1.0 - bias_power((double)beta1, step);
  const double bc2 = 1.0 - bias_power((double)beta2, step);
  s.beta1 = beta1;
  s.beta2 = beta2;
  s.eps = eps;
  s.omb1 = 1.0f - beta1;
  s.omb2 = 1.0f - beta2;
  s.step_size = (float)((double)lr / bc1);
  s.inv_sbc2 = (float)(1.0 / std::sqrt(bc2));
  s.decay = l2 ? 1.0f : 1.0f - lr * wd;
  s.ils = inv_loss_scale;
  s.wd = wd;
  s.l2 = l2 ? 1 : 0;
  s.clip = nullptr;
  s.dev = nullptr;
  s.step_out = nullptr;
  return s;
}

static_assert(sizeof(fp8opt_step_state) == sizeof(DevState) &&
                  offsetof(fp8opt_step_state, lr) == offsetof(DevState, lr) &&
                  offsetof(fp8opt_step_state, inv_loss_scale) ==
                      offsetof(DevState, inv_loss_scale) &&
                  offsetof(fp8opt_step_state, step) == offsetof(DevState, step),
              "fp8opt_step_state and DevState must share one layout");

// The scalars of a device-resident step: the constants from the host, the
// per-step values from the DevScalars the scalars kernel writes, and the
// caller's step count to advance.
StepScalars make_dev_scalars(float beta1, float beta2, float eps, float wd,
                             bool l2, const DevScalars* dev, long long* step_out) {
  StepScalars s = make_scalars(0.0f, beta1, beta2, eps, wd, 1, 1.0f, l2);
  s.step_size = s.inv_sbc2 = s.ils = 0.0f;
  s.decay = 1.0f;
  s.dev = dev;
  s.step_out = step_out;
  return s;
}

int check_dev_state(const char* fn, const fp8opt_step_state* state) {
  if (state == nullptr ||
      (reinterpret_cast<uintptr_t>(state) & (alignof(fp8opt_step_state) - 1)) != 0)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": state is NULL or misaligned");
  return FP8OPT_OK;
}

// The workspace's DevScalars for a *_dev call.
int dev_scalars_buf(const char* fn, Workspace* ws, DevScalars** out) {
  cudaError_t e = ws->dev_scalars.reserve(sizeof(DevScalars));
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": workspace").c_str());
  *out = static_cast<DevScalars*>(ws->dev_scalars.ptr);
  return FP8OPT_OK;
}

// A *_dev call without chunks: the step is taken (nothing can be non-finite),
// so the scalars kernel advances the step count itself.
int empty_dev_step(const char* fn, fp8opt_step_state* state, float beta1,
                   float beta2, float wd, bool l2, uint32_t* found_inf_dev,
                   Workspace* ws, cudaStream_t stream) {
  DevScalars* ds = nullptr;
  int st = dev_scalars_buf(fn, ws, &ds);
  if (st != FP8OPT_OK) return st;
  cudaError_t e = launch_step_scalars(reinterpret_cast<DevState*>(state), beta1,
                                      beta2, wd, l2, ds, true, stream);
  if (e == cudaSuccess && found_inf_dev != nullptr)
    e = cudaMemsetAsync(found_inf_dev, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  return FP8OPT_OK;
}

// The workspace's cast tables for this item list (uploaded when the list
// differs from the cached one).
int ensure_cast_tables(const char* fn, Workspace* ws,
                       const fp8opt_cast_item* items, int n,
                       cudaStream_t stream) {
  if (ws->have_cast && same_list(ws->cast_key, items, n)) return FP8OPT_OK;
  if (capturing(stream) || ws->frozen) return refuse_capture(fn);
  if ((uint32_t)n >= kMaxListTensors)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": too many tensors");
  DeviceInfo* info = nullptr;
  cudaError_t ie = device_info(ws->device, &info);
  if (ie != cudaSuccess) return cuda_fail(ie, (std::string(fn) + ": device query").c_str());
  const int shift = chunk_shift_for(n, [&](int i) { return items[i].numel; },
                                    info->sms, true);
  std::vector<CastDesc> descs((size_t)n);
  std::vector<Chunk> chunks;
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += chunks_of(items[i].numel, shift);
  if (total > 0xFFFFFFFFull)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": list too long");
  chunks.reserve(total);
  for (int i = 0; i < n; ++i) {
    const fp8opt_cast_item& it = items[i];
    CastDesc& d = descs[(size_t)i];
    d.src = it.src;
    d.codes = it.codes;
    d.amax_out = it.amax;
    d.scale_out = it.scale;
    d.numel = it.numel;
    d.dtype = it.dtype;
    d.vec_ok = aligned(it.src, 16) && aligned(it.codes, 8);
    for (uint32_t c = 0, nc = (uint32_t)chunks_of(it.numel, shift); c < nc; ++c)
      chunks.push_back(make_chunk((uint32_t)i, c, shift, it.numel));
  }
  ws->have_cast = false;
  cudaError_t e;
  if ((e = upload(ws->cast_descs, descs.data(), descs.size() * sizeof(CastDesc),
                  stream)) != cudaSuccess ||
      (e = upload(ws->cast_chunks, chunks.data(), chunks.size() * sizeof(Chunk),
                  stream)) != cudaSuccess)
    return cuda_fail(e, (std::string(fn) + ": table upload").c_str());
  ws->cast_key.assign(items, items + n);
  ws->cast_nchunks = (uint32_t)chunks.size();
  ws->have_cast = true;
  return FP8OPT_OK;
}

// The workspace's step tables: the main chunk list, then the O3 chunks.
int ensure_step_tables(const char* fn, Workspace* ws, const fp8opt_param* params,
                       int n, cudaStream_t stream) {
  if (ws->have_step && same_list(ws->step_key, params, n)) return FP8OPT_OK;
  if (capturing(stream) || ws->frozen) return refuse_capture(fn);
  if ((uint32_t)n >= kMaxListTensors)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": too many tensors");
  DeviceInfo* info = nullptr;
  cudaError_t ie = device_info(ws->device, &info);
  if (ie != cudaSuccess) return cuda_fail(ie, (std::string(fn) + ": device query").c_str());
  const int shift = chunk_shift_for(n, [&](int i) { return params[i].numel; },
                                    info->sms, false);
  std::vector<StepDesc> descs((size_t)n);
  std::vector<Chunk> chunks, chunks_o3;
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += 2 * (size_t)chunks_of(params[i].numel, shift);
  if (total > 0xFFFFFFFFull)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": list too long");
  for (int i = 0; i < n; ++i) {
    const fp8opt_param& p = params[i];
    StepDesc& d = descs[(size_t)i];
    d.g = p.g;
    d.m = p.m;
    d.v = p.v;
    d.w = p.w;
    d.w8 = p.w8;
    d.g_scale = p.g_scale;
    d.m_scale = p.m_scale;
    d.w8_scale = p.w8_scale;
    d.w8_amax = p.w8_amax;
    d.v_bound = p.v_bound;
    d.numel = p.numel;
    d.g_fmt = p.g_fmt;
    d.o3 = p.w8_scale != nullptr;
    d.vec_ok = aligned(p.g, 8) && aligned(p.m, 8) && aligned(p.v, 16) &&
               aligned(p.w, 16) && (p.w8 == nullptr || aligned(p.w8, 8));
    for (uint32_t c = 0, nc = (uint32_t)chunks_of(p.numel, shift); c < nc; ++c) {
      chunks.push_back(make_chunk((uint32_t)i, c, shift, p.numel));
      if (d.o3) chunks_o3.push_back(make_chunk((uint32_t)i, c, shift, p.numel));
    }
  }
  const uint32_t nmain = (uint32_t)chunks.size();
  const uint32_t no3 = (uint32_t)chunks_o3.size();
  chunks.insert(chunks.end(), chunks_o3.begin(), chunks_o3.end());
  ws->have_step = false;
  cudaError_t e;
  if ((e = upload(ws->step_descs, descs.data(), descs.size() * sizeof(StepDesc),
                  stream)) != cudaSuccess ||
      (e = upload(ws->step_chunks, chunks.data(), chunks.size() * sizeof(Chunk),
                  stream)) != cudaSuccess)
    return cuda_fail(e, (std::string(fn) + ": table upload").c_str());
  ws->step_key.assign(params, params + n);
  ws->step_nchunks = nmain;
  ws->step_nchunks_o3 = no3;
  ws->step_any_vs = false;
  ws->step_fmts = 0;
  for (int i = 0; i < n; ++i) {
    ws->step_any_vs |= params[i].v_bound != nullptr;
    ws->step_fmts |= 1 << params[i].g_fmt;
  }
  ws->have_step = true;
  return FP8OPT_OK;
}

int check_reduce_args(const char* fn, const fp8opt_reduce_item* items, int n,
                      int k, int in_fmt, int out_fmt) {
  if (n < 0 || (n > 0 && items == nullptr))
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": n < 0 or items is NULL");
  if (k < 1 || k > FP8OPT_MAX_SHARDS)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": k outside [1, FP8OPT_MAX_SHARDS]");
  if ((in_fmt != FP8OPT_E4M3 && in_fmt != FP8OPT_E5M2) ||
      (out_fmt != FP8OPT_E4M3 && out_fmt != FP8OPT_E5M2))
    return fail(FP8OPT_ERR_UNSUPPORTED, std::string(fn) + ": unknown format");
  for (int i = 0; i < n; ++i) {
    const fp8opt_reduce_item& it = items[i];
    const std::string at = std::string(fn) + ": item " + std::to_string(i);
    if (it.numel < 0 || it.stride < it.numel || it.amax == nullptr ||
        it.scale == nullptr ||
        (it.numel > 0 && (it.src == nullptr || it.src_scale == nullptr ||
                          it.codes == nullptr)))
      return fail(FP8OPT_ERR_ARG, at + ": bad numel or stride, or NULL pointer");
    if (it.numel > 0 && it.stride > (INT64_MAX - it.numel) / k)
      return fail(FP8OPT_ERR_ARG, at + ": k * stride overflows");
  }
  return FP8OPT_OK;
}

// The workspace's reduction tables for this item list.
int ensure_reduce_tables(const char* fn, Workspace* ws,
                         const fp8opt_reduce_item* items, int n,
                         cudaStream_t stream) {
  if (ws->have_reduce && same_list(ws->reduce_key, items, n)) return FP8OPT_OK;
  if (capturing(stream) || ws->frozen) return refuse_capture(fn);
  if ((uint32_t)n >= kMaxListTensors)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": too many tensors");
  DeviceInfo* info = nullptr;
  cudaError_t ie = device_info(ws->device, &info);
  if (ie != cudaSuccess) return cuda_fail(ie, (std::string(fn) + ": device query").c_str());
  const int shift = chunk_shift_for(n, [&](int i) { return items[i].numel; },
                                    info->sms, false);
  std::vector<ReduceDesc> descs((size_t)n);
  std::vector<Chunk> chunks;
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += chunks_of(items[i].numel, shift);
  if (total > 0xFFFFFFFFull)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": list too long");
  chunks.reserve(total);
  for (int i = 0; i < n; ++i) {
    const fp8opt_reduce_item& it = items[i];
    ReduceDesc& d = descs[(size_t)i];
    d.src = it.src;
    d.src_scale = it.src_scale;
    d.codes = it.codes;
    d.amax_out = it.amax;
    d.scale_out = it.scale;
    d.numel = it.numel;
    d.stride = it.stride;
    d.vec_ok = aligned(it.src, 16) && aligned(it.codes, 16) && it.stride % 16 == 0;
    d.pad = 0;
    for (uint32_t c = 0, nc = (uint32_t)chunks_of(it.numel, shift); c < nc; ++c)
      chunks.push_back(make_chunk((uint32_t)i, c, shift, it.numel));
  }
  ws->have_reduce = false;
  cudaError_t e;
  if ((e = upload(ws->reduce_descs, descs.data(), descs.size() * sizeof(ReduceDesc),
                  stream)) != cudaSuccess ||
      (e = upload(ws->reduce_chunks, chunks.data(), chunks.size() * sizeof(Chunk),
                  stream)) != cudaSuccess)
    return cuda_fail(e, (std::string(fn) + ": table upload").c_str());
  ws->reduce_key.assign(items, items + n);
  ws->reduce_nchunks = (uint32_t)chunks.size();
  ws->have_reduce = true;
  return FP8OPT_OK;
}

// A fused cast + step call: params[i] must take grads[i]'s output.
int check_takes_cast(const char* fn, const fp8opt_cast_item* grads,
                     const fp8opt_param* params, int n, int fmt) {
  for (int i = 0; i < n; ++i) {
    const fp8opt_param& p = params[i];
    if (p.g != grads[i].codes || p.g_scale != grads[i].scale ||
        p.numel != grads[i].numel || p.g_fmt != fmt)
      return fail(FP8OPT_ERR_ARG, std::string(fn) + ": param " + std::to_string(i) +
                                      " does not take item " + std::to_string(i) +
                                      "'s codes, scale, numel and format");
  }
  return FP8OPT_OK;
}

// The empty-list result of a step call.
int empty_step(const char* fn, int* found_inf, uint32_t* found_inf_dev,
               cudaStream_t stream) {
  if (found_inf != nullptr) *found_inf = 0;
  if (found_inf_dev != nullptr) {
    cudaError_t e = cudaMemsetAsync(found_inf_dev, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": found_inf_dev").c_str());
  }
  return FP8OPT_OK;
}

// Waits for the stream and reads this call's found_inf word.  Called after
// g_mu is released: the read blocks until the stream has run the call's
// kernels, and other threads' calls on other streams must not wait for that.
// The word stays valid meanwhile: only calls on this stream (one host thread
// at a time) reuse this stream's workspace.
int read_found(const char* fn, const unsigned long long* found, uint32_t epoch,
               cudaStream_t stream, int* out) {
  unsigned long long tag = 0;
  cudaError_t e = cudaMemcpyAsync(&tag, found, sizeof(tag), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": found_inf read").c_str());
  *out = tag == (((unsigned long long)epoch << 32) | 1ull) ? 1 : 0;
  return FP8OPT_OK;
}

}  // namespace
}  // namespace fp8opt

extern "C" int fp8_cast_scaled(const fp8opt_cast_item* items, int n, int fmt,
                               void* stream_ptr) {
  const char* fn = "fp8_cast_scaled";
  int st = check_cast_args(fn, items, n, fmt);
  if (st != FP8OPT_OK || n == 0) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if ((st = ensure_cast_tables(fn, ws, items, n, stream)) != FP8OPT_OK) return st;

  uint32_t epoch = 0;
  cudaError_t e = prepare_slots(ws, (size_t)n, stream, &epoch);   // [0, n) amax
  if (e != cudaSuccess) return cuda_fail(e, "fp8_cast_scaled: workspace");
  e = launch_cast(static_cast<const CastDesc*>(ws->cast_descs.ptr),
                  static_cast<const Chunk*>(ws->cast_chunks.ptr), ws->cast_nchunks,
                  static_cast<unsigned long long*>(ws->slots.ptr), epoch, fmt,
                  info->cast_amax, info->cast_encode, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, "fp8_cast_scaled: launch");
  return FP8OPT_OK;
}

namespace fp8opt {
namespace {

// What a reduction call runs: its passes (phase), the amax pass's per-item
// values exported (amax_out) or the encode pass's imported (amax_in), and
// the norm of the outputs (with_norm) as terms or as exact limbs, with
// found_inf (found, may be NULL).
struct ReduceReq {
  int phase = kReduceBothPasses;
  uint32_t* amax_out = nullptr;
  const uint32_t* amax_in = nullptr;
  bool with_norm = false;
  float ils = 1.0f;
  double* terms = nullptr;
  long long* limbs = nullptr;
  uint32_t* found = nullptr;
};

// The reduction entry points.
int reduce_call(const char* fn, const fp8opt_reduce_item* items, int n, int k,
                int in_fmt, int out_fmt, float post, const ReduceReq& rq,
                void* stream_ptr) {
  int st = check_reduce_args(fn, items, n, k, in_fmt, out_fmt);
  if (st != FP8OPT_OK) return st;
  if (rq.with_norm && n > 0 && rq.terms == nullptr && rq.limbs == nullptr)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": terms_dev is NULL");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0)
    return rq.with_norm ? empty_step(fn, nullptr, rq.found, stream) : FP8OPT_OK;

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if ((st = ensure_reduce_tables(fn, ws, items, n, stream)) != FP8OPT_OK) return st;

  // slots: [0, n) amax, [n] found_inf; norm: 2n words of exact sums
  uint32_t epoch = 0;
  cudaError_t e = prepare_slots(ws, (size_t)n + 1, stream, &epoch);
  const size_t sum_bytes = 2 * (size_t)n * sizeof(unsigned long long);
  if (e == cudaSuccess && rq.with_norm) e = ws->norm_buf.reserve(sum_bytes);
  if (e == cudaSuccess && rq.with_norm)
    e = cudaMemsetAsync(ws->norm_buf.ptr, 0, sum_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": workspace").c_str());
  unsigned long long* slots = static_cast<unsigned long long*>(ws->slots.ptr);
  if (rq.amax_in != nullptr)
    e = launch_slots_import(slots, epoch, n, rq.amax_in, stream);
  ReduceNorm norm = {static_cast<unsigned long long*>(ws->norm_buf.ptr),
                     slots + n, rq.ils, n, rq.terms, rq.found, rq.limbs};
  // the k-specialised passes' grids: k <= 2, k = 4, k = 8
  const int ks = k <= 2 ? 0 : k == 4 ? 1 : k == 8 ? 2 : -1;
  if (e == cudaSuccess)
    e = launch_reduce(static_cast<const ReduceDesc*>(ws->reduce_descs.ptr),
                      static_cast<const Chunk*>(ws->reduce_chunks.ptr),
                      ws->reduce_nchunks, slots, epoch, k, in_fmt, out_fmt, post,
                      ks >= 0 ? info->reduce_amax_small[ks] : info->reduce_amax,
                      rq.with_norm ? (ks >= 0 ? info->reduce_encode_sq_small[ks]
                                              : info->reduce_encode_sq)
                      : ks >= 0 ? info->reduce_encode_small[ks]
                                : info->reduce_encode,
                      rq.with_norm ? &norm : nullptr, stream, launch_mark(),
                      rq.phase);
  if (e == cudaSuccess && rq.amax_out != nullptr)
    e = launch_slots_export(slots, epoch, n, rq.amax_out, stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  return FP8OPT_OK;
}

}  // namespace
}  // namespace fp8opt

extern "C" int fp8_reduce_scaled(const fp8opt_reduce_item* items, int n, int k,
                                 int in_fmt, int out_fmt, float post,
                                 void* stream_ptr) {
  return reduce_call("fp8_reduce_scaled", items, n, k, in_fmt, out_fmt, post,
                     ReduceReq(), stream_ptr);
}

extern "C" int fp8_reduce_scaled_norm(const fp8opt_reduce_item* items, int n,
                                      int k, int in_fmt, int out_fmt, float post,
                                      float inv_loss_scale, double* terms_dev,
                                      uint32_t* found_dev, void* stream_ptr) {
  ReduceReq rq;
  rq.with_norm = true;
  rq.ils = inv_loss_scale;
  rq.terms = terms_dev;
  rq.found = found_dev;
  return reduce_call("fp8_reduce_scaled_norm", items, n, k, in_fmt, out_fmt, post,
                     rq, stream_ptr);
}

extern "C" int fp8_reduce_scaled_begin(const fp8opt_reduce_item* items, int n,
                                       int k, int in_fmt, float post,
                                       uint32_t* amax_bits_dev, void* stream_ptr) {
  if (n > 0 && amax_bits_dev == nullptr)
    return fail(FP8OPT_ERR_ARG, "fp8_reduce_scaled_begin: amax_bits_dev is NULL");
  ReduceReq rq;
  rq.phase = kReduceAmaxPass;
  rq.amax_out = amax_bits_dev;
  return reduce_call("fp8_reduce_scaled_begin", items, n, k, in_fmt, in_fmt, post,
                     rq, stream_ptr);
}

extern "C" int fp8_reduce_scaled_finish(const fp8opt_reduce_item* items, int n,
                                        int k, int in_fmt, int out_fmt,
                                        float post, const uint32_t* amax_bits_dev,
                                        float inv_loss_scale, int64_t* limbs_dev,
                                        uint32_t* found_dev, void* stream_ptr) {
  if (n > 0 && amax_bits_dev == nullptr)
    return fail(FP8OPT_ERR_ARG, "fp8_reduce_scaled_finish: amax_bits_dev is NULL");
  if (found_dev != nullptr && limbs_dev == nullptr)
    return fail(FP8OPT_ERR_ARG,
                "fp8_reduce_scaled_finish: found_dev is given without limbs_dev");
  ReduceReq rq;
  rq.phase = kReduceEncodePass;
  rq.amax_in = amax_bits_dev;
  if (limbs_dev != nullptr) {
    rq.with_norm = true;
    rq.ils = inv_loss_scale;
    rq.limbs = reinterpret_cast<long long*>(limbs_dev);
    rq.found = found_dev;
  }
  return reduce_call("fp8_reduce_scaled_finish", items, n, k, in_fmt, out_fmt,
                     post, rq, stream_ptr);
}

extern "C" int fp8_norm_terms_from_limbs(const int64_t* limbs_dev,
                                         const uint32_t* amax_bits_dev, int n,
                                         int fmt, float inv_loss_scale,
                                         double* terms_dev, void* stream_ptr) {
  if (n < 0 || (n > 0 && (limbs_dev == nullptr || amax_bits_dev == nullptr ||
                          terms_dev == nullptr)))
    return fail(FP8OPT_ERR_ARG,
                "fp8_norm_terms_from_limbs: n < 0 or a NULL device array");
  if (fmt != FP8OPT_E4M3 && fmt != FP8OPT_E5M2)
    return fail(FP8OPT_ERR_UNSUPPORTED, "fp8_norm_terms_from_limbs: unknown format");
  cudaError_t e = launch_limbs_terms(reinterpret_cast<const long long*>(limbs_dev),
                                     amax_bits_dev, n, fmt, inv_loss_scale,
                                     terms_dev, static_cast<cudaStream_t>(stream_ptr));
  if (e != cudaSuccess) return cuda_fail(e, "fp8_norm_terms_from_limbs: launch");
  return FP8OPT_OK;
}

namespace fp8opt {
namespace {

// The gradient-norm request of a call: the norm pass runs when `on`; the
// step (if any) clips to max_norm when max_norm > 0.
struct NormReq {
  bool on = false;
  float max_norm = 0.0f;
  double* norm = nullptr;      // host out, or NULL
  float* norm_dev = nullptr;   // device out, or NULL
};

// Waits for the stream and reads this call's found_inf word and norm; called
// after g_mu is released, as read_found.
int read_results(const char* fn, const unsigned long long* found, uint32_t epoch,
                 const double* norm_dev, cudaStream_t stream, int* found_out,
                 double* norm_out) {
  unsigned long long tag = 0;
  double norm = 0.0;
  cudaError_t e = cudaSuccess;
  if (found_out != nullptr)
    e = cudaMemcpyAsync(&tag, found, sizeof(tag), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess && norm_out != nullptr)
    e = cudaMemcpyAsync(&norm, norm_dev, sizeof(norm), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": result read").c_str());
  if (found_out != nullptr)
    *found_out = tag == (((unsigned long long)epoch << 32) | 1ull) ? 1 : 0;
  if (norm_out != nullptr) *norm_out = norm;
  return FP8OPT_OK;
}

// One step call's device state: tables, slots and scratch on the stream's
// workspace, with this call's epoch.
struct StepCall {
  cudaStream_t stream = nullptr;
  DeviceInfo* info = nullptr;
  Workspace* ws = nullptr;
  uint32_t epoch = 0;
  StepScratch sc;
  const StepDesc* descs = nullptr;
  const Chunk* chunks = nullptr;
  unsigned long long* sums = nullptr;   // norm: 2n words
  double* terms = nullptr;              // norm: n terms
  double* norm = nullptr;               // norm: the norm
  float* clip = nullptr;                // norm: the clip coefficient
};

// Tables and scratch for n records; fresh = false keeps the current epoch
// (the finish of a begun step).  Must run under g_mu.
int setup_step(const char* fn, const fp8opt_param* params, int n,
               void* stream_ptr, bool with_norm, bool fresh, StepCall* c) {
  c->stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  int st = current_device_and_info(&dev, &c->info);
  if (st != FP8OPT_OK) return st;
  Workspace* ws = c->ws = workspace(dev, c->stream);
  if ((st = ensure_step_tables(fn, ws, params, n, c->stream)) != FP8OPT_OK) return st;
  // slots: [0, n) amax of m, [n, 2n) amax of the master, [2n, 3n) max |g|,
  // [3n] found_inf; saved: [0, n) m_scale, [n, 2n) v_bound; norm: [0, 2n)
  // 128-bit sums, n terms, the norm (double) and the clip coefficient (float)
  cudaError_t e = cudaSuccess;
  if (fresh) e = prepare_slots(ws, 3 * (size_t)n + 1, c->stream, &c->epoch);
  else c->epoch = ws->epoch;
  if (e == cudaSuccess) e = ws->saved_scales.reserve(2 * (size_t)n * sizeof(float));
  const size_t sum_bytes = 2 * (size_t)n * sizeof(unsigned long long);
  const size_t norm_bytes = sum_bytes + (size_t)n * sizeof(double) + 16;
  if (e == cudaSuccess && with_norm) e = ws->norm_buf.reserve(norm_bytes);
  if (e == cudaSuccess && with_norm)
    e = cudaMemsetAsync(ws->norm_buf.ptr, 0, sum_bytes, c->stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": workspace").c_str());
  unsigned long long* slots = static_cast<unsigned long long*>(ws->slots.ptr);
  c->sc.amax_m = slots;
  c->sc.amax_w = slots + n;
  c->sc.amax_g = slots + 2 * (size_t)n;
  c->sc.found = slots + 3 * (size_t)n;
  c->sc.old_m_scale = static_cast<float*>(ws->saved_scales.ptr);
  c->sc.old_v_bound = c->sc.old_m_scale + n;
  c->descs = static_cast<const StepDesc*>(ws->step_descs.ptr);
  c->chunks = static_cast<const Chunk*>(ws->step_chunks.ptr);
  if (with_norm) {
    char* nb = static_cast<char*>(ws->norm_buf.ptr);
    c->sums = reinterpret_cast<unsigned long long*>(nb);
    c->terms = reinterpret_cast<double*>(nb + sum_bytes);
    c->norm = c->terms + n;
    c->clip = reinterpret_cast<float*>(c->norm + 1);
  }
  return FP8OPT_OK;
}

// The step entry points: AdamW (l2 false) or Adam with L2 decay, optionally
// with the gradient-norm pass (and clipping); run_step false runs the norm
// pass alone.
int adam_step(const char* fn, bool l2, const fp8opt_param* params, int n,
              float lr, float beta1, float beta2, float eps, float wd,
              int64_t step, float inv_loss_scale, int* found_inf,
              uint32_t* found_inf_dev, void* stream_ptr,
              const NormReq& nr = NormReq(), bool run_step = true) {
  int st = check_step_args(fn, params, n, step);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) {
    if (nr.norm != nullptr) *nr.norm = 0.0;
    if (nr.norm_dev != nullptr) {
      cudaError_t e = cudaMemsetAsync(nr.norm_dev, 0, sizeof(float), stream);
      if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": norm_dev").c_str());
    }
    return empty_step(fn, found_inf, found_inf_dev, stream);
  }
  StepScalars s =
      make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale, l2);

  std::unique_lock<std::mutex> lock(g_mu);
  StepCall c;
  if ((st = setup_step(fn, params, n, stream_ptr, nr.on, true, &c)) != FP8OPT_OK)
    return st;
  Workspace* ws = c.ws;
  cudaError_t e = cudaSuccess;
  if (nr.on) {
    // the norm pass, then the terms, norm and clip coefficient in one launch
    e = launch_grad_norm_terms(c.descs, c.chunks, ws->step_nchunks, 0,
                               inv_loss_scale, nullptr, c.sums, c.sc.found,
                               c.epoch, c.terms, nullptr, c.info->grad_norm,
                               ws->step_fmts, stream, launch_mark());
    if (e == cudaSuccess)
      e = launch_norm_finish(c.descs, n, inv_loss_scale, nullptr, c.sums,
                             c.sc.found, c.epoch, c.terms,
                             run_step ? nr.max_norm : 0.0f, c.norm, c.clip,
                             nr.norm_dev, stream, launch_mark());
    if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
    if (nr.max_norm > 0.0f) s.clip = c.clip;
  }
  if (run_step) {
    e = launch_step(c.descs, c.chunks, ws->step_nchunks,
                    c.chunks + ws->step_nchunks, ws->step_nchunks_o3, c.sc, s,
                    c.epoch, found_inf_dev, c.info->step_amax,
                    c.info->step_update, c.info->step_update_var,
                    c.info->step_w8, ws->step_any_vs, stream, launch_mark());
    if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  }
  lock.unlock();   // before any wait for the stream
  if (found_inf != nullptr || nr.norm != nullptr)
    return read_results(fn, c.sc.found, c.epoch, c.norm, stream, found_inf, nr.norm);
  return FP8OPT_OK;
}

}  // namespace
}  // namespace fp8opt

extern "C" int fp8_grad_norm(const fp8opt_param* params, int n,
                             float inv_loss_scale, double* norm, float* norm_dev,
                             int* found_inf, void* stream_ptr) {
  NormReq nr;
  nr.on = true;
  nr.norm = norm;
  nr.norm_dev = norm_dev;
  return adam_step("fp8_grad_norm", false, params, n, 0.0f, 0.0f, 0.0f, 0.0f,
                   0.0f, 1, inv_loss_scale, found_inf, nullptr, stream_ptr, nr,
                   false);
}

extern "C" int fp8_adam_step_clipped(const fp8opt_param* params, int n, float lr,
                                     float beta1, float beta2, float eps,
                                     float wd, int64_t step, float inv_loss_scale,
                                     int l2, float max_grad_norm,
                                     double* grad_norm, float* grad_norm_dev,
                                     int* found_inf, uint32_t* found_inf_dev,
                                     void* stream_ptr) {
  if (l2 != 0 && l2 != 1)
    return fail(FP8OPT_ERR_ARG, "fp8_adam_step_clipped: l2 must be 0 or 1");
  if (std::isnan(max_grad_norm))
    return fail(FP8OPT_ERR_ARG, "fp8_adam_step_clipped: max_grad_norm is NaN");
  NormReq nr;
  nr.on = true;
  nr.max_norm = max_grad_norm;
  nr.norm = grad_norm;
  nr.norm_dev = grad_norm_dev;
  return adam_step("fp8_adam_step_clipped", l2 != 0, params, n, lr, beta1, beta2,
                   eps, wd, step, inv_loss_scale, found_inf, found_inf_dev,
                   stream_ptr, nr, true);
}

extern "C" int fp8_grad_norm_terms(const fp8opt_param* params, int n,
                                   float inv_loss_scale, double* terms_dev,
                                   uint32_t* found_dev, void* stream_ptr) {
  const char* fn = "fp8_grad_norm_terms";
  int st = check_step_args(fn, params, n, 1);
  if (st != FP8OPT_OK) return st;
  if (n > 0 && terms_dev == nullptr)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": terms_dev is NULL");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) return empty_step(fn, nullptr, found_dev, stream);
  std::lock_guard<std::mutex> lock(g_mu);
  StepCall c;
  if ((st = setup_step(fn, params, n, stream_ptr, true, true, &c)) != FP8OPT_OK)
    return st;
  cudaError_t e = launch_grad_norm_terms(
      c.descs, c.chunks, c.ws->step_nchunks, n, inv_loss_scale, nullptr, c.sums,
      c.sc.found, c.epoch, terms_dev, found_dev, c.info->grad_norm,
      c.ws->step_fmts, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, "fp8_grad_norm_terms: launch");
  return FP8OPT_OK;
}

extern "C" int fp8_clip_coef(const double* terms_dev, int n,
                             const uint32_t* found_dev, float max_grad_norm,
                             double* norm_dev, float* clip_dev,
                             void* stream_ptr) {
  if (n < 0 || (n > 0 && terms_dev == nullptr) || clip_dev == nullptr ||
      std::isnan(max_grad_norm))
    return fail(FP8OPT_ERR_ARG,
                "fp8_clip_coef: n < 0, NULL terms or clip, or a NaN max_grad_norm");
  std::lock_guard<std::mutex> lock(g_mu);
  cudaError_t e = launch_clip_coef(terms_dev, n, nullptr, 0, found_dev,
                                   max_grad_norm, norm_dev, clip_dev, nullptr,
                                   static_cast<cudaStream_t>(stream_ptr),
                                   launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, "fp8_clip_coef: launch");
  return FP8OPT_OK;
}

namespace fp8opt {
namespace {

int check_phase_args(const char* fn, int l2) {
  if (l2 != 0 && l2 != 1) return fail(FP8OPT_ERR_ARG, std::string(fn) + ": l2 must be 0 or 1");
  return FP8OPT_OK;
}

}  // namespace
}  // namespace fp8opt

extern "C" int fp8_adam_step_begin(const fp8opt_param* params, int n, float lr,
                                   float beta1, float beta2, float eps, float wd,
                                   int64_t step, float inv_loss_scale, int l2,
                                   const float* clip_dev, uint32_t* found_dev,
                                   uint32_t* maxima_out, void* stream_ptr) {
  const char* fn = "fp8_adam_step_begin";
  int st = check_phase_args(fn, l2);
  if (st == FP8OPT_OK) st = check_step_args(fn, params, n, step);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) return empty_step(fn, nullptr, found_dev, stream);
  StepScalars s = make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale,
                               l2 != 0);
  s.clip = clip_dev;
  std::lock_guard<std::mutex> lock(g_mu);
  StepCall c;
  if ((st = setup_step(fn, params, n, stream_ptr, false, true, &c)) != FP8OPT_OK)
    return st;
  cudaError_t e = launch_step_amax(c.descs, c.chunks, c.ws->step_nchunks, c.sc, s,
                                   c.epoch, c.info->step_amax, stream,
                                   launch_mark());
  if (e == cudaSuccess && found_dev != nullptr)
    e = launch_found(c.sc.found, c.epoch, nullptr, found_dev, stream, launch_mark());
  if (e == cudaSuccess && maxima_out != nullptr)
    e = launch_slots_export(c.sc.amax_m, c.epoch, n, maxima_out, stream);
  if (e == cudaSuccess && maxima_out != nullptr)
    e = launch_slots_export(c.sc.amax_g, c.epoch, n, maxima_out + n, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fp8_adam_step_begin: launch");
  c.ws->begin_epoch = c.epoch;
  c.ws->copy_epoch = 0;
  return FP8OPT_OK;
}

extern "C" int fp8_adam_step_finish(const fp8opt_param* params, int n, float lr,
                                    float beta1, float beta2, float eps,
                                    float wd, int64_t step, float inv_loss_scale,
                                    int l2, const float* clip_dev,
                                    const uint32_t* found_in_dev,
                                    uint32_t* found_dev,
                                    const uint32_t* maxima_in,
                                    uint32_t* master_amax_out, void* stream_ptr) {
  const char* fn = "fp8_adam_step_finish";
  int st = check_phase_args(fn, l2);
  if (st == FP8OPT_OK) st = check_step_args(fn, params, n, step);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) return empty_step(fn, nullptr, found_dev, stream);
  StepScalars s = make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale,
                               l2 != 0);
  s.clip = clip_dev;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if (!ws->have_step || !same_list(ws->step_key, params, n) ||
      ws->begin_epoch == 0 || ws->begin_epoch != ws->epoch)
    return fail(FP8OPT_ERR_ARG, std::string(fn) +
                                    ": no fp8_adam_step_begin of this list is "
                                    "pending on this stream");
  StepCall c;
  if ((st = setup_step(fn, params, n, stream_ptr, false, false, &c)) != FP8OPT_OK)
    return st;
  ws->begin_epoch = 0;
  cudaError_t e = launch_found(c.sc.found, c.epoch, found_in_dev, nullptr, stream,
                               launch_mark());
  // the whole tensors' maxima, combined over the ranks holding their pieces
  if (e == cudaSuccess && maxima_in != nullptr)
    e = launch_slots_import(c.sc.amax_m, c.epoch, n, maxima_in, stream);
  if (e == cudaSuccess && maxima_in != nullptr)
    e = launch_slots_import(c.sc.amax_g, c.epoch, n, maxima_in + n, stream);
  // with master_amax_out the O3 weight copy waits for fp8_adam_step_copy
  const bool copy_now = master_amax_out == nullptr;
  if (e == cudaSuccess)
    e = launch_step_update(c.descs, c.chunks, ws->step_nchunks,
                           c.chunks + ws->step_nchunks,
                           copy_now ? ws->step_nchunks_o3 : 0, c.sc, s, c.epoch,
                           found_dev, info->step_update, info->step_update_var,
                           info->step_w8, ws->step_any_vs, stream, launch_mark());
  if (e == cudaSuccess && !copy_now)
    e = launch_slots_export(c.sc.amax_w, c.epoch, n, master_amax_out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fp8_adam_step_finish: launch");
  ws->copy_epoch = copy_now ? 0 : c.epoch;
  return FP8OPT_OK;
}

extern "C" int fp8_adam_step_copy(const fp8opt_param* params, int n,
                                  const uint32_t* master_amax_in,
                                  void* stream_ptr) {
  const char* fn = "fp8_adam_step_copy";
  int st = check_step_args(fn, params, n, 1);
  if (st != FP8OPT_OK) return st;
  if (n > 0 && master_amax_in == nullptr)
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": master_amax_in is NULL");
  if (n == 0) return FP8OPT_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if (!ws->have_step || !same_list(ws->step_key, params, n) ||
      ws->copy_epoch == 0 || ws->copy_epoch != ws->epoch)
    return fail(FP8OPT_ERR_ARG, std::string(fn) +
                                    ": no fp8_adam_step_finish of this list with "
                                    "master_amax_out is pending on this stream");
  StepCall c;
  if ((st = setup_step(fn, params, n, stream_ptr, false, false, &c)) != FP8OPT_OK)
    return st;
  ws->copy_epoch = 0;
  cudaError_t e = launch_slots_import(c.sc.amax_w, c.epoch, n, master_amax_in, stream);
  if (e == cudaSuccess)
    e = launch_step_w8(c.descs, c.chunks + ws->step_nchunks, ws->step_nchunks_o3,
                       c.sc, c.epoch, info->step_w8, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, "fp8_adam_step_copy: launch");
  return FP8OPT_OK;
}

extern "C" int fp8_adamw_step(const fp8opt_param* params, int n, float lr,
                              float beta1, float beta2, float eps, float wd,
                              int64_t step, float inv_loss_scale, int* found_inf,
                              uint32_t* found_inf_dev, void* stream_ptr) {
  return adam_step("fp8_adamw_step", false, params, n, lr, beta1, beta2, eps, wd,
                   step, inv_loss_scale, found_inf, found_inf_dev, stream_ptr);
}

extern "C" int fp8_adam_step(const fp8opt_param* params, int n, float lr,
                             float beta1, float beta2, float eps, float wd,
                             int64_t step, float inv_loss_scale, int* found_inf,
                             uint32_t* found_inf_dev, void* stream_ptr) {
  return adam_step("fp8_adam_step", true, params, n, lr, beta1, beta2, eps, wd,
                   step, inv_loss_scale, found_inf, found_inf_dev, stream_ptr);
}

extern "C" int fp8_cast_adamw_step(const fp8opt_cast_item* grads,
                                   const fp8opt_param* params, int n, int fmt,
                                   float lr, float beta1, float beta2, float eps,
                                   float wd, int64_t step, float inv_loss_scale,
                                   int* found_inf, uint32_t* found_inf_dev,
                                   void* stream_ptr) {
  const char* fn = "fp8_cast_adamw_step";
  int st = check_cast_args(fn, grads, n, fmt);
  if (st == FP8OPT_OK) st = check_step_args(fn, params, n, step);
  if (st == FP8OPT_OK) st = check_takes_cast(fn, grads, params, n, fmt);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) return empty_step(fn, found_inf, found_inf_dev, stream);
  const StepScalars s =
      make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale, false);

  std::unique_lock<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if ((st = ensure_cast_tables(fn, ws, grads, n, stream)) != FP8OPT_OK) return st;
  if ((st = ensure_step_tables(fn, ws, params, n, stream)) != FP8OPT_OK) return st;

  // slots: [0, n) gradient amax, [n, 2n) amax of m, [2n, 3n) amax of the
  // master, [3n, 4n) max |g|, [4n] found_inf; saved: m_scale, v_bound
  uint32_t epoch = 0;
  cudaError_t e = prepare_slots(ws, 4 * (size_t)n + 1, stream, &epoch);
  if (e == cudaSuccess) e = ws->saved_scales.reserve(2 * (size_t)n * sizeof(float));
  if (e != cudaSuccess) return cuda_fail(e, "fp8_cast_adamw_step: workspace");
  unsigned long long* slots = static_cast<unsigned long long*>(ws->slots.ptr);
  StepScratch sc;
  sc.amax_m = slots + n;
  sc.amax_w = slots + 2 * (size_t)n;
  sc.amax_g = slots + 3 * (size_t)n;
  sc.found = slots + 4 * (size_t)n;
  sc.old_m_scale = static_cast<float*>(ws->saved_scales.ptr);
  sc.old_v_bound = sc.old_m_scale + n;
  const Chunk* chunks = static_cast<const Chunk*>(ws->step_chunks.ptr);
  e = launch_cast_step(static_cast<const CastDesc*>(ws->cast_descs.ptr),
                       static_cast<const StepDesc*>(ws->step_descs.ptr), chunks,
                       ws->step_nchunks, chunks + ws->step_nchunks,
                       ws->step_nchunks_o3, slots, sc, s, epoch, fmt,
                       found_inf_dev, info->cast_amax, info->cast_step,
                       info->step_update, info->step_update_var,
                       info->step_w8, ws->step_any_vs, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, "fp8_cast_adamw_step: launch");
  lock.unlock();   // before any wait for the stream
  if (found_inf != nullptr) return read_found(fn, sc.found, epoch, stream, found_inf);
  return FP8OPT_OK;
}

extern "C" int fp8_adam_step_dev(const fp8opt_param* params, int n, float beta1,
                                 float beta2, float eps, float wd, int l2,
                                 fp8opt_step_state* state,
                                 uint32_t* found_inf_dev, void* stream_ptr) {
  const char* fn = "fp8_adam_step_dev";
  int st = check_step_args(fn, params, n, 1);
  if (st == FP8OPT_OK) st = check_dev_state(fn, state);
  if (st == FP8OPT_OK && l2 != 0 && l2 != 1)
    st = fail(FP8OPT_ERR_ARG, std::string(fn) + ": l2 must be 0 or 1");
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  std::lock_guard<std::mutex> lock(g_mu);
  if (n == 0) {
    int dev = 0;
    DeviceInfo* info = nullptr;
    if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
    return empty_dev_step(fn, state, beta1, beta2, wd, l2 != 0, found_inf_dev,
                          workspace(dev, stream), stream);
  }
  StepCall c;
  if ((st = setup_step(fn, params, n, stream_ptr, false, true, &c)) != FP8OPT_OK)
    return st;
  Workspace* ws = c.ws;
  if (ws->step_nchunks == 0)
    return empty_dev_step(fn, state, beta1, beta2, wd, l2 != 0, found_inf_dev, ws,
                          stream);
  DevScalars* ds = nullptr;
  if ((st = dev_scalars_buf(fn, ws, &ds)) != FP8OPT_OK) return st;
  const StepScalars s = make_dev_scalars(beta1, beta2, eps, wd, l2 != 0, ds,
                                         reinterpret_cast<long long*>(&state->step));
  cudaError_t e = launch_step_scalars(reinterpret_cast<DevState*>(state), beta1,
                                      beta2, wd, l2 != 0, ds, false, stream);
  if (e == cudaSuccess)
    e = launch_step(c.descs, c.chunks, ws->step_nchunks,
                    c.chunks + ws->step_nchunks, ws->step_nchunks_o3, c.sc, s,
                    c.epoch, found_inf_dev, c.info->step_amax,
                    c.info->step_update, c.info->step_update_var,
                    c.info->step_w8, ws->step_any_vs, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  return FP8OPT_OK;
}

extern "C" int fp8_cast_adamw_step_dev(const fp8opt_cast_item* grads,
                                       const fp8opt_param* params, int n, int fmt,
                                       float beta1, float beta2, float eps,
                                       float wd, fp8opt_step_state* state,
                                       uint32_t* found_inf_dev, void* stream_ptr) {
  const char* fn = "fp8_cast_adamw_step_dev";
  int st = check_cast_args(fn, grads, n, fmt);
  if (st == FP8OPT_OK) st = check_step_args(fn, params, n, 1);
  if (st == FP8OPT_OK) st = check_takes_cast(fn, grads, params, n, fmt);
  if (st == FP8OPT_OK) st = check_dev_state(fn, state);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if (n == 0)
    return empty_dev_step(fn, state, beta1, beta2, wd, false, found_inf_dev, ws,
                          stream);
  if ((st = ensure_cast_tables(fn, ws, grads, n, stream)) != FP8OPT_OK) return st;
  if ((st = ensure_step_tables(fn, ws, params, n, stream)) != FP8OPT_OK) return st;
  if (ws->step_nchunks == 0)
    return empty_dev_step(fn, state, beta1, beta2, wd, false, found_inf_dev, ws,
                          stream);

  // slots as in fp8_cast_adamw_step
  uint32_t epoch = 0;
  cudaError_t e = prepare_slots(ws, 4 * (size_t)n + 1, stream, &epoch);
  if (e == cudaSuccess) e = ws->saved_scales.reserve(2 * (size_t)n * sizeof(float));
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": workspace").c_str());
  DevScalars* ds = nullptr;
  if ((st = dev_scalars_buf(fn, ws, &ds)) != FP8OPT_OK) return st;
  unsigned long long* slots = static_cast<unsigned long long*>(ws->slots.ptr);
  StepScratch sc;
  sc.amax_m = slots + n;
  sc.amax_w = slots + 2 * (size_t)n;
  sc.amax_g = slots + 3 * (size_t)n;
  sc.found = slots + 4 * (size_t)n;
  sc.old_m_scale = static_cast<float*>(ws->saved_scales.ptr);
  sc.old_v_bound = sc.old_m_scale + n;
  const StepScalars s = make_dev_scalars(beta1, beta2, eps, wd, false, ds,
                                         reinterpret_cast<long long*>(&state->step));
  const Chunk* chunks = static_cast<const Chunk*>(ws->step_chunks.ptr);
  e = launch_step_scalars(reinterpret_cast<DevState*>(state), beta1, beta2, wd,
                          false, ds, false, stream);
  if (e == cudaSuccess)
    e = launch_cast_step(static_cast<const CastDesc*>(ws->cast_descs.ptr),
                         static_cast<const StepDesc*>(ws->step_descs.ptr), chunks,
                         ws->step_nchunks, chunks + ws->step_nchunks,
                         ws->step_nchunks_o3, slots, sc, s, epoch, fmt,
                         found_inf_dev, info->cast_amax, info->cast_step,
                         info->step_update, info->step_update_var,
                         info->step_w8, ws->step_any_vs, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  return FP8OPT_OK;
}

// fp8_cast_adam_step_clipped, and with state set its device-resident form
// (lr, step and inv_loss_scale from *state; host outputs not allowed).
static int cast_adam_clipped(const char* fn, const fp8opt_cast_item* grads,
                             const fp8opt_param* params, int n, int fmt, float lr,
                             float beta1, float beta2, float eps, float wd,
                             int64_t step, float inv_loss_scale, int l2,
                             float max_grad_norm, double* grad_norm,
                             float* grad_norm_dev, int* found_inf,
                             uint32_t* found_inf_dev, fp8opt_step_state* state,
                             void* stream_ptr) {
  if (l2 != 0 && l2 != 1) return fail(FP8OPT_ERR_ARG, std::string(fn) + ": l2 must be 0 or 1");
  if (std::isnan(max_grad_norm))
    return fail(FP8OPT_ERR_ARG, std::string(fn) + ": max_grad_norm is NaN");
  int st = check_cast_args(fn, grads, n, fmt);
  if (st == FP8OPT_OK) st = check_step_args(fn, params, n, state ? 1 : step);
  if (st == FP8OPT_OK) st = check_takes_cast(fn, grads, params, n, fmt);
  if (st == FP8OPT_OK && state != nullptr) st = check_dev_state(fn, state);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0 && state == nullptr) {
    if (grad_norm != nullptr) *grad_norm = 0.0;
    if (grad_norm_dev != nullptr) {
      cudaError_t e = cudaMemsetAsync(grad_norm_dev, 0, sizeof(float), stream);
      if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": norm_dev").c_str());
    }
    return empty_step(fn, found_inf, found_inf_dev, stream);
  }

  std::unique_lock<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if (n > 0) {
    if ((st = ensure_cast_tables(fn, ws, grads, n, stream)) != FP8OPT_OK) return st;
    if ((st = ensure_step_tables(fn, ws, params, n, stream)) != FP8OPT_OK) return st;
  }
  if (state != nullptr && (n == 0 || ws->step_nchunks == 0)) {
    if (grad_norm_dev != nullptr) {
      cudaError_t e = cudaMemsetAsync(grad_norm_dev, 0, sizeof(float), stream);
      if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": norm_dev").c_str());
    }
    return empty_dev_step(fn, state, beta1, beta2, wd, l2 != 0, found_inf_dev, ws,
                          stream);
  }
  StepScalars s;
  const float* ils_dev = nullptr;
  DevScalars* ds = nullptr;
  if (state != nullptr) {
    if ((st = dev_scalars_buf(fn, ws, &ds)) != FP8OPT_OK) return st;
    s = make_dev_scalars(beta1, beta2, eps, wd, l2 != 0, ds,
                         reinterpret_cast<long long*>(&state->step));
    ils_dev = &ds->ils;
  } else {
    s = make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale, l2 != 0);
  }

  // slots: [0, n) gradient amax, then the step's [n, 4n + 1) (amax of m, of
  // the master, max |g|, found_inf); norm: sums, terms, norm, clip
  uint32_t epoch = 0;
  cudaError_t e = prepare_slots(ws, 4 * (size_t)n + 1, stream, &epoch);
  if (e == cudaSuccess) e = ws->saved_scales.reserve(2 * (size_t)n * sizeof(float));
  const size_t sum_bytes = 2 * (size_t)n * sizeof(unsigned long long);
  if (e == cudaSuccess)
    e = ws->norm_buf.reserve(sum_bytes + (size_t)n * sizeof(double) + 16);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws->norm_buf.ptr, 0, sum_bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": workspace").c_str());
  unsigned long long* slots = static_cast<unsigned long long*>(ws->slots.ptr);
  StepScratch sc;
  sc.amax_m = slots + n;
  sc.amax_w = slots + 2 * (size_t)n;
  sc.amax_g = slots + 3 * (size_t)n;
  sc.found = slots + 4 * (size_t)n;
  sc.old_m_scale = static_cast<float*>(ws->saved_scales.ptr);
  sc.old_v_bound = sc.old_m_scale + n;
  char* nb = static_cast<char*>(ws->norm_buf.ptr);
  unsigned long long* sums = reinterpret_cast<unsigned long long*>(nb);
  double* terms = reinterpret_cast<double*>(nb + sum_bytes);
  double* norm = terms + n;
  float* clip = reinterpret_cast<float*>(norm + 1);
  const CastDesc* cdescs = static_cast<const CastDesc*>(ws->cast_descs.ptr);
  const StepDesc* sdescs = static_cast<const StepDesc*>(ws->step_descs.ptr);
  const Chunk* cchunks = static_cast<const Chunk*>(ws->cast_chunks.ptr);
  const Chunk* schunks = static_cast<const Chunk*>(ws->step_chunks.ptr);
  LaunchMark mark = launch_mark();
  // the norm only when it clips or is asked for (Adam with L2 decay alone
  // takes the fused cast and step of fp8_cast_adamw_step)
  const bool want_norm = max_grad_norm > 0.0f || grad_norm != nullptr ||
                         grad_norm_dev != nullptr;
  if (state != nullptr)
    e = launch_step_scalars(reinterpret_cast<DevState*>(state), beta1, beta2, wd,
                            l2 != 0, ds, false, stream);
  if (!want_norm) {
    // the cast's encode pass fused with the step's first pass (on the step's
    // chunk table, as fp8_cast_adamw_step), then the update
    if (e == cudaSuccess)
      e = launch_cast_step(cdescs, sdescs, schunks, ws->step_nchunks,
                           schunks + ws->step_nchunks, ws->step_nchunks_o3, slots,
                           sc, s, epoch, fmt, found_inf_dev, info->cast_amax,
                           info->cast_step, info->step_update,
                           info->step_update_var, info->step_w8,
                           ws->step_any_vs, stream, mark);
  } else {
    if (e == cudaSuccess)
      e = launch_cast_amax(cdescs, cchunks, ws->cast_nchunks, slots, epoch,
                           info->cast_amax, stream, mark);
    if (e == cudaSuccess)
      e = launch_cast_encode_sq(cdescs, cchunks, ws->cast_nchunks, slots, epoch,
                                fmt, info->cast_encode_sq[fmt], sums, sc.found,
                                inv_loss_scale, ils_dev, stream, mark);
    if (e == cudaSuccess)
      e = launch_norm_finish(sdescs, n, inv_loss_scale, ils_dev, sums, sc.found,
                             epoch, terms, max_grad_norm, norm, clip,
                             grad_norm_dev, stream, mark);
    if (max_grad_norm > 0.0f) s.clip = clip;
    if (e == cudaSuccess)
      e = launch_step(sdescs, schunks, ws->step_nchunks, schunks + ws->step_nchunks,
                      ws->step_nchunks_o3, sc, s, epoch, found_inf_dev,
                      info->step_amax, info->step_update,
                      info->step_update_var, info->step_w8, ws->step_any_vs,
                      stream, mark);
  }
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  lock.unlock();   // before any wait for the stream
  if (found_inf != nullptr || grad_norm != nullptr)
    return read_results(fn, sc.found, epoch, norm, stream, found_inf, grad_norm);
  return FP8OPT_OK;
}

extern "C" int fp8_cast_adam_step_clipped(
    const fp8opt_cast_item* grads, const fp8opt_param* params, int n, int fmt,
    float lr, float beta1, float beta2, float eps, float wd, int64_t step,
    float inv_loss_scale, int l2, float max_grad_norm, double* grad_norm,
    float* grad_norm_dev, int* found_inf, uint32_t* found_inf_dev,
    void* stream_ptr) {
  return cast_adam_clipped("fp8_cast_adam_step_clipped", grads, params, n, fmt, lr,
                           beta1, beta2, eps, wd, step, inv_loss_scale, l2,
                           max_grad_norm, grad_norm, grad_norm_dev, found_inf,
                           found_inf_dev, nullptr, stream_ptr);
}

extern "C" int fp8_cast_adam_step_clipped_dev(
    const fp8opt_cast_item* grads, const fp8opt_param* params, int n, int fmt,
    float beta1, float beta2, float eps, float wd, int l2, float max_grad_norm,
    fp8opt_step_state* state, float* grad_norm_dev, uint32_t* found_inf_dev,
    void* stream_ptr) {
  const char* fn = "fp8_cast_adam_step_clipped_dev";
  const int st = check_dev_state(fn, state);   // NULL would mean the host form
  if (st != FP8OPT_OK) return st;
  return cast_adam_clipped(fn, grads, params, n, fmt,
                           0.0f, beta1, beta2, eps, wd, 1, 1.0f, l2,
                           max_grad_norm, nullptr, grad_norm_dev, nullptr,
                           found_inf_dev, state, stream_ptr);
}

extern "C" const char* fp8opt_strerror(int status) {
  switch (status) {
    case FP8OPT_OK: return "success";
    case FP8OPT_ERR_ARG: return "invalid argument";
    case FP8OPT_ERR_UNSUPPORTED: return "unsupported format or element type";
    case FP8OPT_ERR_CUDA: return "CUDA error";
    case FP8OPT_ERR_LIMIT: return "size above a fixed maximum";
    default: return "unknown status";
  }
}

extern "C" const char* fp8opt_last_error(void) { return t_last_error.c_str(); }

extern "C" int fp8opt_timing_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (on) {
    cudaError_t e = timing_collect();
    if (e != cudaSuccess) return cuda_fail(e, "fp8opt_timing_enable");
    for (int k = 0; k < kNumKernels; ++k) {
      g_timing.launches[k] = 0;
      g_timing.ms[k] = 0.0;
    }
  }
  g_timing.on = on != 0;
  return FP8OPT_OK;
}

extern "C" int fp8opt_timing_read(const char* kernel, int* launches,
                                  double* total_ms) {
  if (kernel == nullptr || launches == nullptr || total_ms == nullptr)
    return fail(FP8OPT_ERR_ARG, "fp8opt_timing_read: NULL argument");
  int k = 0;
  while (k < kNumKernels && std::strcmp(kKernelNames[k], kernel) != 0) ++k;
  if (k == kNumKernels)
    return fail(FP8OPT_ERR_ARG, std::string("fp8opt_timing_read: unknown kernel ") + kernel);
  std::lock_guard<std::mutex> lock(g_mu);
  cudaError_t e = timing_collect();
  if (e != cudaSuccess) return cuda_fail(e, "fp8opt_timing_read");
  *launches = g_timing.launches[k];
  *total_ms = g_timing.ms[k];
  return FP8OPT_OK;
}

extern "C" void fp8opt_release_stream(void* stream_ptr) {
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  auto it = g_ws.find(std::make_pair(dev, static_cast<cudaStream_t>(stream_ptr)));
  if (it == g_ws.end()) return;
  it->second->release();
  delete it->second;
  g_ws.erase(it);
}

extern "C" void fp8opt_release(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto& kv : g_ws) {
    cudaSetDevice(kv.first.first);
    kv.second->release();
    delete kv.second;
  }
  g_ws.clear();
  if (cur >= 0) cudaSetDevice(cur);
}
