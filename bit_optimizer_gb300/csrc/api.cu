// The libfp8opt C ABI (include/fp8opt.h): argument checks, the per-(device,
// stream) workspace with its cached tensor and chunk tables, the per-call
// scalars, and the kernel launches.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

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
                        int grid_w8, bool any_vs, cudaStream_t stream,
                        LaunchMark mark);
cudaError_t step_occupancy(int* amax_per_sm, int* update_per_sm, int* w8_per_sm);
cudaError_t launch_cast_step(const CastDesc* cdescs, const StepDesc* sdescs,
                             const Chunk* chunks, uint32_t nchunks,
                             const Chunk* chunks_o3, uint32_t nchunks_o3,
                             unsigned long long* gslots, const StepScratch& sc,
                             const StepScalars& s, uint32_t epoch, int fmt,
                             uint32_t* found_dev, int grid_amax, int grid_fused,
                             int grid_update, int grid_w8, bool any_vs,
                             cudaStream_t stream, LaunchMark mark);
cudaError_t cast_step_occupancy(int* per_sm);

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

// A device buffer that only grows.
struct DevBuf {
  void* ptr = nullptr;
  size_t cap = 0;
  cudaError_t reserve(size_t bytes) {
    if (bytes <= cap) return cudaSuccess;
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
  int step_amax = 0, step_update = 0, step_w8 = 0;
  int cast_step = 0;
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
  // cast tables
  std::vector<fp8opt_cast_item> cast_key;
  DevBuf cast_descs, cast_chunks;
  uint32_t cast_nchunks = 0;
  // step tables
  std::vector<fp8opt_param> step_key;
  DevBuf step_descs, step_chunks;
  uint32_t step_nchunks = 0, step_nchunks_o3 = 0;
  bool step_any_vs = false;   // some record has a scaled second moment
  bool have_cast = false, have_step = false;

  void release() {
    slots.release();
    saved_scales.release();
    cast_descs.release();
    cast_chunks.release();
    step_descs.release();
    step_chunks.release();
    cast_key.clear();
    step_key.clear();
    have_cast = have_step = false;
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
  if ((e = step_occupancy(&a, &b, &c)) != cudaSuccess) return e;
  info.step_amax = info.sms * (a > 0 ? a : 1);
  info.step_update = info.sms * (b > 0 ? b : 1);
  info.step_w8 = info.sms * (c > 0 ? c : 1);
  if ((e = cast_step_occupancy(&a)) != cudaSuccess) return e;
  info.cast_step = info.sms * (a > 0 ? a : 1);
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

// `words` tagged slots for this call, zeroed when (re)allocated or when the
// epoch wraps; returns the call's epoch.
cudaError_t prepare_slots(Workspace* ws, size_t words, cudaStream_t stream,
                          uint32_t* epoch_out) {
  const size_t bytes = words * sizeof(unsigned long long);
  bool fresh = false;
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
    cudaError_t e = cudaMemsetAsync(ws->slots.ptr, 0, ws->slots.cap, stream);
    if (e != cudaSuccess) return e;
  }
  *epoch_out = ws->epoch;
  return cudaSuccess;
}

// ------------------------------------------------------- per-kernel timing

const char* const kKernelNames[kNumKernels] = {
    "cast_amax", "cast_encode", "step_amax", "step_update", "step_w8",
    "cast_step_amax"};

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
  cudaEvent_t e = timing_event();
  cudaEventRecord(e, stream);
  if (!end) {
    g_timing.open_start[kernel] = e;
  } else {
    g_timing.pending.push_back({kernel, g_timing.open_start[kernel], e});
    g_timing.open_start[kernel] = nullptr;
  }
}

LaunchMark launch_mark() { return g_timing.on ? timing_mark : nullptr; }

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

uint32_t chunks_of(int64_t numel) {
  return numel == 0 ? 1u : (uint32_t)((numel + kChunkElems - 1) / kChunkElems);
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

// Per-call scalars: the bias corrections 1 - beta^t in double, entering only
// through lr / bc1 and 1 / sqrt(bc2), each rounded to fp32 once.
StepScalars make_scalars(float lr, float beta1, float beta2, float eps, float wd,
                         int64_t step, float inv_loss_scale, bool l2) {
  StepScalars s;
  const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
  const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
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
  return s;
}

// The workspace's cast tables for this item list (uploaded when the list
// differs from the cached one).
int ensure_cast_tables(const char* fn, Workspace* ws,
                       const fp8opt_cast_item* items, int n,
                       cudaStream_t stream) {
  if (ws->have_cast && same_list(ws->cast_key, items, n)) return FP8OPT_OK;
  std::vector<CastDesc> descs((size_t)n);
  std::vector<Chunk> chunks;
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += chunks_of(items[i].numel);
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
    for (uint32_t c = 0, nc = chunks_of(it.numel); c < nc; ++c)
      chunks.push_back(Chunk{(uint32_t)i, c});
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
  std::vector<StepDesc> descs((size_t)n);
  std::vector<Chunk> chunks, chunks_o3;
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += 2 * (size_t)chunks_of(params[i].numel);
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
    for (uint32_t c = 0, nc = chunks_of(p.numel); c < nc; ++c) {
      chunks.push_back(Chunk{(uint32_t)i, c});
      if (d.o3) chunks_o3.push_back(Chunk{(uint32_t)i, c});
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
  for (int i = 0; i < n; ++i) ws->step_any_vs |= params[i].v_bound != nullptr;
  ws->have_step = true;
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

// Waits for the stream and reads this call's found_inf word.
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

// The two step entry points: AdamW (l2 false) and Adam with L2 decay.
int adam_step(const char* fn, bool l2, const fp8opt_param* params, int n,
              float lr, float beta1, float beta2, float eps, float wd,
              int64_t step, float inv_loss_scale, int* found_inf,
              uint32_t* found_inf_dev, void* stream_ptr) {
  int st = check_step_args(fn, params, n, step);
  if (st != FP8OPT_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) return empty_step(fn, found_inf, found_inf_dev, stream);
  const StepScalars s =
      make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale, l2);

  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  DeviceInfo* info = nullptr;
  if ((st = current_device_and_info(&dev, &info)) != FP8OPT_OK) return st;
  Workspace* ws = workspace(dev, stream);
  if ((st = ensure_step_tables(fn, ws, params, n, stream)) != FP8OPT_OK) return st;

  uint32_t epoch = 0;
  // slots: [0, n) amax of m, [n, 2n) amax of the master, [2n, 3n) max |g|,
  // [3n] found_inf; saved: [0, n) m_scale, [n, 2n) v_bound
  cudaError_t e = prepare_slots(ws, 3 * (size_t)n + 1, stream, &epoch);
  if (e == cudaSuccess) e = ws->saved_scales.reserve(2 * (size_t)n * sizeof(float));
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": workspace").c_str());
  unsigned long long* slots = static_cast<unsigned long long*>(ws->slots.ptr);
  StepScratch sc;
  sc.amax_m = slots;
  sc.amax_w = slots + n;
  sc.amax_g = slots + 2 * (size_t)n;
  sc.found = slots + 3 * (size_t)n;
  sc.old_m_scale = static_cast<float*>(ws->saved_scales.ptr);
  sc.old_v_bound = sc.old_m_scale + n;
  const Chunk* chunks = static_cast<const Chunk*>(ws->step_chunks.ptr);
  e = launch_step(static_cast<const StepDesc*>(ws->step_descs.ptr), chunks,
                  ws->step_nchunks, chunks + ws->step_nchunks, ws->step_nchunks_o3,
                  sc, s, epoch, found_inf_dev, info->step_amax, info->step_update,
                  info->step_w8, ws->step_any_vs, stream, launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, (std::string(fn) + ": launch").c_str());
  if (found_inf != nullptr) return read_found(fn, sc.found, epoch, stream, found_inf);
  return FP8OPT_OK;
}

}  // namespace
}  // namespace fp8opt

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
  if (st != FP8OPT_OK) return st;
  for (int i = 0; i < n; ++i) {
    const fp8opt_param& p = params[i];
    if (p.g != grads[i].codes || p.g_scale != grads[i].scale ||
        p.numel != grads[i].numel || p.g_fmt != fmt)
      return fail(FP8OPT_ERR_ARG, std::string(fn) + ": param " + std::to_string(i) +
                                      " does not take item " + std::to_string(i) +
                                      "'s codes, scale, numel and format");
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (n == 0) return empty_step(fn, found_inf, found_inf_dev, stream);
  const StepScalars s =
      make_scalars(lr, beta1, beta2, eps, wd, step, inv_loss_scale, false);

  std::lock_guard<std::mutex> lock(g_mu);
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
                       info->step_update, info->step_w8, ws->step_any_vs, stream,
                       launch_mark());
  if (e != cudaSuccess) return cuda_fail(e, "fp8_cast_adamw_step: launch");
  if (found_inf != nullptr) return read_found(fn, sc.found, epoch, stream, found_inf);
  return FP8OPT_OK;
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
