// dec_attend_noalloc: dec_attend without a caller-provided scratch buffer.
//
// Some callers cannot obtain device memory of their own: a plug-in hosted by a
// framework whose pooled allocator has already reserved the GPU's memory, or
// code on a latency-critical path where cudaMalloc (which can synchronise the
// device and can fail under memory pressure) is not allowed.  For them the
// split-K partials and the step counters of the attention kernel live in one
// fixed array in device memory, compiled into this library.
#include <mutex>

#include "runtime.h"

namespace {

// The whole scratch of one call: step state + split-K partials.  1 MiB covers
// e.g. 32 query heads x 32 splits x head_dim 128.  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) unsigned char g_attend_scratch[kNoAllocScratchBytes];

// Device address of g_attend_scratch per device.  In host code the symbol is
// only a host-side stand-in, never a device address, so it is translated with
// cudaGetSymbolAddress while that device is current.  The address belongs to the
// device's current context: after cudaDeviceReset (or a released and re-created
// primary context) the module is loaded again and the array may move, so each
// cached address is kept with the context it was resolved in and looked up again
// when the context changes.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
void* g_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = int (*)(void**);   // cuCtxGetCurrent(CUcontext*) -> CUresult

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return cudaErrorDeviceUninitialized;
  void* ctx = nullptr;   // stays NULL until the runtime has made a context current
  if (get(&ctx) != 0) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_addr[dev] || g_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attend_scratch);   // makes the device's primary context current
    if (e != cudaSuccess) return e;
    if (get(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

using namespace dec;

extern "C" dec_status dec_attend_noalloc(const float* q, const void* k, const void* v, int32_t n_heads,
                                         int32_t n_kv_heads, int32_t head_dim, int32_t max_seq,
                                         int32_t sliding_window, int32_t kv_dtype, int32_t pos, float* out,
                                         void* cuda_stream) {
  AttendLayout lay;
  const char* why = nullptr;
  if (!attend_check(q, k, v, out, n_heads, n_kv_heads, head_dim, max_seq, sliding_window, kv_dtype, pos, lay,
                    &why)) {
    set_global_error(why);
    return DEC_EINVAL;
  }
  if (lay.total > kNoAllocScratchBytes) {
    set_global_error("dec_attend_noalloc: these sizes need more than the library's fixed 1 MiB scratch; "
                     "use dec_attend with a caller buffer");
    return DEC_EINVAL;
  }
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) {
    set_global_error(cudaGetErrorString(e));
    return DEC_ECUDA;
  }
  // launch_attend's first kernel rewrites the position and zeroes the
  // counters, so nothing left by an earlier call is read.
  char* b = (char*)base;
  launch_attend(q, k, v, n_heads, n_kv_heads, head_dim, max_seq, sliding_window, kv_dtype, pos, lay.nsplit,
                (DeviceState*)b, (float*)(b + lay.part_offset), out, (cudaStream_t)cuda_stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error(cudaGetErrorString(e));
    return DEC_ECUDA;
  }
  return DEC_OK;
}
