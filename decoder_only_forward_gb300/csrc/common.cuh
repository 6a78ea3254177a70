// Shared device helpers for the decoder kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dec {

// Device error word bits (DeviceState::err).
constexpr unsigned ERR_TIMEOUT = 1u;   // a bounded wait gave up
constexpr unsigned ERR_TOKEN = 2u;     // a device-side token outside [0, vocab)
constexpr unsigned ERR_LAYOUT = 4u;    // a kernel's shared-memory window could not hold its tile layout

// Per-handle device-resident step state.  Kernels of a decode step read the
// position and token from here, so one captured CUDA graph serves every step.
struct DeviceState {
  int32_t pos;        // absolute position of the token being decoded
  int32_t token;      // token id being decoded
  unsigned err;       // ERR_* bits, sticky until the host clears them
  unsigned where;     // identifier of the first wait that timed out
  unsigned counters[256];  // last-CTA-done counters (split combine, argmax), self-resetting
};

// CNT_ATTN + kv head index (< 193); CNT_MK_*: grid barrier of the persistent decode kernel.
enum CounterSlot { CNT_ARGMAX = 0, CNT_ATTN = 1, CNT_MK_BAR = 240, CNT_MK_GEN = 241 };

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 16-byte streaming load that bypasses L1 (weights are read once per step).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Element type traits: how many elements one 16-byte chunk holds, and the
// widening of a chunk to fp32.
template <typename T> struct Chunk;
template <> struct Chunk<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void widen(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
};
template <> struct Chunk<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void widen(const uint4& u, float* f) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Spin budget of every bounded device wait: about two seconds.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor still runs.  Everything
// before pdl_wait() must touch only data no in-flight kernel writes (weights,
// KV of earlier steps); pdl_wait() returns once the predecessor grid has
// completed and its writes are visible.  Without the launch attribute both
// are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// 16-byte asynchronous global -> shared copies (L2 only).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void raise_error(DeviceState* st, unsigned bits, unsigned where) {
  if (atomicOr(&st->err, bits) == 0u) st->where = where;
}

}  // namespace dec
