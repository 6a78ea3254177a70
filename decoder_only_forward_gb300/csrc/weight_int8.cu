// 8-bit projection weights (Pantheon "Llama Forward Pass", weight modes: the
// projections stay quantised and are expanded a block at a time).  A weight row
// is stored in groups of 32 input columns, each as round(w / s) with one float32
// scale s = max|w| / 127 -- the int8 rule rml "The decoder" gives for the K/V
// cache, applied to weight rows.  The decision is taken in float32: w as f32,
// s = max|w| / 127 and w / s each one correctly rounded f32 operation, round =
// halves away from zero, codes clamped to [-127, 127]; an all-zero group keeps
// s = 0 and codes 0.  The forward pass uses float32(code * s).
#include <stdint.h>

#include "runtime.h"

namespace dec {

constexpr int WQ_GROUP = 32;

// One warp per 32-column group (lane = column): max |w| over the group by xor
// shuffles, then each lane's code; lane 0 stores the scale.
template <typename T>
__global__ void __launch_bounds__(256) k_weight_quant(const T* __restrict__ w, size_t groups, int8_t* __restrict__ codes,
                                                      float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
  for (size_t g = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < groups; g += warps) {
    const float x = to_f32(w[g * WQ_GROUP + lane]);
    float m = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = __fdiv_rn(m, 127.0f);
    int q = 0;
    if (s > 0.f) {
      q = (int)roundf(__fdiv_rn(x, s));
      q = q > 127 ? 127 : (q < -127 ? -127 : q);
    }
    codes[g * WQ_GROUP + lane] = (int8_t)q;
    if (lane == 0) scales[g] = s;
  }
}

// Expansion for the row GEMMs: element i -> w = f32(code * s), then either the
// bf16 pair hi = bf16(w), lo = bf16(w - hi) or w itself.  Four elements per
// thread and iteration.
__global__ void __launch_bounds__(256) k_weight_dequant_hilo(const int8_t* __restrict__ codes,
                                                             const float* __restrict__ scales, size_t n4,
                                                             __nv_bfloat16* __restrict__ hi,
                                                             __nv_bfloat16* __restrict__ lo) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const char4 c = reinterpret_cast<const char4*>(codes)[i];
    const float s = scales[(4 * i) / WQ_GROUP];
    const float w0 = __fmul_rn((float)c.x, s), w1 = __fmul_rn((float)c.y, s);
    const float w2 = __fmul_rn((float)c.z, s), w3 = __fmul_rn((float)c.w, s);
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(w0, w1), h23 = __floats2bfloat162_rn(w2, w3);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(w0 - __low2float(h01), w1 - __high2float(h01));
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(w2 - __low2float(h23), w3 - __high2float(h23));
    reinterpret_cast<__nv_bfloat162*>(hi)[2 * i] = h01;
    reinterpret_cast<__nv_bfloat162*>(hi)[2 * i + 1] = h23;
    reinterpret_cast<__nv_bfloat162*>(lo)[2 * i] = l01;
    reinterpret_cast<__nv_bfloat162*>(lo)[2 * i + 1] = l23;
  }
}

__global__ void __launch_bounds__(256) k_weight_dequant_f32(const int8_t* __restrict__ codes,
                                                            const float* __restrict__ scales, size_t n4,
                                                            float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const char4 c = reinterpret_cast<const char4*>(codes)[i];
    const float s = scales[(4 * i) / WQ_GROUP];
    reinterpret_cast<float4*>(out)[i] =
        make_float4(__fmul_rn((float)c.x, s), __fmul_rn((float)c.y, s), __fmul_rn((float)c.z, s),
                    __fmul_rn((float)c.w, s));
  }
}

static int grid_for(size_t items, int per_block) {
  const size_t b = (items + per_block - 1) / per_block;
  const size_t cap = (size_t)device_sm_count() * 8;
  return (int)(b < 1 ? 1 : (b > cap ? cap : b));
}

cudaError_t launch_weight_quant(const void* w, bool w_bf16, size_t rows, int cols, int8_t* codes, float* scales,
                                cudaStream_t s) {
  const size_t groups = rows * (size_t)(cols / WQ_GROUP);
  if (groups == 0) return cudaSuccess;
  const int grid = grid_for(groups, 8);
  if (w_bf16) k_weight_quant<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)w, groups, codes, scales);
  else k_weight_quant<float><<<grid, 256, 0, s>>>((const float*)w, groups, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_weight_dequant_hilo(const QMat& q, size_t rows, int cols, __nv_bfloat16* hi, __nv_bfloat16* lo,
                                       cudaStream_t s) {
  const size_t n4 = rows * (size_t)cols / 4;
  k_weight_dequant_hilo<<<grid_for(n4, 256), 256, 0, s>>>(q.codes, q.scales, n4, hi, lo);
  return cudaGetLastError();
}

cudaError_t launch_weight_dequant_f32(const QMat& q, size_t rows, int cols, float* out, cudaStream_t s) {
  const size_t n4 = rows * (size_t)cols / 4;
  k_weight_dequant_f32<<<grid_for(n4, 256), 256, 0, s>>>(q.codes, q.scales, n4, out);
  return cudaGetLastError();
}

}  // namespace dec

using namespace dec;

extern "C" dec_status dec_weight_quantize_int8(const void* w, int32_t weight_dtype, int64_t rows, int32_t cols,
                                               int8_t* codes, float* scales, void* cuda_stream) {
  if (!w || !codes || !scales || rows <= 0 || cols <= 0 || cols % WQ_GROUP != 0 ||
      (weight_dtype != DEC_F32 && weight_dtype != DEC_BF16)) {
    set_global_error("dec_weight_quantize_int8: NULL pointer, non-positive size, cols not a multiple of 32, "
                     "or weight_dtype not DEC_F32 / DEC_BF16");
    return DEC_EINVAL;
  }
  const cudaError_t e = launch_weight_quant(w, weight_dtype == DEC_BF16, (size_t)rows, cols, codes, scales,
                                            (cudaStream_t)cuda_stream);
  if (e != cudaSuccess) {
    set_global_error(cudaGetErrorString(e));
    return DEC_ECUDA;
  }
  return DEC_OK;
}
