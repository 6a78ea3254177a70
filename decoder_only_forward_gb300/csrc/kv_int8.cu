// int8 K/V cache rows (rml "The decoder", KV cache): each group of G channels
// (G the largest power of two dividing head_dim, at most 32, so a group never
// spans two heads) is stored as round(x / s) with one f32 scale
// s = max|x| / 127.  A ring row is [scales: kd/G f32, padded to 16 bytes]
// [codes: kd int8, padded to 16 bytes]; attention reads code * s.
//
// The decision is taken in f32 with correctly rounded operations: s =
// max|x| / 127, the quotient x / s, C round() (halves away from zero), codes
// clamped to [-127, 127]; an all-zero group keeps s = 0 and codes 0.
#include "runtime.h"

namespace dec {

// Rows of n x kd f32 (src_k, src_v) -> int8 ring rows.  Row r goes to ring row
// dst_rows[r] when given, else to the slot of position pos0 + r (pos % max_seq
// under a window); rows below t_first are not stored (a later row of the same
// call owns their slot).  rt_k / rt_v (nullable) receive the values read back.
// One warp per 32 channels of one row; the lanes of a group reduce max|x| with
// xor shuffles.  blockIdx.z: 0 = K, 1 = V.
// src and rt may be the same rows (read back in place): each element is read
// once, before its own store.
__global__ void __launch_bounds__(256) k_kv_quant(const float* src_k, const float* src_v,
                                                  int n, int kd, int G, const int32_t* __restrict__ dst_rows,
                                                  const KvPaging pg, int seq, int pos0, int sliding, int max_seq,
                                                  int t_first,
                                                  char* __restrict__ ring_k, char* __restrict__ ring_v,
                                                  int row_bytes, int code_off, float* rt_k, float* rt_v) {
  const int lane = threadIdx.x & 31;
  const int ch = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32 + lane;
  const int r = blockIdx.y;
  const bool is_v = blockIdx.z != 0;
  if (ch - lane >= kd) return;   // whole warp past the row (kd is a multiple of 32 or of G <= 32)
  const float* src = is_v ? src_v : src_k;
  const bool in = ch < kd;
  const float x = in ? src[(size_t)r * kd + ch] : 0.f;
  float m = fabsf(x);
  for (int o = G >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s = __fdiv_rn(m, 127.0f);
  int code = 0;
  if (s > 0.f) {
    const float q = roundf(__fdiv_rn(x, s));
    code = (int)fminf(fmaxf(q, -127.0f), 127.0f);
  }
  if (!in) return;
  float* rt = is_v ? rt_v : rt_k;
  if (rt) rt[(size_t)r * kd + ch] = __fmul_rn((float)code, s);
  if (r < t_first) return;
  long long row;
  if (dst_rows) {
    row = dst_rows[r];
  } else {
    const int p = pos0 + r;
    row = kv_phys_row(pg, seq, sliding > 0 ? p % max_seq : p);
  }
  char* dst = (is_v ? ring_v : ring_k) + row * (long long)row_bytes;
  dst[code_off + ch] = (char)(signed char)code;
  if (ch % G == 0) reinterpret_cast<float*>(dst)[ch / G] = s;
}

// Ring rows of positions h0 .. h0 + count - 1 (slot p % max_seq) -> f32 rows,
// read back as code * s.
__global__ void k_kv_gather_i8(const char* __restrict__ ring_k, const char* __restrict__ ring_v, const KvPaging pg,
                               int seq, int max_seq, int kd, int G, int row_bytes, int code_off, int h0, int count,
                               float* __restrict__ lin_k, float* __restrict__ lin_v) {
  const size_t total = (size_t)count * kd;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / kd), c = (int)(i % kd);
    const size_t row = (size_t)kv_phys_row(pg, seq, (h0 + r) % max_seq) * row_bytes;
    const float sk = reinterpret_cast<const float*>(ring_k + row)[c / G];
    const float sv = reinterpret_cast<const float*>(ring_v + row)[c / G];
    lin_k[i] = __fmul_rn((float)(signed char)ring_k[row + code_off + c], sk);
    lin_v[i] = __fmul_rn((float)(signed char)ring_v[row + code_off + c], sv);
  }
}

void launch_kv_quant(const dec_config& c, const float* src_k, const float* src_v, int n, const int32_t* dst_rows,
                     const KvPaging& pg, int seq, int pos0, int t_first, void* ring_k, void* ring_v, float* rt_k,
                     float* rt_v, cudaStream_t s, int planes) {
  const KvRowLayout L = kv_row_layout(c);
  const int kd = c.n_kv_heads * c.head_dim;
  const int warps = 8;
  const dim3 grid((kd + 32 * warps - 1) / (32 * warps), n, planes);
  k_kv_quant<<<grid, 32 * warps, 0, s>>>(src_k, src_v, n, kd, L.group, dst_rows, pg, seq, pos0, c.sliding_window,
                                         c.max_seq, t_first, (char*)ring_k, (char*)ring_v, L.bytes, L.code_off, rt_k,
                                         rt_v);
}

void launch_kv_gather_i8(const dec_config& c, const void* ring_k, const void* ring_v, const KvPaging& pg, int seq,
                         int h0, int count, float* lin_k, float* lin_v, cudaStream_t s) {
  const KvRowLayout L = kv_row_layout(c);
  k_kv_gather_i8<<<device_sm_count(), 256, 0, s>>>((const char*)ring_k, (const char*)ring_v, pg, seq, c.max_seq,
                                     c.n_kv_heads * c.head_dim, L.group, L.bytes, L.code_off, h0, count, lin_k,
                                     lin_v);
}

__global__ void k_set_pages(int32_t* __restrict__ table, const __grid_constant__ PageSet ps) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < ps.n) table[ps.idx[i]] = ps.val[i];
}

void launch_set_pages(int32_t* table, const PageSet& ps, cudaStream_t s) {
  if (ps.n > 0) k_set_pages<<<1, 256, 0, s>>>(table, ps);
}

}  // namespace dec

using namespace dec;

// Quantises rows of K (or V) with the cache's kernel (see dec.h).
extern "C" dec_status dec_kv_quantize_int8(const float* x, int32_t n_rows, int32_t n_kv_heads, int32_t head_dim,
                                           void* out, void* cuda_stream) {
  if (!x || !out || n_rows <= 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim % 16 != 0 || n_rows > 65535) {
    set_global_error("dec_kv_quantize_int8: NULL pointer, non-positive size, head_dim not a multiple of 16, "
                     "or more than 65535 rows");
    return DEC_EINVAL;
  }
  dec_config c{};
  c.n_kv_heads = n_kv_heads;
  c.head_dim = head_dim;
  c.kv_dtype = DEC_I8;
  c.max_seq = n_rows;
  KvPaging pg{};
  pg.ring_rows = n_rows;
  launch_kv_quant(c, x, nullptr, n_rows, nullptr, pg, 0, 0, 0, out, nullptr, nullptr, nullptr,
                  (cudaStream_t)cuda_stream, 1);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error(cudaGetErrorString(e));
    return DEC_ECUDA;
  }
  return DEC_OK;
}
