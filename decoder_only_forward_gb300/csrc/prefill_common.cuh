// Epilogues shared by the prefill GEMMs (SIMT and tcgen05): every GEMM hands
// its accumulators over as pairs of adjacent output columns of one row.
#pragma once

#include "runtime.h"

namespace dec {

enum EpiMode : int {
  EPI_QKV = 0,     // +bias, adjacent-pair RoPE, q -> Q rows, k/v -> K/V rows (cache or linear scratch)
  EPI_RESID = 1,   // out[row][col] += v  (residual stream, f32)
  EPI_SWIGLU = 2,  // columns (2j, 2j+1) = (gate, up) -> act[row][j] = silu(gate) * up
  EPI_STORE = 3,   // out[row][col] = v (f32)
};

struct GemmEpi {
  int mode;
  int n_out;            // valid output columns (N)
  // EPI_RESID / EPI_STORE: f32 rows of n_out columns
  float* out_f32;
  // EPI_SWIGLU: rows of n_out/2 activations, bf16 when act_bf16 else f32;
  // with act_lo set, act holds bf16 hi and act_lo the bf16 remainder (a = hi + lo)
  void* act;
  int act_bf16;
  __nv_bfloat16* act_lo;
  // EPI_QKV
  const float* bias;      // nullable
  const float2* rope;     // [row][hd/2] (cos, sin) of the row's position
  int qd, kd, hd;
  void* q_out;            // [row][qd], bf16 when q_bf16 else f32
  int q_bf16;
  __nv_bfloat16* q_lo;    // with q_bf16: the bf16 remainder plane (q = hi + lo); nullable
  void* k_dst;            // K rows: row r goes to row (r + kv_row0), kd columns
  void* v_dst;
  int kv_bf16;
  int kv_row0;
  const int32_t* kv_rows;  // nullable: row r's K/V go to row kv_rows[r] instead of r + kv_row0
  // Grouped (MoE) GEMMs: rows of group g are [offset[g], offset[g] + count[g]).
  const int32_t* group_offset;   // nullable = one group of all rows
};

// Destination of an activation row buffer: f32, or a bf16 (hi, lo) pair of
// planes with value = hi + lo (the A operand of the tensor-core GEMMs).
struct RowOut {
  void* hi;
  __nv_bfloat16* lo;
  int f32;
};
__device__ __forceinline__ void row_store(const RowOut& o, size_t i, float v) {
  if (o.f32) {
    reinterpret_cast<float*>(o.hi)[i] = v;
  } else {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    reinterpret_cast<__nv_bfloat16*>(o.hi)[i] = h;
    if (o.lo) o.lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// Four consecutive values (i a multiple of 4).
__device__ __forceinline__ void row_store4(const RowOut& o, size_t i, float4 v) {
  if (o.f32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(o.hi) + i) = v;
  } else {
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
    uint2 hh;
    hh.x = *reinterpret_cast<const uint32_t*>(&h01);
    hh.y = *reinterpret_cast<const uint32_t*>(&h23);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(o.hi) + i) = hh;
    if (o.lo) {
      const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - __low2float(h01), v.y - __high2float(h01));
      const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - __low2float(h23), v.w - __high2float(h23));
      uint2 ll;
      ll.x = *reinterpret_cast<const uint32_t*>(&l01);
      ll.y = *reinterpret_cast<const uint32_t*>(&l23);
      *reinterpret_cast<uint2*>(o.lo + i) = ll;
    }
  }
}

template <typename T>
__device__ __forceinline__ void store_pair(T* p, float a, float b);
template <>
__device__ __forceinline__ void store_pair<float>(float* p, float a, float b) {
  *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16* p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// Applies the epilogue to columns (col, col+1) of global row `row`.  col is even.
__device__ __forceinline__ void epi_pair(const GemmEpi& e, int row, int col, float v0, float v1) {
  if (col >= e.n_out) return;
  switch (e.mode) {
    case EPI_RESID: {
      float* p = e.out_f32 + (size_t)row * e.n_out + col;
      if ((e.n_out & 1) == 0) {
        float2 x = *reinterpret_cast<float2*>(p);
        x.x += v0;
        x.y += v1;
        *reinterpret_cast<float2*>(p) = x;
      } else {   // odd rows: no 8-byte alignment, and the last column stands alone
        p[0] += v0;
        if (col + 1 < e.n_out) p[1] += v1;
      }
      break;
    }
    case EPI_STORE: {
      float* p = e.out_f32 + (size_t)row * e.n_out + col;
      if ((e.n_out & 1) == 0) {
        store_pair(p, v0, v1);
      } else {
        p[0] = v0;
        if (col + 1 < e.n_out) p[1] = v1;
      }
      break;
    }
    case EPI_SWIGLU: {
      const float a = silu_f(v0) * v1;
      const size_t o = (size_t)row * (e.n_out / 2) + (col >> 1);
      if (e.act_bf16) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(a);
        reinterpret_cast<__nv_bfloat16*>(e.act)[o] = hi;
        if (e.act_lo) e.act_lo[o] = __float2bfloat16_rn(a - __bfloat162float(hi));
      } else {
        reinterpret_cast<float*>(e.act)[o] = a;
      }
      break;
    }
    case EPI_QKV: {
      if (e.bias) {
        v0 += e.bias[col];
        v1 += e.bias[col + 1];
      }
      if (e.rope && col < e.qd + e.kd) {   // no table: q and k left unrotated (QK-norm comes first)
        const int d = (col < e.qd ? col : col - e.qd) % e.hd;
        const float2 cs = e.rope[(size_t)row * (e.hd / 2) + (d >> 1)];
        const float a = v0 * cs.x - v1 * cs.y;
        const float b = v0 * cs.y + v1 * cs.x;
        v0 = a;
        v1 = b;
      }
      if (col < e.qd) {
        const size_t o = (size_t)row * e.qd + col;
        if (e.q_bf16) {
          const __nv_bfloat162 hi = __floats2bfloat162_rn(v0, v1);
          *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(e.q_out) + o) = hi;
          if (e.q_lo)
            *reinterpret_cast<__nv_bfloat162*>(e.q_lo + o) =
                __floats2bfloat162_rn(v0 - __low2float(hi), v1 - __high2float(hi));
        } else {
          store_pair(reinterpret_cast<float*>(e.q_out) + o, v0, v1);
        }
      } else {
        const bool is_k = col < e.qd + e.kd;
        const size_t kr = e.kv_rows ? (size_t)e.kv_rows[row] : (size_t)(row + e.kv_row0);
        const size_t o = kr * e.kd + (is_k ? col - e.qd : col - e.qd - e.kd);
        void* dst = is_k ? e.k_dst : e.v_dst;
        if (e.kv_bf16) store_pair(reinterpret_cast<__nv_bfloat16*>(dst) + o, v0, v1);
        else store_pair(reinterpret_cast<float*>(dst) + o, v0, v1);
      }
      break;
    }
  }
}

}  // namespace dec
