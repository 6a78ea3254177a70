// Causal GQA prefill attention on the tensor cores (tcgen05, kind::f16):
// one CTA = 128 query rows of one query head, looping over 64-key tiles of its
// kv head with a one-pass online softmax (rml "The decoder", Attend; the
// ZLLM page's softmax(QK^T/sqrt(d) + mask)V).
//
//   S  = Q . K^T   M=128, N=64,  K=HD   (TMEM columns [0, 64))
//   O += P . V     M=128, N=HD,  K=64   (TMEM columns [64, 64+HD))
//
// Every operand x is carried as a pair of bf16 planes, hi = bf16(x) and
// lo = bf16(x - hi), and each product as hi.hi + hi.lo + lo.hi: the dropped
// lo.lo term and the rounding of lo leave a relative error near 2^-16, close
// to fp32 arithmetic (one-plane tf32 or bf16 operands are not: truncating K
// to tf32 alone moves the logits of a 32-layer model by about 1e-2).
//
// Operands sit in shared memory K-major with 128-byte swizzling: the Q planes
// come from the QKV epilogue, the K planes and a transposed V (V^T rows of
// keys) from k_kv_split, P from the softmax threads.  Roles: warp 0 TMA
// producer, warp 1 MMA issuer (and TMEM owner), warps 2-5 softmax: thread i
// of those owns query row i (TMEM lane i), keeps its running max and sum in
// registers, and rescales its O row in TMEM when the max grows.
#include <cudaTypedefs.h>

#include <mutex>

#include "prefill_common.cuh"
#include "tc.cuh"

namespace dec {

constexpr int AT_BM = 128, AT_BN = 64, AT_THREADS = 192;

template <int HD>
struct AtCfg {
  static constexpr int QS = HD / 64;                     // 64 bf16 = 128 B per slab row
  static constexpr int Q_PLANE = QS * AT_BM * 128;       // one of hi / lo
  static constexpr int K_PLANE = QS * AT_BN * 128;
  static constexpr int V_PLANE = HD * 128;               // V^T: HD rows x 64 keys
  static constexpr int P_PLANE = AT_BM * 128;            // 128 rows x 64 keys
  static constexpr int STAGE_BYTES = 2 * K_PLANE + 2 * V_PLANE;
  static constexpr int SMEM = 2 * Q_PLANE + 2 * STAGE_BYTES + 2 * P_PLANE + 1024 + 256;
  static constexpr int TMEM_COLS = (AT_BN + HD) <= 128 ? 128 : 256;
};
static_assert(AtCfg<128>::SMEM <= 232448, "shared memory of the HD=128 attention tile");

struct AtArgs {
  int n, start, base_pos, nq, nkv, sliding;
  int qd;
  float scale_log2;      // log2(e) / sqrt(HD)
  RowOut out;            // [n][qd]
  DeviceState* st;
};

// Two bf16 values -> one 32-bit word (first value in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int HD>
__global__ void __launch_bounds__(AT_THREADS, 1) k_attn_prefill_tc(const __grid_constant__ CUtensorMap tm_q,
                                                                  const __grid_constant__ CUtensorMap tm_k,
                                                                  const __grid_constant__ CUtensorMap tm_vt,
                                                                  AtArgs a) {
  using C = AtCfg<HD>;
  extern __shared__ uint8_t at_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                      // hi plane, then lo plane
  uint8_t* sKV = sQ + 2 * C::Q_PLANE;                      // 2 stages of (K hi, K lo, V^T hi, V^T lo)
  uint8_t* sP = sKV + 2 * C::STAGE_BYTES;                  // hi plane, then lo plane
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * C::P_PLANE);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;    // [2]
  uint64_t* kv_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* p_ready = bars + 6;
  uint64_t* o_done = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, g = (h * a.nkv) / a.nq;
  const int nqt = (a.n + AT_BM - 1) / AT_BM;
  const int qt = nqt - 1 - (int)blockIdx.x;                // longest rows first
  const int t0 = qt * AT_BM;
  // Key tiles (columns relative to base_pos) this query tile can see.
  const int kmax = a.start + min(t0 + AT_BM, a.n) - 1;
  const int kmin = a.sliding > 0 ? max(0, a.start + t0 - a.sliding + 1) : 0;
  const int kt0 = (kmin - a.base_pos) / AT_BN, kt1 = (kmax - a.base_pos) / AT_BN;
  const int ntiles = kt1 - kt0 + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 128);
    mbar_init(o_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_vt);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + AT_BN;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::Q_PLANE);
      for (int p = 0; p < 2; ++p)
        for (int s = 0; s < C::QS; ++s)
          tma_load_3d(sQ + p * C::Q_PLANE + s * AT_BM * 128, &tm_q, q_full, h * HD + 64 * s, t0, p);
      for (int j = 0; j < ntiles; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, abort_flag, a.st, 121)) break;
        const int r0 = (kt0 + j) * AT_BN;
        uint8_t* sK = sKV + st * C::STAGE_BYTES;
        uint8_t* sV = sK + 2 * C::K_PLANE;
        mbar_arrive_expect_tx(&kv_full[st], C::STAGE_BYTES);
        for (int p = 0; p < 2; ++p) {
          for (int s = 0; s < C::QS; ++s)
            tma_load_3d(sK + p * C::K_PLANE + s * AT_BN * 128, &tm_k, &kv_full[st], g * HD + 64 * s, r0, p);
          tma_load_3d(sV + p * C::V_PLANE, &tm_vt, &kv_full[st], r0, g * HD, p);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(AT_BM, AT_BN);
      constexpr uint32_t id_o = idesc_bf16_f32(AT_BM, HD);
      bool ok = mbar_wait(q_full, 0, abort_flag, a.st, 122);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_full[st], (j >> 1) & 1, abort_flag, a.st, 123)) break;
        tc_fence_after();
        const uint8_t* sK = sKV + st * C::STAGE_BYTES;
        const uint8_t* sV = sK + 2 * C::K_PLANE;
        // S = Qh.Kh + Qh.Kl + Ql.Kh, 16 head-dim elements (32 bytes) per step.
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;
          const uint32_t qa = smem_u32(sQ + (ks >> 2) * AT_BM * 128 + off);
          const uint32_t kb = smem_u32(sK + (ks >> 2) * AT_BN * 128 + off);
          const uint64_t qh = sw128_kmajor_desc(qa), ql = sw128_kmajor_desc(qa + C::Q_PLANE);
          const uint64_t kh = sw128_kmajor_desc(kb), kl = sw128_kmajor_desc(kb + C::K_PLANE);
          tc_mma_bf16(tS, qh, kh, id_s, ks > 0 ? 1u : 0u);
          tc_mma_bf16(tS, qh, kl, id_s, 1u);
          tc_mma_bf16(tS, ql, kh, id_s, 1u);
        }
        tc_commit(s_full);
        if (!mbar_wait(p_ready, j & 1, abort_flag, a.st, 124)) break;
        tc_fence_after();
        // O += Ph.Vh + Ph.Vl + Pl.Vh over the tile's 64 keys.
#pragma unroll
        for (int ks = 0; ks < AT_BN / 16; ++ks) {
          const uint32_t off = ks * 32;
          const uint32_t pa = smem_u32(sP + off);
          const uint32_t vb = smem_u32(sV + off);
          const uint64_t ph = sw128_kmajor_desc(pa), pl = sw128_kmajor_desc(pa + C::P_PLANE);
          const uint64_t vh = sw128_kmajor_desc(vb), vl = sw128_kmajor_desc(vb + C::V_PLANE);
          tc_mma_bf16(tO, ph, vh, id_o, (j > 0 || ks > 0) ? 1u : 0u);
          tc_mma_bf16(tO, ph, vl, id_o, 1u);
          tc_mma_bf16(tO, pl, vh, id_o, 1u);
        }
        tc_commit(&kv_empty[st]);
        tc_commit(o_done);
      }
    }
  } else {
    // Softmax warps: thread -> query row r (TMEM lane r).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int t = t0 + r;
    const bool row_ok = t < a.n;
    const int qpos = a.start + t;
    const int lo = a.sliding > 0 ? max(0, qpos - a.sliding + 1) : 0;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // tcgen05.ld / st are warp-collective: every branch around them is taken
    // by the whole warp (__all_sync / __any_sync), also when a wait gives up.
    for (int j = 0; j < ntiles && ok; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, j & 1, abort_flag, a.st, 125))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[AT_BN];
      tmem_ld32(tS + lane_off, sv);
      tmem_ld32(tS + lane_off + 32, sv + 32);
      const int kabs0 = (kt0 + j) * AT_BN + a.base_pos;
      float mt = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < AT_BN; ++jj) {
        const int kp = kabs0 + jj;
        const bool valid = row_ok && kp <= qpos && kp >= lo;
        sv[jj] = valid ? sv[jj] * a.scale_log2 : -INFINITY;
        mt = fmaxf(mt, sv[jj]);
      }
      const float mnew = fmaxf(m, mt);
      const float alpha = m == -INFINITY ? 0.f : exp2f(m - mnew);
      float psum = 0.f;
#pragma unroll
      for (int jj = 0; jj < AT_BN; ++jj) {
        const float pv = mnew == -INFINITY ? 0.f : exp2f(sv[jj] - mnew);
        sv[jj] = pv;
        psum += pv;
      }
      l = l * alpha + psum;
      m = mnew;
      // P and O are still in use by the previous tile's P.V until it completes.
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, a.st, 126))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          for (int c = 0; c < HD; c += 32) {
            float ov[32];
            tmem_ld32(tO + lane_off + c, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
            tmem_st32(tO + lane_off + c, ov);
          }
        }
      }
      // P row r into the swizzled K-major planes: 16-byte chunk c (keys
      // 8c..8c+7) of row r sits at chunk c ^ (r % 8).
      uint8_t* rowh = sP + r * 128;
      uint8_t* rowl = rowh + C::P_PLANE;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = sv[8 * c + 2 * i], x1 = sv[8 * c + 2 * i + 1];
          hw[i] = pack_bf16(x0, x1);
          lw[i] = pack_bf16(x0 - bf16_lo(hw[i]), x1 - bf16_hi(hw[i]));
        }
        const int cc = (c ^ (r & 7)) * 16;
        *reinterpret_cast<uint4*>(rowh + cc) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(rowl + cc) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_ready);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(o_done, (ntiles - 1) & 1, abort_flag, a.st, 127))) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      for (int c = 0; c < HD; c += 32) {
        float ov[32];
        tmem_ld32(tO + lane_off + c, ov);
        if (row_ok)
#pragma unroll
          for (int e = 0; e < 32; ++e) row_store(a.out, (size_t)t * a.qd + h * HD + c + e, ov[e] * inv);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A role gave up: let issued MMAs finish before the TMEM goes back.
    volatile int no_abort = 0;
    if (threadIdx.x == 32) mbar_wait(o_done, (ntiles - 1) & 1, &no_abort, nullptr, 0, 100000000ull);
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// K rows -> bf16 (hi, lo) row planes, V rows -> transposed bf16 (hi, lo)
// planes, for rows [r0, r1) of f32 K/V row buffers of kd columns (kd a
// multiple of 32); 32 x 32 tiles, the V tile transposed through shared memory.
__global__ void __launch_bounds__(256) k_kv_split(const float* __restrict__ K, const float* __restrict__ V, int kd,
                                                  int r0, int r1, __nv_bfloat16* __restrict__ Kb, size_t k_plane,
                                                  __nv_bfloat16* __restrict__ Vt, int vt_ld, size_t v_plane) {
  __shared__ float tile[32][33];
  const int rb = r0 + blockIdx.x * 32, cb = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = rb + i;
    if (r < r1) {
      const size_t o = (size_t)r * kd + cb + threadIdx.x;
      const float k = K[o];
      const __nv_bfloat16 kh = __float2bfloat16_rn(k);
      Kb[o] = kh;
      Kb[k_plane + o] = __float2bfloat16_rn(k - __bfloat162float(kh));
      tile[i][threadIdx.x] = V[o];
    }
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = rb + threadIdx.x;
    if (r < r1) {
      const float v = tile[threadIdx.x][i];
      const __nv_bfloat16 vh = __float2bfloat16_rn(v);
      const size_t o = (size_t)(cb + i) * vt_ld + r;
      Vt[o] = vh;
      Vt[v_plane + o] = __float2bfloat16_rn(v - __bfloat162float(vh));
    }
  }
}

static PFN_cuTensorMapEncodeTiled_v12000 at_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3D bf16 map (x, row, plane) with 128-byte swizzling and a box of 64 x rows x 1.
static bool at_map(CUtensorMap* m, const void* base, uint64_t x, uint64_t rows, uint64_t row_bytes,
                   uint64_t plane_bytes, uint32_t box_rows) {
  auto fn = at_encode();
  if (!fn) return false;
  const cuuint64_t dims[3] = {x, rows, 2};
  const cuuint64_t strides[2] = {row_bytes, plane_bytes};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_kv_split(const float* K, const float* V, int kd, int r0, int r1, const AttnTcPlanes& pl,
                            cudaStream_t s) {
  if (r1 <= r0) return cudaSuccess;
  if (kd % 32 || r1 > pl.kcap || r1 > pl.vt_ld) return cudaErrorInvalidValue;
  const dim3 grid((r1 - r0 + 31) / 32, kd / 32);
  k_kv_split<<<grid, dim3(32, 8), 0, s>>>(K, V, kd, r0, r1, pl.Kb, (size_t)pl.kcap * kd, pl.Vt, pl.vt_ld,
                                          (size_t)kd * pl.vt_ld);
  return cudaGetLastError();
}

cudaError_t launch_attn_prefill_tc(const AttnTcPlanes& pl, int n, int start, int base_pos, int nq, int nkv, int hd,
                                   int sliding, RowOut out, DeviceState* st, cudaStream_t s) {
  if (hd != 64 && hd != 128) return cudaErrorInvalidValue;
  const int qd = nq * hd, kd = nkv * hd;
  const int kcount = start + n - base_pos;   // key columns 0 .. kcount-1 hold keys base_pos ..
  if (n <= 0 || n > pl.qcap || kcount <= 0 || kcount > pl.kcap || kcount > pl.vt_ld || (pl.vt_ld & 7))
    return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv;
  if (!at_map(&mq, pl.Qb, qd, n, (uint64_t)qd * 2, (uint64_t)pl.qcap * qd * 2, AT_BM) ||
      !at_map(&mk, pl.Kb, kd, kcount, (uint64_t)kd * 2, (uint64_t)pl.kcap * kd * 2, AT_BN) ||
      !at_map(&mv, pl.Vt, kcount, kd, (uint64_t)pl.vt_ld * 2, (uint64_t)kd * pl.vt_ld * 2, hd))
    return cudaErrorInvalidValue;
  AtArgs a;
  a.n = n;
  a.start = start;
  a.base_pos = base_pos;
  a.nq = nq;
  a.nkv = nkv;
  a.sliding = sliding;
  a.qd = qd;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
  a.out = out;
  a.st = st;
  const dim3 grid((n + AT_BM - 1) / AT_BM, nq);
  if (hd == 128) {
    cudaFuncSetAttribute(k_attn_prefill_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, AtCfg<128>::SMEM);
    k_attn_prefill_tc<128><<<grid, AT_THREADS, AtCfg<128>::SMEM, s>>>(mq, mk, mv, a);
  } else {
    cudaFuncSetAttribute(k_attn_prefill_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, AtCfg<64>::SMEM);
    k_attn_prefill_tc<64><<<grid, AT_THREADS, AtCfg<64>::SMEM, s>>>(mq, mk, mv, a);
  }
  return cudaGetLastError();
}

}  // namespace dec
