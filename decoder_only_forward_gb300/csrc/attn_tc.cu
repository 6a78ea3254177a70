// Causal GQA prefill attention on the tensor cores (tcgen05, kind::f16):
// one CTA = 128 query rows of one query head, looping over 64-key tiles of its
// kv head with a one-pass online softmax (rml "The decoder", Attend; the
// ZLLM page's softmax(QK^T/sqrt(d) + mask)V).
//
//   S(j) = Q . K(j)^T   M=128, N=64, K=HD   (TMEM columns [64 (j%2), 64 (j%2) + 64))
//   O   += P(j) . V(j)  M=128, N=HD, K=64   (TMEM columns [128, 128 + HD))
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
// producer (separate K and V^T rings, so K runs two tiles ahead), warp 1 MMA
// issuer and TMEM owner (S of the next tile is issued before P.V of this one,
// into the other S buffer), warps 2-9 softmax: two threads per query row, each
// owning half of a tile's keys and half of O's columns.
#include <cudaTypedefs.h>

#include <mutex>

#include "prefill_common.cuh"
#include "tc.cuh"

namespace dec {

constexpr int AT_BM = 128, AT_BN = 64;
constexpr int AT_SOFT = 256;                 // softmax threads: two per query row
constexpr int AT_THREADS = 64 + AT_SOFT;     // + TMA producer warp + MMA warp

// Shared-memory layout (offsets from a 1024-byte aligned base).
template <int HD>
struct AtCfg {
  static constexpr int QS = HD / 64;                     // 64 bf16 = 128 B per slab row
  static constexpr int Q_PLANE = QS * AT_BM * 128;       // one of hi / lo
  static constexpr int K_PLANE = QS * AT_BN * 128;
  static constexpr int V_PLANE = HD * 128;               // V^T: HD rows x 64 keys
  static constexpr int P_PLANE = AT_BM * 128;            // 128 rows x 64 keys
  static constexpr int K_STAGE = 2 * K_PLANE, V_STAGE = 2 * V_PLANE;
  static constexpr int OFF_K = 2 * Q_PLANE;              // K ring: 2 stages
  static constexpr int OFF_V = OFF_K + 2 * K_STAGE;      // V^T ring: 2 stages
  static constexpr int OFF_P = OFF_V + 2 * V_STAGE;
  static constexpr int OFF_X = OFF_P + 2 * P_PLANE;      // row max exchange [2 buffers][2 halves][128] f32
  static constexpr int OFF_BAR = OFF_X + 2 * 2 * AT_BM * 4;
  static constexpr int LAYOUT = OFF_BAR + 128;
  static constexpr int SLACK = 896;                      // room to align a 128-byte aligned window base
  static constexpr int SMEM = LAYOUT + SLACK;
  static constexpr int O_LD = HD + 4;                    // staged output rows (f32), in the K/V rings
  static constexpr int TMEM_COLS = 256;                  // S double buffer [0, 128), O [128, 128 + HD)
};
static_assert(AtCfg<128>::SMEM <= 232448, "shared memory of the HD=128 attention tile");
static_assert(AT_BM * AtCfg<128>::O_LD * 4 <= AtCfg<128>::OFF_P - AtCfg<128>::OFF_K, "output staging");
static_assert(AT_BM * AtCfg<64>::O_LD * 4 <= AtCfg<64>::OFF_P - AtCfg<64>::OFF_K, "output staging");

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

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Barrier 1 over the softmax threads; returns whether any of them passed `pred`.
__device__ __forceinline__ bool soft_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(AT_SOFT)
      : "memory");
  return r != 0;
}

// Rows whose running max grows by less than this (log2 units) keep the stale
// max: P then reaches up to 2^8, which the (hi, lo) planes carry exactly as
// well, and O needs no rescale.  The final O / l is the same either way.
constexpr float AT_RESCALE_LOG2 = 8.f;

template <int HD>
__global__ void __launch_bounds__(AT_THREADS, 1) k_attn_prefill_tc(const __grid_constant__ CUtensorMap tm_q,
                                                                  const __grid_constant__ CUtensorMap tm_k,
                                                                  const __grid_constant__ CUtensorMap tm_vt,
                                                                  AtArgs a) {
  using C = AtCfg<HD>;
  extern __shared__ uint8_t at_raw[];
  const uint32_t pad = (1024u - (smem_u32(at_raw) & 1023u)) & 1023u;
  if (pad > (uint32_t)C::SLACK) {  // same window for every thread: a uniform exit
    if (threadIdx.x == 0) raise_error(a.st, ERR_LAYOUT, 120);
    return;
  }
  uint8_t* smem = at_raw + pad;
  uint8_t* sQ = smem;                  // hi plane, then lo plane
  uint8_t* sK = smem + C::OFF_K;       // stage s: hi plane, lo plane
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;       // hi plane, then lo plane
  float* xmax = reinterpret_cast<float*>(smem + C::OFF_X);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;     // [2]
  uint64_t* k_empty = bars + 3;    // [2]
  uint64_t* v_full = bars + 5;     // [2]
  uint64_t* v_empty = bars + 7;    // [2]
  uint64_t* s_full = bars + 9;     // [2] one per S buffer
  uint64_t* p_ready = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* drained = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
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
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
    mbar_init(p_ready, AT_SOFT);
    mbar_init(o_done, 1);
    mbar_init(drained, 1);
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
  const uint32_t tO = tmem + 2 * AT_BN;

  if (warp == 0) {
    if (lane == 0) {
      // K of tile j waits only for S(j-2); V^T of tile j for P.V(j-2).
      mbar_arrive_expect_tx(q_full, 2 * C::Q_PLANE);
      for (int p = 0; p < 2; ++p)
        for (int s = 0; s < C::QS; ++s)
          tma_load_3d(sQ + p * C::Q_PLANE + s * AT_BM * 128, &tm_q, q_full, h * HD + 64 * s, t0, p);
      int nk = 0, nv = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j & 1;
        const uint32_t ph = ((j >> 1) & 1) ^ 1;
        const int r0 = (kt0 + j) * AT_BN;
        if (!mbar_wait(&k_empty[st], ph, abort_flag, a.st, 121)) break;
        mbar_arrive_expect_tx(&k_full[st], C::K_STAGE);
        for (int p = 0; p < 2; ++p)
          for (int s = 0; s < C::QS; ++s)
            tma_load_3d(sK + st * C::K_STAGE + p * C::K_PLANE + s * AT_BN * 128, &tm_k, &k_full[st],
                        g * HD + 64 * s, r0, p);
        ++nk;
        if (!mbar_wait(&v_empty[st], ph, abort_flag, a.st, 128)) break;
        mbar_arrive_expect_tx(&v_full[st], C::V_STAGE);
        for (int p = 0; p < 2; ++p)
          tma_load_3d(sV + st * C::V_STAGE + p * C::V_PLANE, &tm_vt, &v_full[st], r0, g * HD, p);
        ++nv;
      }
      if (*abort_flag) {
        // Let this CTA's copies land before its shared memory is given back.
        volatile int no_abort = 0;
        mbar_wait(q_full, 0, &no_abort, nullptr, 0, 100000000ull);
        for (int j = max(0, nk - 2); j < nk; ++j)
          mbar_wait(&k_full[j & 1], (j >> 1) & 1, &no_abort, nullptr, 0, 100000000ull);
        for (int j = max(0, nv - 2); j < nv; ++j)
          mbar_wait(&v_full[j & 1], (j >> 1) & 1, &no_abort, nullptr, 0, 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16_f32(AT_BM, AT_BN);
      constexpr uint32_t id_o = idesc_bf16_f32(AT_BM, HD);
      // S(j) = Qh.Kh + Qh.Kl + Ql.Kh into S buffer j & 1, 16 head-dim elements per step.
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, a.st, 123)) return false;
        tc_fence_after();
        const uint8_t* kbase = sK + st * C::K_STAGE;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks & 3) * 32;
          const uint32_t qa = smem_u32(sQ + (ks >> 2) * AT_BM * 128 + off);
          const uint32_t kb = smem_u32(kbase + (ks >> 2) * AT_BN * 128 + off);
          const uint64_t qh = sw128_kmajor_desc(qa), ql = sw128_kmajor_desc(qa + C::Q_PLANE);
          const uint64_t kh = sw128_kmajor_desc(kb), kl = sw128_kmajor_desc(kb + C::K_PLANE);
          const uint32_t d = tmem + st * AT_BN;
          tc_mma_bf16(d, qh, kh, id_s, ks > 0 ? 1u : 0u);
          tc_mma_bf16(d, qh, kl, id_s, 1u);
          tc_mma_bf16(d, ql, kh, id_s, 1u);
        }
        tc_commit(&s_full[st]);
        tc_commit(&k_empty[st]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, a.st, 122) && issue_s(0);
      for (int j = 0; j < ntiles && ok; ++j) {
        // S of the next tile runs while the softmax threads work on this one.
        if (j + 1 < ntiles && !issue_s(j + 1)) break;
        if (!mbar_wait(p_ready, j & 1, abort_flag, a.st, 124)) break;
        if (!mbar_wait(&v_full[j & 1], (j >> 1) & 1, abort_flag, a.st, 129)) break;
        tc_fence_after();
        // O += Ph.Vh + Ph.Vl + Pl.Vh over the tile's 64 keys.
        const uint8_t* vbase = sV + (j & 1) * C::V_STAGE;
#pragma unroll
        for (int ks = 0; ks < AT_BN / 16; ++ks) {
          const uint32_t pa = smem_u32(sP + ks * 32);
          const uint32_t vb = smem_u32(vbase + ks * 32);
          const uint64_t ph = sw128_kmajor_desc(pa), pl = sw128_kmajor_desc(pa + C::P_PLANE);
          const uint64_t vh = sw128_kmajor_desc(vb), vl = sw128_kmajor_desc(vb + C::V_PLANE);
          tc_mma_bf16(tO, ph, vh, id_o, (j > 0 || ks > 0) ? 1u : 0u);
          tc_mma_bf16(tO, ph, vl, id_o, 1u);
          tc_mma_bf16(tO, pl, vh, id_o, 1u);
        }
        tc_commit(&v_empty[j & 1]);
        tc_commit(o_done);
      }
      // Every MMA issued here completes before the TMEM goes back.
      tc_commit(drained);
      volatile int no_abort = 0;
      mbar_wait(drained, 0, &no_abort, nullptr, 0, 100000000ull);
    }
  } else {
    // Softmax: warps 2-5 take keys 0-31 of each tile and O columns [0, HD/2),
    // warps 6-9 keys 32-63 and O columns [HD/2, HD); thread -> query row r
    // (TMEM lane r: warp w reaches lanes 32 (w % 4) .. 32 (w % 4) + 31).
    // The two threads of a row share the tile max through shared memory and
    // agree on every decision, so they keep identical running maxima.
    // Branches around tcgen05.ld / st are warp-uniform and every exit from
    // the tile loop is agreed by all softmax threads at barrier 1.
    const int hf = (warp - 2) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int t = t0 + r;
    const bool row_ok = t < a.n;
    const int qpos = a.start + t;
    const int lo = a.sliding > 0 ? max(0, qpos - a.sliding + 1) : 0;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float scale = a.scale_log2;
    float m = -INFINITY, l = 0.f;   // running max (log2 units) and this half's sum
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
      const bool got = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, a.st, 125));
      float sv[32];
      float mt = -INFINITY;
      if (got) {
        tc_fence_after();
        tmem_ld32(tmem + (j & 1) * AT_BN + hf * 32 + lane_off, sv);
        const int kabs0 = (kt0 + j) * AT_BN + a.base_pos + hf * 32;
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int kp = kabs0 + jj + u;
            if (!(row_ok && kp <= qpos && kp >= lo)) sv[jj + u] = -INFINITY;
          }
          mx0 = fmaxf(mx0, sv[jj]);
          mx1 = fmaxf(mx1, sv[jj + 1]);
          mx2 = fmaxf(mx2, sv[jj + 2]);
          mx3 = fmaxf(mx3, sv[jj + 3]);
        }
        mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      }
      float* xb = xmax + (j & 1) * 2 * AT_BM;
      xb[hf * AT_BM + r] = mt;
      if (soft_sync_or(!got || bad)) {
        bad = true;
        break;
      }
      const float ms = fmaxf(mt, xb[(hf ^ 1) * AT_BM + r]) * scale;   // -inf stays -inf
      float alpha = 1.f;
      if (ms > m + AT_RESCALE_LOG2) {
        alpha = m == -INFINITY ? 0.f : ex2_approx(m - ms);
        m = ms;
      }
      float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
      if (m == -INFINITY) {
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) sv[jj] = 0.f;
      } else {
        const float negm = -m;
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4) {
          sv[jj] = ex2_approx(fmaf(sv[jj], scale, negm));
          sv[jj + 1] = ex2_approx(fmaf(sv[jj + 1], scale, negm));
          sv[jj + 2] = ex2_approx(fmaf(sv[jj + 2], scale, negm));
          sv[jj + 3] = ex2_approx(fmaf(sv[jj + 3], scale, negm));
          ps0 += sv[jj];
          ps1 += sv[jj + 1];
          ps2 += sv[jj + 2];
          ps3 += sv[jj + 3];
        }
      }
      l = l * alpha + ((ps0 + ps1) + (ps2 + ps3));
      // P and O are still in use by the previous tile's P.V until it completes.
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, a.st, 126))) {
          bad = true;   // the next barrier takes everyone out
          continue;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < HD / 2; c += 32) {
            float ov[32];
            const uint32_t ta = tO + lane_off + hf * (HD / 2) + c;
            tmem_ld32(ta, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= alpha;
            tmem_st32(ta, ov);
          }
        }
      }
      // This half of P row r into the swizzled K-major planes: 16-byte chunk
      // cg (keys 8cg..8cg+7) of row r sits at chunk cg ^ (r % 8).
      uint8_t* rowh = sP + r * 128;
      uint8_t* rowl = rowh + C::P_PLANE;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = sv[8 * c + 2 * i], x1 = sv[8 * c + 2 * i + 1];
          hw[i] = pack_bf16(x0, x1);
          lw[i] = pack_bf16(x0 - bf16_lo(hw[i]), x1 - bf16_hi(hw[i]));
        }
        const int cc = ((hf * 4 + c) ^ (r & 7)) * 16;
        *reinterpret_cast<uint4*>(rowh + cc) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(rowl + cc) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_ready);
    }
    // Epilogue: row sums of both halves, O / l staged in the (now idle) K/V
    // rings, then stored row by row with consecutive threads on consecutive
    // columns.
    float* xb = xmax + (ntiles & 1) * 2 * AT_BM;
    xb[hf * AT_BM + r] = l;
    const bool got =
        !bad && __all_sync(0xffffffffu, mbar_wait(o_done, (ntiles - 1) & 1, abort_flag, a.st, 127));
    if (!soft_sync_or(!got)) {
      tc_fence_after();
      const float lt = l + xb[(hf ^ 1) * AT_BM + r];
      const float inv = lt > 0.f ? 1.0f / lt : 0.f;
      float* sO = reinterpret_cast<float*>(sK);
#pragma unroll
      for (int c = 0; c < HD / 2; c += 32) {
        float ov[32];
        tmem_ld32(tO + lane_off + hf * (HD / 2) + c, ov);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(sO + r * C::O_LD + hf * (HD / 2) + c + e) =
              make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv, ov[e + 3] * inv);
      }
      soft_sync_or(false);
      const int sid = threadIdx.x - 64;
      for (int idx = sid; idx < AT_BM * (HD / 4); idx += AT_SOFT) {
        const int row = idx / (HD / 4), c4 = idx % (HD / 4);
        if (t0 + row < a.n)
          row_store4(a.out, (size_t)(t0 + row) * a.qd + h * HD + 4 * c4,
                     *reinterpret_cast<const float4*>(sO + row * C::O_LD + 4 * c4));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
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
