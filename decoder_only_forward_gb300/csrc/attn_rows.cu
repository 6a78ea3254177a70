// Decode attention for a batch of independent sequences (one query position
// per row, each row reading its own sequence's KV rings).
//
// Row b of a batched step is the query of sequence seq[b] at position pos[b]:
// its G = nq/nkv query heads of kv head g attend to the readable keys of that
// sequence, min(pos+1, max_seq) slots under a sliding window and pos+1
// otherwise (Pantheon "Llama Forward Pass", Sliding Window and Grouped Query
// Attention; rml "The decoder", Attend).  CTA (g, split, b) runs the online
// softmax over its key range and leaves a (max, sum, output) triple per head;
// k_attn_rows_merge combines the splits of a head in split order.  Key order
// does not change the softmax, so slots are visited in slot order.
#include "prefill_common.cuh"
#include "runtime.h"

namespace dec {

constexpr int AR_THREADS = 128;
constexpr int AR_TILE = 32;   // keys staged per step (one key per lane when scoring)

// Shared-memory K tile: rows of HD floats as float4 chunks, chunk c of row r
// stored at c ^ (r & 7) so that 8 lanes reading chunk c of 8 consecutive rows
// hit 8 different 16-byte bank groups.
template <int HD>
__device__ __forceinline__ int ar_swz(int row, int c) {
  constexpr int M = (HD / 4) < 8 ? (HD / 4) - 1 : 7;
  return c ^ (row & M);
}

// 16 int8 codes of one scale group read back as code * s.  A code c becomes a
// float without a conversion instruction: the byte c ^ 0x80 = c + 128 (0..255)
// is placed under the exponent of 2^23, giving the float 2^23 + c + 128
// exactly, and 2^23 + 128 is subtracted (exact for every c).
__device__ __forceinline__ void widen_i8(const uint4& u, float s, float* f) {
  const uint32_t w[4] = {u.x ^ 0x80808080u, u.y ^ 0x80808080u, u.z ^ 0x80808080u, u.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    // bytes of the result: (byte i & 3 of the word, 0x00, 0x00, 0x4B)
    const uint32_t bits = __byte_perm(w[i >> 2], 0x4B000000u, 0x7540u + (i & 3));
    f[i] = __fmul_rn(__int_as_float(bits) - 8388736.0f, s);
  }
}

// Shared-memory layout of one CTA (G query heads per kv head):
//   qs   [G][C4] float4        scaled queries
//   kv   [2][AR_TILE][C4]      K (swizzled) and V of the tile; reused at the end
//                              for the cross-warp sum of the outputs [4][G][C4]
//   red  [4][G][AR_TILE] f32   per-warp partial scores
//   ps   [AR_TILE][AR_PSW] f32 softmax weights of the tile, key-major
//   mrow, lrow, alpha [G]
constexpr int AR_PSW = 20;   // >= MAX_GROUP, a multiple of 4 (float4 rows)

template <int HD>
__host__ __device__ constexpr size_t ar_smem_bytes(int G) {
  return 16 * ((size_t)G * (HD / 4) + 2 * (size_t)AR_TILE * (HD / 4)) +
         4 * (4 * (size_t)G * AR_TILE + (size_t)AR_TILE * AR_PSW + 3 * (size_t)G);
}

// KV: float, __nv_bfloat16 or int8_t (rows of the int8 format: scales, then
// codes at byte code_off; qgroup channels per scale).  Rows are row_bytes apart.
//
// Work split inside a 32-key tile: for the scores, warp w takes a quarter of
// head_dim for all 32 keys (lane = key) and all G heads, so each K chunk read
// from shared memory serves every head; the partial dot products meet in
// shared memory.  For P.V, warp w takes a quarter of the keys, each lane one
// float4 of head_dim for all G heads, so each V chunk serves every head; the
// warps' sums meet once, after the last tile.
// NHG: head groups of 4 held in registers (G <= 4 * NHG).
template <typename KV, int HD, int NHG>
__global__ void __launch_bounds__(AR_THREADS) k_attn_rows(
    const float* __restrict__ Q, const char* __restrict__ kc, const char* __restrict__ vc, const KvPaging pg,
    int row_bytes, int code_off, int qgroup, const int32_t* __restrict__ seq, const int32_t* __restrict__ pos, int nq,
    int nkv, int max_seq, int sliding, float* __restrict__ part) {
  constexpr bool I8 = std::is_same<KV, int8_t>::value;
  constexpr int CE = I8 ? 16 : 16 / (int)sizeof(KV);   // elements per 16-byte global chunk
  constexpr int CPR = HD / CE;            // global chunks per row
  constexpr int C4 = HD / 4;              // float4 chunks per row
  constexpr int CW = C4 / 4;              // score chunks per warp
  constexpr int LPT = (AR_TILE * CPR + AR_THREADS - 1) / AR_THREADS;
  constexpr int KPP = 32 / C4;            // keys per P.V pass of a warp (lanes: chunk, key)
  extern __shared__ __align__(16) uint8_t ar_smem[];

  const int g = blockIdx.x, split = blockIdx.y, nsplit = gridDim.y, b = blockIdx.z;
  const int G = nq / nkv;
  float4* qs = reinterpret_cast<float4*>(ar_smem);                      // [G][C4]
  float4* kvb = qs + (size_t)G * C4;                                     // [2][AR_TILE][C4]
  float4* ks = kvb;
  float4* vs = kvb + AR_TILE * C4;
  float* red = reinterpret_cast<float*>(kvb + 2 * AR_TILE * C4);        // [4][G][AR_TILE]
  float* ps = red + 4 * G * AR_TILE;                                     // [AR_TILE][AR_PSW]
  float* mrow = ps + AR_TILE * AR_PSW;
  float* lrow = mrow + G;
  float* alpha = lrow + G;

  const int p = pos[b];
  const int m = sliding > 0 ? min(p + 1, max_seq) : p + 1;
  const int per = ((m + nsplit - 1) / nsplit + AR_TILE - 1) / AR_TILE * AR_TILE;
  const int j0 = split * per, j1 = min(m, j0 + per);
  const char* K = kc;   // the layer's bases; rows through pg
  const char* V = vc;
  const int sq = seq[b];
  const float* q = Q + (size_t)b * nq * HD + (size_t)g * G * HD;
  const float scale = 1.0f / sqrtf((float)HD);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < G * C4; i += AR_THREADS) {
    float4 v = reinterpret_cast<const float4*>(q)[i];
    v.x *= scale;
    v.y *= scale;
    v.z *= scale;
    v.w *= scale;
    qs[i] = v;
  }
  if (tid < G) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.f;
  }
  // P.V accumulators: head group hg, head u of the group, float4 chunk pc.
  const int pc = lane % C4, pr = lane / C4;
  float4 acc[NHG][4];
#pragma unroll
  for (int hg = 0; hg < NHG; ++hg)
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[hg][u] = make_float4(0.f, 0.f, 0.f, 0.f);

  // The next tile's K/V chunks are loaded into registers while the current
  // tile is scored from shared memory.
  uint4 kr[LPT], vr[LPT];
  float ksc[LPT], vsc[LPT];   // int8: the chunk's group scale
  auto load = [&](int t0) {
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int i = tid + j * AR_THREADS, row = i / CPR, c = i % CPR;
      if (i < AR_TILE * CPR && t0 + row < j1) {
        const size_t rb = (size_t)kv_phys_row(pg, sq, t0 + row) * row_bytes;
        const int ch = g * HD + c * CE;   // first channel of the chunk
        const size_t off = I8 ? rb + code_off + ch : rb + (size_t)ch * sizeof(KV);
        kr[j] = __ldcs(reinterpret_cast<const uint4*>(K + off));
        vr[j] = __ldcs(reinterpret_cast<const uint4*>(V + off));
        if constexpr (I8) {
          ksc[j] = __ldcs(reinterpret_cast<const float*>(K + rb) + ch / qgroup);
          vsc[j] = __ldcs(reinterpret_cast<const float*>(V + rb) + ch / qgroup);
        }
      }
    }
  };
  if (j0 < j1) load(j0);
  for (int t0 = j0; t0 < j1; t0 += AR_TILE) {
    const int nt = min(AR_TILE, j1 - t0);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int i = tid + j * AR_THREADS, row = i / CPR, c = i % CPR;
      if (i < AR_TILE * CPR && row < nt) {
        float kf[CE], vf[CE];
        if constexpr (I8) {
          widen_i8(kr[j], ksc[j], kf);
          widen_i8(vr[j], vsc[j], vf);
        } else {
          Chunk<KV>::widen(kr[j], kf);
          Chunk<KV>::widen(vr[j], vf);
        }
#pragma unroll
        for (int h4 = 0; h4 < CE / 4; ++h4) {
          const int c4 = c * (CE / 4) + h4;
          ks[row * C4 + ar_swz<HD>(row, c4)] =
              make_float4(kf[4 * h4], kf[4 * h4 + 1], kf[4 * h4 + 2], kf[4 * h4 + 3]);
          vs[row * C4 + c4] = make_float4(vf[4 * h4], vf[4 * h4 + 1], vf[4 * h4 + 2], vf[4 * h4 + 3]);
        }
      }
    }
    __syncthreads();
    if (t0 + AR_TILE < j1) load(t0 + AR_TILE);
    // Partial scores: key = lane, chunks [warp*CW, warp*CW + CW), all heads.
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg) {
      if (hg * 4 < G) {
        float sp[4] = {0.f, 0.f, 0.f, 0.f};
        if (lane < nt) {
#pragma unroll
          for (int cc = 0; cc < CW; ++cc) {
            const int c = warp * CW + cc;
            const float4 kv = ks[lane * C4 + ar_swz<HD>(lane, c)];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (hg * 4 + u < G) {
                const float4 qv = qs[(hg * 4 + u) * C4 + c];
                sp[u] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, fmaf(qv.w, kv.w, sp[u]))));
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (hg * 4 + u < G) red[(warp * G + hg * 4 + u) * AR_TILE + lane] = sp[u];
      }
    }
    __syncthreads();
    // Scores, online softmax: warp per head, lane per key.
    for (int hh = warp; hh < G; hh += AR_THREADS / 32) {
      float s = -INFINITY;
      if (lane < nt)
        s = red[(0 * G + hh) * AR_TILE + lane] + red[(1 * G + hh) * AR_TILE + lane] +
            red[(2 * G + hh) * AR_TILE + lane] + red[(3 * G + hh) * AR_TILE + lane];
      const float mnew = fmaxf(mrow[hh], warp_max(s));
      const float e = lane < nt ? __expf(s - mnew) : 0.f;
      const float esum = warp_sum(e);
      ps[lane * AR_PSW + hh] = e;
      __syncwarp();
      if (lane == 0) {
        const float a = __expf(mrow[hh] - mnew);
        alpha[hh] = a;
        lrow[hh] = lrow[hh] * a + esum;
        mrow[hh] = mnew;
      }
    }
    __syncthreads();
    // P.V: this warp's keys of the tile, lane = (chunk pc, key pr of the pass).
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg) {
      if (hg * 4 < G) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (hg * 4 + u < G) {
            const float a = alpha[hg * 4 + u];
            acc[hg][u].x *= a;
            acc[hg][u].y *= a;
            acc[hg][u].z *= a;
            acc[hg][u].w *= a;
          }
        }
      }
    }
    for (int kg = warp; kg * KPP < nt; kg += 4) {
      const int j = kg * KPP + pr;
      if (j < nt) {
        const float4 v = vs[j * C4 + pc];
#pragma unroll
        for (int hg = 0; hg < NHG; ++hg) {
          if (hg * 4 < G) {
            const float4 pw = *reinterpret_cast<const float4*>(ps + j * AR_PSW + hg * 4);
            const float pu[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              acc[hg][u].x = fmaf(pu[u], v.x, acc[hg][u].x);
              acc[hg][u].y = fmaf(pu[u], v.y, acc[hg][u].y);
              acc[hg][u].z = fmaf(pu[u], v.z, acc[hg][u].z);
              acc[hg][u].w = fmaf(pu[u], v.w, acc[hg][u].w);
            }
          }
        }
      }
    }
  }
  // Lanes holding the same chunk for different keys, then the four warps.
#pragma unroll
  for (int o = C4; o < 32; o <<= 1) {
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[hg][u].x += __shfl_xor_sync(0xffffffffu, acc[hg][u].x, o);
        acc[hg][u].y += __shfl_xor_sync(0xffffffffu, acc[hg][u].y, o);
        acc[hg][u].z += __shfl_xor_sync(0xffffffffu, acc[hg][u].z, o);
        acc[hg][u].w += __shfl_xor_sync(0xffffffffu, acc[hg][u].w, o);
      }
    }
  }
  __syncthreads();   // the tile buffers become the cross-warp sum [4][G][C4]
  float4* sum4 = kvb;
  if (pr == 0) {
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (hg * 4 + u < G) sum4[(warp * G + hg * 4 + u) * C4 + pc] = acc[hg][u];
  }
  __syncthreads();
  // part[((b*nq + head) * nsplit + split) * (HD+2) + {0..HD-1: output, HD: max, HD+1: sum}];
  // an empty split leaves (-inf, 0, zeros), which the merge skips.
  for (int i = tid; i < G * C4; i += AR_THREADS) {
    const int hh = i / C4, c = i % C4;
    float4 o = sum4[(0 * G + hh) * C4 + c];
#pragma unroll
    for (int w2 = 1; w2 < 4; ++w2) {
      const float4 t = sum4[(w2 * G + hh) * C4 + c];
      o.x += t.x;
      o.y += t.y;
      o.z += t.z;
      o.w += t.w;
    }
    float* pp = part + (((size_t)b * nq + g * G + hh) * nsplit + split) * (HD + 2) + 4 * c;
    pp[0] = o.x;
    pp[1] = o.y;
    pp[2] = o.z;
    pp[3] = o.w;
  }
  if (tid < G) {
    float* pp = part + (((size_t)b * nq + g * G + tid) * nsplit + split) * (HD + 2);
    pp[HD] = mrow[tid];
    pp[HD + 1] = lrow[tid];
  }
}

// int8 code c (as the byte c ^ 0x80 in a word) -> float c, exactly (see widen_i8).
__device__ __forceinline__ float i8_to_f(uint32_t wx, int byte) {
  return __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u + byte)) - 8388736.0f;
}

// Compact tiles for bf16 and int8 rings (head_dim 64 or 128): the tile stays in
// its stored form in shared memory (2 or 1 bytes per element, the int8 scales
// beside it) and is widened as it is read.  For int8 a warp's quarter of
// head_dim lies inside one 32-channel scale group, so the key's scale
// multiplies the warp's partial dot product once; V is read back as code * s.
// Work split as in k_attn_rows.
template <typename KV, int HD>
struct ArcLayout {
  static constexpr bool I8 = std::is_same<KV, int8_t>::value;
  static constexpr int EB = I8 ? 1 : 2;            // bytes per stored element
  static constexpr int RBY = HD * EB;               // bytes of one tile row
  static constexpr int NCH = RBY / 16;              // 16-byte chunks per row
  static constexpr int NG = HD / 32;                // int8 scale groups per row of one head
  static constexpr int TILE_BYTES = 2 * AR_TILE * RBY + (I8 ? 2 * AR_TILE * NG * 4 : 0);
  __host__ __device__ static size_t region(int G) {  // the tile, later the cross-warp sum [4][G][HD/4] float4
    const size_t sum = (size_t)4 * G * HD * 4;
    return (size_t)TILE_BYTES > sum ? (size_t)TILE_BYTES : sum;
  }
  __host__ __device__ static size_t bytes(int G) {
    return 16 * (size_t)G * (HD / 4) + region(G) + 4 * (4 * (size_t)G * AR_TILE + (size_t)AR_TILE * AR_PSW + 3 * (size_t)G);
  }
};

template <typename KV, int HD, int NHG>
__global__ void __launch_bounds__(AR_THREADS) k_attn_rows_c(
    const float* __restrict__ Q, const char* __restrict__ kc, const char* __restrict__ vc, const KvPaging pg,
    int row_bytes, int code_off, const int32_t* __restrict__ seq, const int32_t* __restrict__ pos, int nq, int nkv,
    int max_seq, int sliding, float* __restrict__ part) {
  using LY = ArcLayout<KV, HD>;
  constexpr bool I8 = LY::I8;
  constexpr int C4 = HD / 4, NCH = LY::NCH, RBY = LY::RBY, NG = LY::NG;
  constexpr int EPC = 16 / LY::EB;                 // elements per 16-byte chunk
  constexpr int CWR = NCH / 4;                      // score chunks per warp
  constexpr int SWM = (NCH < 8 ? NCH : 8) - 1;      // K chunk swizzle mask
  constexpr int LPT = (AR_TILE * NCH + AR_THREADS - 1) / AR_THREADS;
  constexpr int KPP = 32 / C4;
  extern __shared__ __align__(16) uint8_t ar_smem[];

  const int g = blockIdx.x, split = blockIdx.y, nsplit = gridDim.y, b = blockIdx.z;
  const int G = nq / nkv;
  float4* qs = reinterpret_cast<float4*>(ar_smem);                           // [G][C4]
  uint8_t* reg = ar_smem + 16 * (size_t)G * C4;
  uint4* kraw = reinterpret_cast<uint4*>(reg);                                // [AR_TILE][NCH] swizzled
  uint8_t* vraw = reg + AR_TILE * RBY;                                        // [AR_TILE][RBY]
  float* kscl = reinterpret_cast<float*>(reg + 2 * AR_TILE * RBY);            // [AR_TILE][NG] (int8)
  float* vscl = kscl + AR_TILE * NG;
  float* red = reinterpret_cast<float*>(reg + LY::region(G));                 // [4][G][AR_TILE]
  float* ps = red + 4 * G * AR_TILE;
  float* mrow = ps + AR_TILE * AR_PSW;
  float* lrow = mrow + G;
  float* alpha = lrow + G;

  const int p = pos[b];
  const int m = sliding > 0 ? min(p + 1, max_seq) : p + 1;
  const int per = ((m + nsplit - 1) / nsplit + AR_TILE - 1) / AR_TILE * AR_TILE;
  const int j0 = split * per, j1 = min(m, j0 + per);
  const char* K = kc;   // the layer's bases; rows through pg
  const char* V = vc;
  const int sq = seq[b];
  const float* q = Q + (size_t)b * nq * HD + (size_t)g * G * HD;
  const float scale = 1.0f / sqrtf((float)HD);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < G * C4; i += AR_THREADS) {
    float4 v = reinterpret_cast<const float4*>(q)[i];
    v.x *= scale;
    v.y *= scale;
    v.z *= scale;
    v.w *= scale;
    qs[i] = v;
  }
  if (tid < G) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.f;
  }
  const int pc = lane % C4, pr = lane / C4;
  float4 acc[NHG][4];
#pragma unroll
  for (int hg = 0; hg < NHG; ++hg)
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[hg][u] = make_float4(0.f, 0.f, 0.f, 0.f);

  uint4 kr[LPT], vr[LPT];
  float ksr = 0.f, vsr = 0.f;   // int8: one scale of K and of V per thread (tid < AR_TILE * NG)
  const size_t head_off = I8 ? (size_t)code_off + (size_t)g * HD : (size_t)g * HD * 2;
  auto load = [&](int t0) {
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int i = tid + j * AR_THREADS, row = i / NCH, c = i % NCH;
      if (i < AR_TILE * NCH && t0 + row < j1) {
        const size_t off = (size_t)kv_phys_row(pg, sq, t0 + row) * row_bytes + head_off + c * 16;
        kr[j] = __ldcs(reinterpret_cast<const uint4*>(K + off));
        vr[j] = __ldcs(reinterpret_cast<const uint4*>(V + off));
      }
    }
    if constexpr (I8) {
      const int row = tid / NG, gi = tid % NG;
      if (tid < AR_TILE * NG && t0 + row < j1) {
        const size_t off = (size_t)kv_phys_row(pg, sq, t0 + row) * row_bytes + 4 * ((size_t)g * NG + gi);
        ksr = __ldcs(reinterpret_cast<const float*>(K + off));
        vsr = __ldcs(reinterpret_cast<const float*>(V + off));
      }
    }
  };
  if (j0 < j1) load(j0);
  for (int t0 = j0; t0 < j1; t0 += AR_TILE) {
    const int nt = min(AR_TILE, j1 - t0);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int i = tid + j * AR_THREADS, row = i / NCH, c = i % NCH;
      if (i < AR_TILE * NCH && row < nt) {
        uint4 kw = kr[j], vw = vr[j];
        if constexpr (I8) {   // stored biased, ready for the exponent trick
          kw.x ^= 0x80808080u; kw.y ^= 0x80808080u; kw.z ^= 0x80808080u; kw.w ^= 0x80808080u;
          vw.x ^= 0x80808080u; vw.y ^= 0x80808080u; vw.z ^= 0x80808080u; vw.w ^= 0x80808080u;
        }
        kraw[row * NCH + (c ^ (row & SWM))] = kw;
        *reinterpret_cast<uint4*>(vraw + row * RBY + c * 16) = vw;
      }
    }
    if constexpr (I8) {
      if (tid < AR_TILE * NG && tid / NG < nt) {
        kscl[tid] = ksr;
        vscl[tid] = vsr;
      }
    }
    __syncthreads();
    if (t0 + AR_TILE < j1) load(t0 + AR_TILE);
    // Partial scores: key = lane, this warp's chunks, all heads.
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg) {
      if (hg * 4 < G) {
        float sp[4] = {0.f, 0.f, 0.f, 0.f};
        if (lane < nt) {
#pragma unroll
          for (int cc = 0; cc < CWR; ++cc) {
            const int c = warp * CWR + cc;
            const uint4 kw = kraw[lane * NCH + (c ^ (lane & SWM))];
            const uint32_t wv[4] = {kw.x, kw.y, kw.z, kw.w};
            float kf[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
              if constexpr (I8) kf[e] = i8_to_f(wv[e >> 2], e & 3);
              else kf[e] = (e & 1) ? __uint_as_float(wv[e >> 1] & 0xffff0000u) : __uint_as_float(wv[e >> 1] << 16);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (hg * 4 + u < G) {
#pragma unroll
                for (int f4 = 0; f4 < EPC / 4; ++f4) {
                  const float4 qv = qs[(hg * 4 + u) * C4 + c * (EPC / 4) + f4];
                  sp[u] = fmaf(qv.x, kf[4 * f4], fmaf(qv.y, kf[4 * f4 + 1],
                               fmaf(qv.z, kf[4 * f4 + 2], fmaf(qv.w, kf[4 * f4 + 3], sp[u]))));
                }
              }
            }
          }
          if constexpr (I8) {
            const float sk = kscl[lane * NG + (warp * (HD / 4)) / 32];
#pragma unroll
            for (int u = 0; u < 4; ++u) sp[u] *= sk;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (hg * 4 + u < G) red[(warp * G + hg * 4 + u) * AR_TILE + lane] = sp[u];
      }
    }
    __syncthreads();
    for (int hh = warp; hh < G; hh += AR_THREADS / 32) {
      float sc = -INFINITY;
      if (lane < nt)
        sc = red[(0 * G + hh) * AR_TILE + lane] + red[(1 * G + hh) * AR_TILE + lane] +
             red[(2 * G + hh) * AR_TILE + lane] + red[(3 * G + hh) * AR_TILE + lane];
      const float mnew = fmaxf(mrow[hh], warp_max(sc));
      const float e = lane < nt ? __expf(sc - mnew) : 0.f;
      const float esum = warp_sum(e);
      ps[lane * AR_PSW + hh] = e;
      __syncwarp();
      if (lane == 0) {
        const float a = __expf(mrow[hh] - mnew);
        alpha[hh] = a;
        lrow[hh] = lrow[hh] * a + esum;
        mrow[hh] = mnew;
      }
    }
    __syncthreads();
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg) {
      if (hg * 4 < G) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (hg * 4 + u < G) {
            const float a = alpha[hg * 4 + u];
            acc[hg][u].x *= a;
            acc[hg][u].y *= a;
            acc[hg][u].z *= a;
            acc[hg][u].w *= a;
          }
        }
      }
    }
    for (int kg = warp; kg * KPP < nt; kg += 4) {
      const int j = kg * KPP + pr;
      if (j < nt) {
        float4 v;
        if constexpr (I8) {
          const uint32_t w4 = *reinterpret_cast<const uint32_t*>(vraw + j * RBY + pc * 4);
          const float sv = vscl[j * NG + (pc * 4) / 32];
          v = make_float4(__fmul_rn(i8_to_f(w4, 0), sv), __fmul_rn(i8_to_f(w4, 1), sv),
                          __fmul_rn(i8_to_f(w4, 2), sv), __fmul_rn(i8_to_f(w4, 3), sv));
        } else {
          const uint2 w2 = *reinterpret_cast<const uint2*>(vraw + j * RBY + pc * 8);
          v = make_float4(__uint_as_float(w2.x << 16), __uint_as_float(w2.x & 0xffff0000u),
                          __uint_as_float(w2.y << 16), __uint_as_float(w2.y & 0xffff0000u));
        }
#pragma unroll
        for (int hg = 0; hg < NHG; ++hg) {
          if (hg * 4 < G) {
            const float4 pw = *reinterpret_cast<const float4*>(ps + j * AR_PSW + hg * 4);
            const float pu[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              acc[hg][u].x = fmaf(pu[u], v.x, acc[hg][u].x);
              acc[hg][u].y = fmaf(pu[u], v.y, acc[hg][u].y);
              acc[hg][u].z = fmaf(pu[u], v.z, acc[hg][u].z);
              acc[hg][u].w = fmaf(pu[u], v.w, acc[hg][u].w);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = C4; o < 32; o <<= 1) {
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[hg][u].x += __shfl_xor_sync(0xffffffffu, acc[hg][u].x, o);
        acc[hg][u].y += __shfl_xor_sync(0xffffffffu, acc[hg][u].y, o);
        acc[hg][u].z += __shfl_xor_sync(0xffffffffu, acc[hg][u].z, o);
        acc[hg][u].w += __shfl_xor_sync(0xffffffffu, acc[hg][u].w, o);
      }
    }
  }
  __syncthreads();   // the tile region becomes the cross-warp sum [4][G][C4]
  float4* sum4 = reinterpret_cast<float4*>(reg);
  if (pr == 0) {
#pragma unroll
    for (int hg = 0; hg < NHG; ++hg)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (hg * 4 + u < G) sum4[(warp * G + hg * 4 + u) * C4 + pc] = acc[hg][u];
  }
  __syncthreads();
  for (int i = tid; i < G * C4; i += AR_THREADS) {
    const int hh = i / C4, c = i % C4;
    float4 o = sum4[(0 * G + hh) * C4 + c];
#pragma unroll
    for (int w2 = 1; w2 < 4; ++w2) {
      const float4 t = sum4[(w2 * G + hh) * C4 + c];
      o.x += t.x;
      o.y += t.y;
      o.z += t.z;
      o.w += t.w;
    }
    float* pp = part + (((size_t)b * nq + g * G + hh) * nsplit + split) * (HD + 2) + 4 * c;
    pp[0] = o.x;
    pp[1] = o.y;
    pp[2] = o.z;
    pp[3] = o.w;
  }
  if (tid < G) {
    float* pp = part + (((size_t)b * nq + g * G + tid) * nsplit + split) * (HD + 2);
    pp[HD] = mrow[tid];
    pp[HD + 1] = lrow[tid];
  }
}

// One CTA per (head, row): combines the row's splits and writes the head's
// output into the row's attention vector (the A operand of the O projection).
template <int HD>
__global__ void __launch_bounds__(HD) k_attn_rows_merge(const float* __restrict__ part, int nq, int nsplit,
                                                        RowOut out) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const float* base = part + ((size_t)b * nq + h) * nsplit * (HD + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, base[s * (HD + 2) + HD]);
  float L = 0.f, o = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float* pp = base + s * (HD + 2);
    const float ms = pp[HD];
    if (ms == -INFINITY) continue;
    const float sc = __expf(ms - M);
    L = fmaf(pp[HD + 1], sc, L);
    o = fmaf(pp[d], sc, o);
  }
  row_store(out, (size_t)b * nq * HD + (size_t)h * HD + d, o / L);
}

// Splits per kv head: one per 256 slots of the ring, at most AR_MAX_SPLIT.  It
// depends on the configuration only, never on the batch, so that a row's
// rounding is the same whatever batch it runs in.
int attn_rows_splits(const dec_config& c) {
  const int ns = (c.max_seq + 255) / 256;
  return ns < 1 ? 1 : (ns > AR_MAX_SPLIT ? AR_MAX_SPLIT : ns);
}

template <typename KV, int HD, int NHG>
static void attn_rows_g(const dec_config& c, const float* Q, const void* kc, const void* vc, const KvPaging& pg,
                        const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, cudaStream_t s) {
  const KvRowLayout L = kv_row_layout(c);
  const dim3 grid(c.n_kv_heads, nsplit, B);
  if constexpr (!std::is_same<KV, float>::value && HD != 16) {
    // bf16 / int8 rings: compact tiles.
    const size_t smem = ArcLayout<KV, HD>::bytes(c.n_heads / c.n_kv_heads);
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(k_attn_rows_c<KV, HD, NHG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_attn_rows_c<KV, HD, NHG><<<grid, AR_THREADS, smem, s>>>(Q, (const char*)kc, (const char*)vc, pg,
                                                              L.bytes, L.code_off, seq, pos, c.n_heads,
                                                              c.n_kv_heads, c.max_seq, c.sliding_window, part);
    return;
  }
  const size_t smem = ar_smem_bytes<HD>(c.n_heads / c.n_kv_heads);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(k_attn_rows<KV, HD, NHG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_attn_rows<KV, HD, NHG><<<grid, AR_THREADS, smem, s>>>(Q, (const char*)kc, (const char*)vc, pg, L.bytes, L.code_off,
                                                  L.group, seq, pos, c.n_heads, c.n_kv_heads, c.max_seq,
                                                  c.sliding_window, part);
}

template <typename KV, int HD>
static void attn_rows(const dec_config& c, const float* Q, const void* kc, const void* vc, const KvPaging& pg,
                      const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, RowOut out,
                      cudaStream_t s) {
  const int G = c.n_heads / c.n_kv_heads;
  if (G <= 4) attn_rows_g<KV, HD, 1>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, s);
  else if (G <= 8) attn_rows_g<KV, HD, 2>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, s);
  else attn_rows_g<KV, HD, 4>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, s);
  k_attn_rows_merge<HD><<<dim3(c.n_heads, B), HD, 0, s>>>(part, c.n_heads, nsplit, out);
}

template <int HD>
static void attn_rows_hd(const dec_config& c, const float* Q, const void* kc, const void* vc, const KvPaging& pg,
                         const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, RowOut out,
                         cudaStream_t s) {
  if (c.kv_dtype == DEC_BF16)
    attn_rows<__nv_bfloat16, HD>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, out, s);
  else if (c.kv_dtype == DEC_I8)
    attn_rows<int8_t, HD>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, out, s);
  else
    attn_rows<float, HD>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, out, s);
}

void launch_attn_rows(const dec_config& c, const float* Q, const void* kc, const void* vc, const KvPaging& pg,
                      const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, RowOut out,
                      cudaStream_t s) {
  if (c.head_dim == 16) attn_rows_hd<16>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, out, s);
  else if (c.head_dim == 64) attn_rows_hd<64>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, out, s);
  else attn_rows_hd<128>(c, Q, kc, vc, pg, seq, pos, B, nsplit, part, out, s);
}

}  // namespace dec
