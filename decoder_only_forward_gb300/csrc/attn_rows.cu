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

template <typename KV, int HD>
__global__ void __launch_bounds__(AR_THREADS) k_attn_rows(
    const float* __restrict__ Q, const KV* __restrict__ kc, const KV* __restrict__ vc, size_t ring_elems,
    const int32_t* __restrict__ seq, const int32_t* __restrict__ pos, int nq, int nkv, int max_seq, int sliding,
    float* __restrict__ part) {
  constexpr int CE = 16 / sizeof(KV);     // elements per 16-byte global chunk
  constexpr int CPR = HD / CE;            // global chunks per row
  constexpr int C4 = HD / 4;              // float4 chunks per row
  constexpr int LPT = (AR_TILE * CPR + AR_THREADS - 1) / AR_THREADS;
  constexpr int R = (MAX_GROUP * C4 + AR_THREADS - 1) / AR_THREADS;   // (head, chunk) slots per thread
  __shared__ __align__(16) float4 qs[MAX_GROUP][C4];
  __shared__ __align__(16) float4 ks[AR_TILE][C4];
  __shared__ __align__(16) float4 vs[AR_TILE][C4];
  __shared__ float ps[MAX_GROUP][AR_TILE + 1];
  __shared__ float mrow[MAX_GROUP], lrow[MAX_GROUP], alpha[MAX_GROUP];

  const int g = blockIdx.x, split = blockIdx.y, nsplit = gridDim.y, b = blockIdx.z;
  const int G = nq / nkv, kd = nkv * HD;
  const int p = pos[b];
  const int m = sliding > 0 ? min(p + 1, max_seq) : p + 1;
  const int per = ((m + nsplit - 1) / nsplit + AR_TILE - 1) / AR_TILE * AR_TILE;
  const int j0 = split * per, j1 = min(m, j0 + per);
  const KV* K = kc + (size_t)seq[b] * ring_elems;
  const KV* V = vc + (size_t)seq[b] * ring_elems;
  const float* q = Q + (size_t)b * nq * HD + (size_t)g * G * HD;
  const float scale = 1.0f / sqrtf((float)HD);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < G * C4; i += AR_THREADS) {
    float4 v = reinterpret_cast<const float4*>(q)[i];
    v.x *= scale;
    v.y *= scale;
    v.z *= scale;
    v.w *= scale;
    qs[i / C4][i % C4] = v;
  }
  if (tid < MAX_GROUP) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.f;
  }
  float4 acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);

  // The next tile's K/V chunks are loaded into registers while the current
  // tile is scored from shared memory.
  uint4 kr[LPT], vr[LPT];
  auto load = [&](int t0) {
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      const int i = tid + j * AR_THREADS, row = i / CPR, c = i % CPR;
      if (i < AR_TILE * CPR && t0 + row < j1) {
        const size_t off = (size_t)(t0 + row) * kd + (size_t)g * HD + c * CE;
        kr[j] = __ldcs(reinterpret_cast<const uint4*>(K + off));
        vr[j] = __ldcs(reinterpret_cast<const uint4*>(V + off));
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
        Chunk<KV>::widen(kr[j], kf);
        Chunk<KV>::widen(vr[j], vf);
#pragma unroll
        for (int h4 = 0; h4 < CE / 4; ++h4) {
          const int c4 = c * (CE / 4) + h4;
          ks[row][ar_swz<HD>(row, c4)] = make_float4(kf[4 * h4], kf[4 * h4 + 1], kf[4 * h4 + 2], kf[4 * h4 + 3]);
          vs[row][c4] = make_float4(vf[4 * h4], vf[4 * h4 + 1], vf[4 * h4 + 2], vf[4 * h4 + 3]);
        }
      }
    }
    __syncthreads();
    if (t0 + AR_TILE < j1) load(t0 + AR_TILE);
    // Scores: warp per head, lane per key; float4 reads of the key row and a
    // broadcast of the query.
    for (int hh = warp; hh < G; hh += AR_THREADS / 32) {
      float s = -INFINITY;
      if (lane < nt) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
        for (int c = 0; c < C4; ++c) {
          const float4 kv = ks[lane][ar_swz<HD>(lane, c)], qv = qs[hh][c];
          s0 = fmaf(qv.x, kv.x, s0);
          s1 = fmaf(qv.y, kv.y, s1);
          s0 = fmaf(qv.z, kv.z, s0);
          s1 = fmaf(qv.w, kv.w, s1);
        }
        s = s0 + s1;
      }
      const float mnew = fmaxf(mrow[hh], warp_max(s));
      const float e = lane < nt ? __expf(s - mnew) : 0.f;
      const float esum = warp_sum(e);
      ps[hh][lane] = e;
      __syncwarp();
      if (lane == 0) {
        const float a = __expf(mrow[hh] - mnew);
        alpha[hh] = a;
        lrow[hh] = lrow[hh] * a + esum;
        mrow[hh] = mnew;
      }
    }
    __syncthreads();
    // Weighted sum of V: slot (head, float4 chunk) per thread.
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int slot = tid + r * AR_THREADS;
      if (slot < G * C4) {
        const int hh = slot / C4, c = slot % C4;
        const float a = alpha[hh];
        float4 o = acc[r];
        o.x *= a;
        o.y *= a;
        o.z *= a;
        o.w *= a;
        for (int j = 0; j < nt; ++j) {
          const float pj = ps[hh][j];
          const float4 v = vs[j][c];
          o.x = fmaf(pj, v.x, o.x);
          o.y = fmaf(pj, v.y, o.y);
          o.z = fmaf(pj, v.z, o.z);
          o.w = fmaf(pj, v.w, o.w);
        }
        acc[r] = o;
      }
    }
  }
  __syncthreads();
  // part[((b*nq + head) * nsplit + split) * (HD+2) + {0..HD-1: output, HD: max, HD+1: sum}];
  // an empty split leaves (-inf, 0, zeros), which the merge skips.
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int slot = tid + r * AR_THREADS;
    if (slot < G * C4) {
      const int hh = slot / C4, c = slot % C4;
      float* pp = part + (((size_t)b * nq + g * G + hh) * nsplit + split) * (HD + 2) + 4 * c;
      pp[0] = acc[r].x;
      pp[1] = acc[r].y;
      pp[2] = acc[r].z;
      pp[3] = acc[r].w;
    }
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

template <typename KV, int HD>
static void attn_rows(const dec_config& c, const float* Q, const void* kc, const void* vc, size_t ring_bytes,
                      const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, RowOut out,
                      cudaStream_t s) {
  const dim3 grid(c.n_kv_heads, nsplit, B);
  k_attn_rows<KV, HD><<<grid, AR_THREADS, 0, s>>>(Q, (const KV*)kc, (const KV*)vc, ring_bytes / sizeof(KV), seq,
                                                  pos, c.n_heads, c.n_kv_heads, c.max_seq, c.sliding_window, part);
  k_attn_rows_merge<HD><<<dim3(c.n_heads, B), HD, 0, s>>>(part, c.n_heads, nsplit, out);
}

void launch_attn_rows(const dec_config& c, const float* Q, const void* kc, const void* vc, size_t ring_bytes,
                      const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, RowOut out,
                      cudaStream_t s) {
  const bool kb = c.kv_dtype == DEC_BF16;
  switch (c.head_dim) {
    case 16:
      kb ? attn_rows<__nv_bfloat16, 16>(c, Q, kc, vc, ring_bytes, seq, pos, B, nsplit, part, out, s)
         : attn_rows<float, 16>(c, Q, kc, vc, ring_bytes, seq, pos, B, nsplit, part, out, s);
      break;
    case 64:
      kb ? attn_rows<__nv_bfloat16, 64>(c, Q, kc, vc, ring_bytes, seq, pos, B, nsplit, part, out, s)
         : attn_rows<float, 64>(c, Q, kc, vc, ring_bytes, seq, pos, B, nsplit, part, out, s);
      break;
    default:
      kb ? attn_rows<__nv_bfloat16, 128>(c, Q, kc, vc, ring_bytes, seq, pos, B, nsplit, part, out, s)
         : attn_rows<float, 128>(c, Q, kc, vc, ring_bytes, seq, pos, B, nsplit, part, out, s);
  }
}

}  // namespace dec
