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

template <typename KV, int HD>
__global__ void __launch_bounds__(AR_THREADS) k_attn_rows(
    const float* __restrict__ Q, const KV* __restrict__ kc, const KV* __restrict__ vc, size_t ring_elems,
    const int32_t* __restrict__ seq, const int32_t* __restrict__ pos, int nq, int nkv, int max_seq, int sliding,
    float* __restrict__ part) {
  constexpr int OUTS = (MAX_GROUP * HD + AR_THREADS - 1) / AR_THREADS;
  constexpr int CE = 16 / sizeof(KV);   // elements per 16-byte chunk
  __shared__ float qs[MAX_GROUP][HD];
  __shared__ float ks[AR_TILE][HD + 1];
  __shared__ __align__(16) float vs[AR_TILE][HD];
  __shared__ float ps[MAX_GROUP][AR_TILE];
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

  for (int i = tid; i < G * HD; i += AR_THREADS) qs[i / HD][i % HD] = q[i] * scale;
  if (tid < MAX_GROUP) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.f;
  }
  float acc[OUTS];
#pragma unroll
  for (int r = 0; r < OUTS; ++r) acc[r] = 0.f;

  for (int t0 = j0; t0 < j1; t0 += AR_TILE) {
    const int nt = min(AR_TILE, j1 - t0);
    __syncthreads();
    for (int i = tid; i < nt * (HD / CE); i += AR_THREADS) {
      const int row = i / (HD / CE), c = i % (HD / CE);
      const size_t off = (size_t)(t0 + row) * kd + (size_t)g * HD + c * CE;
      float kf[CE], vf[CE];
      Chunk<KV>::widen(__ldcs(reinterpret_cast<const uint4*>(K + off)), kf);
      Chunk<KV>::widen(__ldcs(reinterpret_cast<const uint4*>(V + off)), vf);
#pragma unroll
      for (int e = 0; e < CE; ++e) {
        ks[row][c * CE + e] = kf[e];
        vs[row][c * CE + e] = vf[e];
      }
    }
    __syncthreads();
    // Scores: warp per head, lane per key.
    for (int hh = warp; hh < G; hh += AR_THREADS / 32) {
      float s = -INFINITY;
      if (lane < nt) {
        s = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; ++d) s = fmaf(qs[hh][d], ks[lane][d], s);
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
#pragma unroll
    for (int r = 0; r < OUTS; ++r) {
      const int idx = tid + r * AR_THREADS;
      if (idx < G * HD) {
        const int hh = idx / HD, d = idx % HD;
        float o = acc[r] * alpha[hh];
        for (int j = 0; j < nt; ++j) o = fmaf(ps[hh][j], vs[j][d], o);
        acc[r] = o;
      }
    }
  }
  __syncthreads();
  // part[((b*nq + head) * nsplit + split) * (HD+2) + {0..HD-1: output, HD: max, HD+1: sum}];
  // an empty split leaves (-inf, 0, zeros), which the merge skips.
#pragma unroll
  for (int r = 0; r < OUTS; ++r) {
    const int idx = tid + r * AR_THREADS;
    if (idx < G * HD) {
      const int hh = idx / HD, d = idx % HD;
      part[(((size_t)b * nq + g * G + hh) * nsplit + split) * (HD + 2) + d] = acc[r];
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
