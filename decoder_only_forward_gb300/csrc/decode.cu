// Decode (one position) kernels: bandwidth-bound fused GEMVs, split-K
// flash-decode GQA attention, MoE router/top-k and expert GEMVs, LM head with
// device argmax.  Weights stream once per step with 16-byte loads; every dot
// product is one warp over the K dimension with fp32 accumulation.
#include <math.h>

#include "runtime.h"

namespace dec {

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_WARPS = GEMV_THREADS / 32;

// ---------------------------------------------------------------------------
// Block-level helpers

// xs[k] = x[k] / sqrt(mean(x^2) + eps) * w[k]   (Pantheon RMSNorm)
__device__ void block_rmsnorm_to_smem(const float* __restrict__ x, const float* __restrict__ w,
                                      int K, float eps, float* xs, float* red) {
  float ss = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    float v = x[k];
    xs[k] = v;
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < nwarps ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[32] / (float)K + eps);
  for (int k = threadIdx.x; k < K; k += blockDim.x) xs[k] = xs[k] * inv * w[k];
  __syncthreads();
}

__device__ void block_copy_to_smem(const float* __restrict__ x, int K, float* xs) {
  for (int k = threadIdx.x; k < K; k += blockDim.x) xs[k] = x[k];
  __syncthreads();
}

// Partial dot products of two weight rows with the smem vector xs over the
// chunks c = c0, c0+32, ... (c0 = lane + 32*i0); K * sizeof(W) is a multiple
// of 16 bytes.  Accumulates into a0, a1 (no reduction).
template <typename W>
__device__ __forceinline__ void warp_dot2_acc(const W* __restrict__ r0, const W* __restrict__ r1,
                                              const float* __restrict__ xs, int K, int c, float& a0, float& a1) {
  // Up to U chunks per lane are in flight at once; the bound checks are
  // predicates, so short rows (K of a few hundred) still issue every load
  // before the first use instead of one DRAM round trip per chunk.
  constexpr int V = Chunk<W>::N, U = 6;
  const int nch = K / V;
  for (; c < nch; c += 32 * U) {
    uint4 u0[U], u1[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int cc = c + 32 * i;
      if (cc < nch) {
        u0[i] = ld_stream16(r0 + (size_t)cc * V);
        u1[i] = ld_stream16(r1 + (size_t)cc * V);
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int cc = c + 32 * i;
      if (cc < nch) {
        float w0[V], w1[V];
        Chunk<W>::widen(u0[i], w0);
        Chunk<W>::widen(u1[i], w1);
        const float* xv = xs + cc * V;
#pragma unroll
        for (int e = 0; e < V; ++e) {
          a0 = fmaf(w0[e], xv[e], a0);
          a1 = fmaf(w1[e], xv[e], a1);
        }
      }
    }
  }
}

// Dot products of two weight rows with xs, one warp; sums in every lane.
template <typename W>
__device__ __forceinline__ void warp_dot2(const W* __restrict__ r0, const W* __restrict__ r1,
                                          const float* __restrict__ xs, int K, float& s0, float& s1) {
  float a0 = 0.f, a1 = 0.f;
  warp_dot2_acc(r0, r1, xs, K, threadIdx.x & 31, a0, a1);
  s0 = warp_sum(a0);
  s1 = warp_sum(a1);
}

// The first PF chunks per lane of a warp's first row pair, loaded before the
// kernel waits on its predecessor (weights are never written, so this overlaps
// the previous kernel).
constexpr int PF = 4;
struct RowPf {
  uint4 a[PF], b[PF];
};

template <typename W>
__device__ __forceinline__ void prefetch_pair(const W* __restrict__ r0, const W* __restrict__ r1, int K, RowPf& pf) {
  constexpr int V = Chunk<W>::N;
  const int nch = K / V, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < PF; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      pf.a[i] = ld_stream16(r0 + (size_t)c * V);
      pf.b[i] = ld_stream16(r1 + (size_t)c * V);
    }
  }
}

// warp_dot2 whose first PF chunks per lane come from a prefetch.
template <typename W>
__device__ __forceinline__ void warp_dot2_pf(const W* __restrict__ r0, const W* __restrict__ r1,
                                             const float* __restrict__ xs, int K, const RowPf& pf, float& s0,
                                             float& s1) {
  constexpr int V = Chunk<W>::N;
  const int nch = K / V, lane = threadIdx.x & 31;
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < PF; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      float w0[V], w1[V];
      Chunk<W>::widen(pf.a[i], w0);
      Chunk<W>::widen(pf.b[i], w1);
      const float* xv = xs + c * V;
#pragma unroll
      for (int e = 0; e < V; ++e) {
        a0 = fmaf(w0[e], xv[e], a0);
        a1 = fmaf(w1[e], xv[e], a1);
      }
    }
  }
  warp_dot2_acc(r0, r1, xs, K, lane + 32 * PF, a0, a1);
  s0 = warp_sum(a0);
  s1 = warp_sum(a1);
}

// ---------------------------------------------------------------------------
// Step setup: position, token, RoPE (cos, sin) of this position.

__global__ void k_set_step(DeviceState* st, const int32_t* d_token, int32_t token, int32_t pos,
                           int32_t vocab, const double* __restrict__ inv_freq, int half,
                           float2* __restrict__ rope_tab) {
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    int t = d_token ? *d_token : token;
    if (t < 0 || t >= vocab) {
      raise_error(st, ERR_TOKEN, 0);
      t = 0;
    }
    st->token = t;
    st->pos = pos;
  }
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    double sn, cs;
    sincos((double)pos * inv_freq[i], &sn, &cs);
    rope_tab[i] = make_float2((float)cs, (float)sn);
  }
}

// ---------------------------------------------------------------------------
// Fused RMSNorm -> [q;k;v] = Wqkv n (+b) -> RoPE on q,k -> K/V written at the
// slot of pos.  A warp owns rows (2i, 2i+1), so the rotation of the pair is
// done in the epilogue (sipllm adjacent-pair RoPE).

template <typename W, typename KV>
__global__ void __launch_bounds__(GEMV_THREADS) k_norm_qkv(
    const float* __restrict__ x, const W* __restrict__ embed, float* __restrict__ x_out,
    const float* __restrict__ nw, float eps, const W* __restrict__ wqkv, const float* __restrict__ bqkv, int K,
    int qd, int kd, int hd, const float2* __restrict__ rope_tab, const DeviceState* __restrict__ st, int max_seq,
    int sliding, float* __restrict__ q_out, KV* __restrict__ kc, KV* __restrict__ vc) {
  extern __shared__ float sm[];
  float* red = sm;
  float* xs = sm + 64;
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int npairs = (qd + 2 * kd) / 2;
  const int p0 = blockIdx.x * GEMV_WARPS + warp;
  RowPf pf;
  if (p0 < npairs) prefetch_pair(wqkv + (size_t)2 * p0 * K, wqkv + (size_t)(2 * p0 + 1) * K, K, pf);
  pdl_wait();
  if (embed) {
    // First layer: the residual starts as the token's embedding row (Pantheon
    // Forward Pass Flow, embed); CTA 0 stores it for the later kernels.
    const W* row = embed + (size_t)st->token * K;
    float* xe = xs;  // staged in xs, then normalised in place below
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      const float v = to_f32(row[k]);
      xe[k] = v;
      if (blockIdx.x == 0) x_out[k] = v;
    }
    __syncthreads();
    x = xe;
  }
  block_rmsnorm_to_smem(x, nw, K, eps, xs, red);
  const int pos = st->pos;
  const int slot = sliding > 0 ? pos % max_seq : pos;
  const int stride = gridDim.x * GEMV_WARPS;
  for (int p = p0; p < npairs; p += stride) {
    const int r = 2 * p;
    RowPf nxt;   // next pair's rows are in flight while this pair is reduced
    if (p + stride < npairs)
      prefetch_pair(wqkv + (size_t)2 * (p + stride) * K, wqkv + (size_t)(2 * (p + stride) + 1) * K, K, nxt);
    float a0, a1;
    warp_dot2_pf(wqkv + (size_t)r * K, wqkv + (size_t)(r + 1) * K, xs, K, pf, a0, a1);
    pf = nxt;
    if (lane == 0) {
      if (bqkv) {
        a0 += bqkv[r];
        a1 += bqkv[r + 1];
      }
      if (r < qd + kd) {
        const int d = (r < qd ? r : r - qd) % hd;
        const float2 cs = rope_tab[d >> 1];
        const float b0 = a0 * cs.x - a1 * cs.y;
        const float b1 = a0 * cs.y + a1 * cs.x;
        a0 = b0;
        a1 = b1;
      }
      if (r < qd) {
        q_out[r] = a0;
        q_out[r + 1] = a1;
      } else if (r < qd + kd) {
        const size_t o = (size_t)slot * kd + (r - qd);
        kc[o] = from_f32<KV>(a0);
        kc[o + 1] = from_f32<KV>(a1);
      } else {
        const size_t o = (size_t)slot * kd + (r - qd - kd);
        vc[o] = from_f32<KV>(a0);
        vc[o + 1] = from_f32<KV>(a1);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Fused RMSNorm (or a given normalised vector) -> act = silu(Wg n) * (Wu n).
// Dense: one matrix [2f, K] with gate row r at 2r and up row r at 2r+1.
// MoE: slot s uses expert ids[s] of the merged [E, 2f, K] tensor; act is [k][f].

template <typename W>
__global__ void __launch_bounds__(GEMV_THREADS) k_gateup(
    const float* __restrict__ x, const float* __restrict__ nw, float eps,
    const float* __restrict__ nvec, const W* __restrict__ wgu, int K, int f,
    const int32_t* __restrict__ ids, int nslots, float* __restrict__ act) {
  extern __shared__ float sm[];
  float* red = sm;
  float* xs = sm + 64;
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ntask = nslots * f;
  const int p0 = blockIdx.x * GEMV_WARPS + warp;
  RowPf pf;
  const bool pre = ids == nullptr && p0 < ntask;   // expert rows are known only after the router
  if (pre) prefetch_pair(wgu + (size_t)2 * p0 * K, wgu + (size_t)(2 * p0 + 1) * K, K, pf);
  pdl_wait();
  if (nvec) block_copy_to_smem(nvec, K, xs);
  else block_rmsnorm_to_smem(x, nw, K, eps, xs, red);
  const int stride = gridDim.x * GEMV_WARPS;
  for (int p = p0; p < ntask; p += stride) {
    const int slot = p / f, j = p - slot * f;
    const size_t e = ids ? (size_t)ids[slot] : 0;
    const W* base = wgu + e * (size_t)2 * f * K + (size_t)2 * j * K;
    float g, u;
    if (pre) {
      RowPf nxt;
      if (p + stride < ntask) prefetch_pair(wgu + (size_t)2 * (p + stride) * K, wgu + (size_t)(2 * (p + stride) + 1) * K, K, nxt);
      warp_dot2_pf(base, base + K, xs, K, pf, g, u);
      pf = nxt;
    } else {
      warp_dot2(base, base + K, xs, K, g, u);
    }
    if (lane == 0) act[(size_t)slot * f + j] = silu_f(g) * u;
  }
}

// ---------------------------------------------------------------------------
// x[r] += sum_s wt_s * (W_s[r] . v_s)  -- output projection (one slot, weight 1)
// and dense / MoE down projection.  Slots are summed in selection order.

template <typename W>
__global__ void __launch_bounds__(GEMV_THREADS) k_gemv_accum(
    const float* __restrict__ v, const W* __restrict__ w, int N, int K,
    const int32_t* __restrict__ ids, const float* __restrict__ wts, int nslots,
    float* __restrict__ x, const float* __restrict__ part, int psplit, int phd) {
  extern __shared__ float sm[];
  float* xs = sm + 64;
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int npairs = (N + 1) / 2;
  const int p0 = blockIdx.x * GEMV_WARPS + warp;
  RowPf pf;
  const bool pre = ids == nullptr && nslots == 1 && p0 < npairs;
  if (pre) prefetch_pair(w + (size_t)2 * p0 * K, w + (size_t)min(2 * p0 + 1, N - 1) * K, K, pf);
  pdl_wait();
  if (part) {
    // Input = attention output merged from its split-K partials (max, sum,
    // unnormalised output per split; rml Attend's online-softmax state).
    // Phase 1: a warp per head turns the splits' (max, sum) into weights
    // exp(m_s - M) / L in shared memory; phase 2: every output sums its splits.
    float* scale = sm + 64 + K;   // [heads][psplit]
    const int heads = K / phd;
    for (int hh = warp; hh < heads; hh += GEMV_WARPS) {
      const float* base = part + (size_t)hh * psplit * (phd + 2);
      float mloc = -INFINITY;
      for (int s2 = lane; s2 < psplit; s2 += 32) mloc = fmaxf(mloc, base[s2 * (phd + 2) + phd]);
      const float M = warp_max(mloc);
      float lsum = 0.f;
      for (int s2 = lane; s2 < psplit; s2 += 32) {
        const float ms = base[s2 * (phd + 2) + phd];
        const float sc = ms == -INFINITY ? 0.f : __expf(ms - M);
        scale[hh * psplit + s2] = sc;
        lsum = fmaf(base[s2 * (phd + 2) + phd + 1], sc, lsum);
      }
      const float L = warp_sum(lsum);
      __syncwarp();
      for (int s2 = lane; s2 < psplit; s2 += 32) scale[hh * psplit + s2] /= L;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < K; idx += blockDim.x) {
      const int hh = idx / phd, d = idx - hh * phd;
      const float* base = part + (size_t)hh * psplit * (phd + 2) + d;
      const float* sc = scale + hh * psplit;
      float o = 0.f;
#pragma unroll 8
      for (int s2 = 0; s2 < psplit; ++s2) o = fmaf(sc[s2], base[(size_t)s2 * (phd + 2)], o);
      xs[idx] = o;
    }
    __syncthreads();
  } else {
    block_copy_to_smem(v, K * nslots, xs);
  }
  const int stride = gridDim.x * GEMV_WARPS;
  for (int p = p0; p < npairs; p += stride) {
    const int r0 = 2 * p;
    const int r1 = min(r0 + 1, N - 1);
    float o0 = 0.f, o1 = 0.f;
    RowPf nxt;
    if (pre && p + stride < npairs)
      prefetch_pair(w + (size_t)2 * (p + stride) * K, w + (size_t)min(2 * (p + stride) + 1, N - 1) * K, K, nxt);
    for (int s = 0; s < nslots; ++s) {
      const size_t e = ids ? (size_t)ids[s] : 0;
      const W* base = w + e * (size_t)N * K;
      float a0, a1;
      if (pre) warp_dot2_pf(base + (size_t)r0 * K, base + (size_t)r1 * K, xs, K, pf, a0, a1);
      else warp_dot2(base + (size_t)r0 * K, base + (size_t)r1 * K, xs + (size_t)s * K, K, a0, a1);
      const float ws = wts ? wts[s] : 1.0f;
      o0 = fmaf(ws, a0, o0);
      o1 = fmaf(ws, a1, o1);
    }
    if (lane == 0) {
      x[r0] += o0;
      if (r1 != r0) x[r1] += o1;
    }
    if (pre) pf = nxt;
  }
}

// ---------------------------------------------------------------------------
// MoE router: RMSNorm -> logits = Wr n -> top-k by repeated selection (ties to
// the lower id) -> weights renormalised over the selection (Pantheon Mixture
// of Experts; rml Mixture of experts).  The softmax denominator over all
// experts cancels in the renormalisation, so weights are
// exp(l_e - M) / sum_sel exp(l_s - M).  One CTA.

template <typename W>
__global__ void __launch_bounds__(GEMV_THREADS) k_moe_router(
    const float* __restrict__ x, const float* __restrict__ nw, float eps,
    const W* __restrict__ router, int K, int E, int k, float* __restrict__ nvec,
    int32_t* __restrict__ ids, float* __restrict__ wts, const DeviceState* __restrict__ st,
    int32_t* __restrict__ trace_ids, float* __restrict__ trace_logits, int trace_cap, int layer) {
  extern __shared__ float sm[];
  float* red = sm;
  float* logits = sm + 64;               // [E] (E <= 256 -> fits in the 64+256 header)
  float* xs = sm + 64 + MAX_EXPERTS;
  pdl_launch_dependents();
  pdl_wait();
  block_rmsnorm_to_smem(x, nw, K, eps, xs, red);
  for (int i = threadIdx.x; i < K; i += blockDim.x) nvec[i] = xs[i];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = warp; e < E; e += GEMV_WARPS) {
    float a, b;
    const W* row = router + (size_t)e * K;
    warp_dot2(row, row, xs, K, a, b);
    if (lane == 0) logits[e] = a;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int sel[MAX_EXPERTS_USED];
    float mx = -INFINITY;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        bool taken = false;
        for (int t = 0; t < j; ++t) taken |= (sel[t] == e);
        if (taken) continue;
        if (best < 0 || logits[e] > logits[best]) best = e;
      }
      sel[j] = best;
      mx = fmaxf(mx, logits[best]);
    }
    float p[MAX_EXPERTS_USED], tot = 0.f;
    for (int j = 0; j < k; ++j) {
      p[j] = expf(logits[sel[j]] - mx);
      tot += p[j];
    }
    for (int j = 0; j < k; ++j) {
      ids[j] = sel[j];
      wts[j] = p[j] / tot;
    }
    if (trace_ids) {
      const size_t row = (size_t)layer * trace_cap + (st->pos % trace_cap);
      for (int j = 0; j < k; ++j) trace_ids[row * k + j] = sel[j];
      for (int e = 0; e < E; ++e) trace_logits[row * E + e] = logits[e];
    }
  }
}

// ---------------------------------------------------------------------------
// Split-K flash-decode: CTA (g, split) handles the G query heads of kv head g
// over a contiguous share of the readable slots, with a one-pass online
// softmax (rml Attend).  The last CTA of a kv head merges the partial
// (max, sum, output) triples in split order.  Key order does not change the
// softmax, so slots are visited in slot order; the readable count is
// min(pos+1, max_seq) under a window (Pantheon Sliding Window), else pos+1.

constexpr int FD_THREADS = 128;
constexpr int FD_TILE = 32;

template <typename KV, int HD>
__global__ void __launch_bounds__(FD_THREADS) k_flash_decode(
    const float* __restrict__ q, const KV* __restrict__ kc, const KV* __restrict__ vc, int nq,
    int nkv, int max_seq, int sliding, DeviceState* __restrict__ st, float* __restrict__ part,
    float* __restrict__ out) {
  constexpr int OUTS = (MAX_GROUP * HD + FD_THREADS - 1) / FD_THREADS;
  __shared__ float qs[MAX_GROUP][HD];
  __shared__ float ks[FD_TILE][HD + 1];
  __shared__ __align__(16) float vs[FD_TILE][HD];
  __shared__ float ps[MAX_GROUP][FD_TILE];
  __shared__ float mrow[MAX_GROUP], lrow[MAX_GROUP], alpha[MAX_GROUP];
  __shared__ int is_last;

  const int g = blockIdx.x, split = blockIdx.y, nsplit = gridDim.y;
  const int G = nq / nkv;
  const int kd = nkv * HD;
  const int pos = st->pos;
  const int m = sliding > 0 ? min(pos + 1, max_seq) : pos + 1;
  const int per = (m + nsplit - 1) / nsplit;
  const int j0 = split * per, j1 = min(m, j0 + per);
  const float scale = 1.0f / sqrtf((float)HD);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < G * HD; i += FD_THREADS) qs[i / HD][i % HD] = q[(size_t)g * G * HD + i] * scale;
  if (tid < MAX_GROUP) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.f;
  }
  float acc[OUTS];
#pragma unroll
  for (int r = 0; r < OUTS; ++r) acc[r] = 0.f;

  constexpr int CV = 16 / sizeof(KV);  // elements per 16-byte chunk
  for (int t0 = j0; t0 < j1; t0 += FD_TILE) {
    const int nt = min(FD_TILE, j1 - t0);
    __syncthreads();
    for (int i = tid; i < nt * (HD / CV); i += FD_THREADS) {
      const int row = i / (HD / CV), c = i % (HD / CV);
      const size_t off = (size_t)(t0 + row) * kd + (size_t)g * HD + c * CV;
      float kf[CV], vf[CV];
      Chunk<KV>::widen(*reinterpret_cast<const uint4*>(kc + off), kf);
      Chunk<KV>::widen(*reinterpret_cast<const uint4*>(vc + off), vf);
#pragma unroll
      for (int e = 0; e < CV; ++e) {
        ks[row][c * CV + e] = kf[e];
        vs[row][c * CV + e] = vf[e];
      }
    }
    __syncthreads();
    for (int hh = warp; hh < G; hh += FD_THREADS / 32) {
      float s = -INFINITY;
      if (lane < nt) {
        s = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; ++d) s = fmaf(qs[hh][d], ks[lane][d], s);
      }
      const float mnew = fmaxf(mrow[hh], warp_max(s));
      const float p = lane < nt ? __expf(s - mnew) : 0.f;
      const float psum = warp_sum(p);
      ps[hh][lane] = p;
      __syncwarp();
      if (lane == 0) {
        const float a = __expf(mrow[hh] - mnew);
        alpha[hh] = a;
        lrow[hh] = lrow[hh] * a + psum;
        mrow[hh] = mnew;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < OUTS; ++r) {
      const int idx = tid + r * FD_THREADS;
      if (idx < G * HD) {
        const int hh = idx / HD, d = idx % HD;
        float o = acc[r] * alpha[hh];
        for (int j = 0; j < nt; ++j) o = fmaf(ps[hh][j], vs[j][d], o);
        acc[r] = o;
      }
    }
  }
  __syncthreads();

  if (nsplit == 1) {
#pragma unroll
    for (int r = 0; r < OUTS; ++r) {
      const int idx = tid + r * FD_THREADS;
      if (idx < G * HD) out[(size_t)g * G * HD + idx] = acc[r] / lrow[idx / HD];
    }
    return;
  }
  // Partials: part[(h * nsplit + split) * (HD + 2) + {0..HD-1: o, HD: max, HD+1: sum}]
#pragma unroll
  for (int r = 0; r < OUTS; ++r) {
    const int idx = tid + r * FD_THREADS;
    if (idx < G * HD) {
      const int hh = idx / HD, d = idx % HD;
      part[((size_t)(g * G + hh) * nsplit + split) * (HD + 2) + d] = acc[r];
    }
  }
  if (tid < G) {
    float* pp = part + ((size_t)(g * G + tid) * nsplit + split) * (HD + 2);
    pp[HD] = mrow[tid];
    pp[HD + 1] = lrow[tid];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&st->counters[CNT_ATTN + g], 1u);
    is_last = (prev == (unsigned)nsplit - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int idx = tid; idx < G * HD; idx += FD_THREADS) {
    const int hh = idx / HD, d = idx % HD;
    const float* base = part + (size_t)(g * G + hh) * nsplit * (HD + 2);
    float M = -INFINITY;
    for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, __ldcg(base + s2 * (HD + 2) + HD));
    float L = 0.f, o = 0.f;
    for (int s2 = 0; s2 < nsplit; ++s2) {
      const float* pp = base + s2 * (HD + 2);
      const float ms = __ldcg(pp + HD);
      if (ms == -INFINITY) continue;
      const float sc = __expf(ms - M);
      L = fmaf(__ldcg(pp + HD + 1), sc, L);
      o = fmaf(__ldcg(pp + d), sc, o);
    }
    out[(size_t)(g * G + hh) * HD + d] = o / L;
  }
  if (tid == 0) st->counters[CNT_ATTN + g] = 0u;
}

// ---------------------------------------------------------------------------
// Decode attention with the KV history prefetched before the dependency wait.
// CTA (g, split) owns the fixed slot range [split*sps, split*sps + sps) of kv
// head g, processed in chunks of AD_KS keys.  Before pdl_wait() it starts
// cp.async copies of the first chunk's slots that earlier steps wrote (bounded
// by the position recorded so far, a hint that can only be one step stale);
// after the wait it copies what is missing plus the current position's slot
// (written by the preceding QKV kernel), then scores, online softmax and the
// weighted sum of V (rml Attend).  The last CTA of a kv head merges the
// per-split (max, sum, output) triples in split order.

constexpr int AD_THREADS = 128;
constexpr int AD_KS = 64;

template <typename KV, int HD>
struct AdLayout {
  static constexpr int CE = 16 / sizeof(KV);   // elements per 16-byte chunk
  static constexpr int KROW = HD + CE;         // padded K row (keeps 16-byte alignment)
  static constexpr int CPR = HD / CE;          // chunks per row
  static size_t bytes(int G) {
    return sizeof(KV) * (size_t)AD_KS * (KROW + HD) + sizeof(float) * ((size_t)G * HD + (size_t)G * AD_KS) + 16;
  }
};

template <typename KV, int HD>
__global__ void __launch_bounds__(AD_THREADS) k_attn_decode(
    const float* __restrict__ q, const KV* __restrict__ kc, const KV* __restrict__ vc, int nq, int nkv,
    int max_seq, int sliding, int sps, DeviceState* __restrict__ st, float* __restrict__ part,
    float* __restrict__ out, int merge_here) {
  using L = AdLayout<KV, HD>;
  constexpr int OUTS = (MAX_GROUP * HD + AD_THREADS - 1) / AD_THREADS;
  extern __shared__ __align__(16) uint8_t ad_smem[];
  const int G = nq / nkv;
  KV* ks = reinterpret_cast<KV*>(ad_smem);
  KV* vs = ks + AD_KS * L::KROW;
  float* qs = reinterpret_cast<float*>(vs + AD_KS * HD);
  float* ps = qs + G * HD;
  __shared__ float mrow[MAX_GROUP], lrow[MAX_GROUP], alpha[MAX_GROUP];

  pdl_launch_dependents();
  const int g = blockIdx.x, split = blockIdx.y, nsplit = gridDim.y;
  const int kd = nkv * HD, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s0 = split * sps, s1 = min(s0 + sps, max_seq);

  // Prefetch (before the wait): slots below the readable count of the last
  // recorded position.  Only ever-written slots of earlier steps are read.
  const int hint = *reinterpret_cast<volatile const int*>(&st->pos);
  const int m_hint = hint < 0 ? 0 : (sliding > 0 ? min(hint + 1, max_seq) : min(hint + 1, max_seq));
  const int pre_end = max(s0, min(min(s0 + AD_KS, s1), m_hint));
  for (int i = tid; i < (pre_end - s0) * L::CPR; i += AD_THREADS) {
    const int r = i / L::CPR, c = i % L::CPR;
    const size_t go = (size_t)(s0 + r) * kd + (size_t)g * HD + c * L::CE;
    cp_async16(ks + r * L::KROW + c * L::CE, kc + go);
    cp_async16(vs + r * HD + c * L::CE, vc + go);
  }
  cp_async_commit();
  pdl_wait();
  cp_async_wait_all();

  const int pos = st->pos;
  const int m = sliding > 0 ? min(pos + 1, max_seq) : pos + 1;
  const int cur = sliding > 0 ? pos % max_seq : pos;
  const int j1 = min(s1, m);
  const float scale = 1.0f / sqrtf((float)HD);
  for (int i = tid; i < G * HD; i += AD_THREADS) qs[i] = q[(size_t)g * G * HD + i] * scale;
  if (tid < MAX_GROUP) {
    mrow[tid] = -INFINITY;
    lrow[tid] = 0.f;
  }
  float acc[OUTS];
#pragma unroll
  for (int r = 0; r < OUTS; ++r) acc[r] = 0.f;

  for (int c0 = s0; c0 < j1; c0 += AD_KS) {
    const int nt = min(AD_KS, j1 - c0);
    const int have = c0 == s0 ? min(pre_end - s0, nt) : 0;
    if (c0 != s0) __syncthreads();   // the previous chunk's readers are done
    for (int i = tid; i < (nt - have) * L::CPR; i += AD_THREADS) {
      const int r = have + i / L::CPR, c = i % L::CPR;
      const size_t go = (size_t)(c0 + r) * kd + (size_t)g * HD + c * L::CE;
      cp_async16(ks + r * L::KROW + c * L::CE, kc + go);
      cp_async16(vs + r * HD + c * L::CE, vc + go);
    }
    if (cur >= c0 && cur - c0 < have) {   // the current slot was prefetched before it was written
      const int r = cur - c0;
      for (int c = tid; c < L::CPR; c += AD_THREADS) {
        const size_t go = (size_t)cur * kd + (size_t)g * HD + c * L::CE;
        cp_async16(ks + r * L::KROW + c * L::CE, kc + go);
        cp_async16(vs + r * HD + c * L::CE, vc + go);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int idx = tid; idx < G * nt; idx += AD_THREADS) {
      const int hh = idx / nt, j = idx - hh * nt;
      const float* qv = qs + hh * HD;
      const KV* kr = ks + j * L::KROW;
      float sdot = 0.f;
#pragma unroll 8
      for (int d = 0; d < HD; ++d) sdot = fmaf(qv[d], to_f32(kr[d]), sdot);
      ps[hh * AD_KS + j] = sdot;
    }
    __syncthreads();
    for (int hh = warp; hh < G; hh += AD_THREADS / 32) {
      float* pr = ps + hh * AD_KS;
      const float sa = lane < nt ? pr[lane] : -INFINITY;
      const float sb = lane + 32 < nt ? pr[lane + 32] : -INFINITY;
      const float mnew = fmaxf(mrow[hh], warp_max(fmaxf(sa, sb)));
      const float pa = lane < nt ? __expf(sa - mnew) : 0.f;
      const float pb = lane + 32 < nt ? __expf(sb - mnew) : 0.f;
      const float psum = warp_sum(pa + pb);
      if (lane < nt) pr[lane] = pa;
      if (lane + 32 < nt) pr[lane + 32] = pb;
      __syncwarp();
      if (lane == 0) {
        const float a = __expf(mrow[hh] - mnew);
        alpha[hh] = a;
        lrow[hh] = lrow[hh] * a + psum;
        mrow[hh] = mnew;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < OUTS; ++r) {
      const int idx = tid + r * AD_THREADS;
      if (idx < G * HD) {
        const int hh = idx / HD, d = idx - hh * HD;
        const float* pr = ps + hh * AD_KS;
        float o = acc[r] * alpha[hh];
        for (int j = 0; j < nt; ++j) o = fmaf(pr[j], to_f32(vs[j * HD + d]), o);
        acc[r] = o;
      }
    }
  }
  __syncthreads();

  if (nsplit == 1) {
#pragma unroll
    for (int r = 0; r < OUTS; ++r) {
      const int idx = tid + r * AD_THREADS;
      if (idx < G * HD) out[(size_t)g * G * HD + idx] = acc[r] / lrow[idx / HD];
    }
    return;
  }
#pragma unroll
  for (int r = 0; r < OUTS; ++r) {
    const int idx = tid + r * AD_THREADS;
    if (idx < G * HD) {
      const int hh = idx / HD, d = idx - hh * HD;
      part[((size_t)(g * G + hh) * nsplit + split) * (HD + 2) + d] = acc[r];
    }
  }
  if (tid < G) {
    float* pp = part + ((size_t)(g * G + tid) * nsplit + split) * (HD + 2);
    pp[HD] = mrow[tid];
    pp[HD + 1] = lrow[tid];
  }
  if (!merge_here) return;  // the output projection merges the splits (k_gemv_accum's prologue)
  // Large partial sets: the last CTA of kv head g merges its G heads' splits.
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = atomicAdd(&st->counters[CNT_ATTN + g], 1u) == (unsigned)nsplit - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  float* wsplit = ps;  // [G][nsplit], nsplit <= AD_KS
  for (int hh = warp; hh < G; hh += AD_THREADS / 32) {
    const float* base = part + (size_t)(g * G + hh) * nsplit * (HD + 2);
    float mloc = -INFINITY;
    for (int s2 = lane; s2 < nsplit; s2 += 32) mloc = fmaxf(mloc, __ldcg(base + s2 * (HD + 2) + HD));
    const float M = warp_max(mloc);
    float lsum = 0.f;
    for (int s2 = lane; s2 < nsplit; s2 += 32) {
      const float ms = __ldcg(base + s2 * (HD + 2) + HD);
      const float sc = ms == -INFINITY ? 0.f : __expf(ms - M);
      wsplit[hh * AD_KS + s2] = sc;
      lsum = fmaf(__ldcg(base + s2 * (HD + 2) + HD + 1), sc, lsum);
    }
    const float Lsum = warp_sum(lsum);
    __syncwarp();
    for (int s2 = lane; s2 < nsplit; s2 += 32) wsplit[hh * AD_KS + s2] /= Lsum;
  }
  __syncthreads();
  for (int idx = tid; idx < G * HD; idx += AD_THREADS) {
    const int hh = idx / HD, d = idx - hh * HD;
    const float* base = part + (size_t)(g * G + hh) * nsplit * (HD + 2) + d;
    const float* sc = wsplit + hh * AD_KS;
    float o = 0.f;
#pragma unroll 8
    for (int s2 = 0; s2 < nsplit; ++s2) o = fmaf(sc[s2], __ldcg(base + (size_t)s2 * (HD + 2)), o);
    out[(size_t)(g * G + hh) * HD + d] = o;
  }
  if (tid == 0) st->counters[CNT_ATTN + g] = 0u;
}

// ---------------------------------------------------------------------------
// Final RMSNorm -> logits = W_out n (fp32), with an optional device argmax:
// per-CTA (value, index) partials, merged by the last CTA (ties -> lower id).

template <typename W>
__global__ void __launch_bounds__(GEMV_THREADS) k_norm_lmhead(
    const float* __restrict__ x, const float* __restrict__ nw, float eps,
    const W* __restrict__ head, int K, int V, float* __restrict__ logits,
    int32_t* __restrict__ d_argmax, float* __restrict__ pval, int32_t* __restrict__ pidx,
    DeviceState* __restrict__ st) {
  extern __shared__ float sm[];
  float* red = sm;
  float* xs = sm + 64;
  __shared__ float wbest[GEMV_WARPS];
  __shared__ int wbidx[GEMV_WARPS];
  __shared__ int is_last;
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int npairs = (V + 1) / 2;
  const int p0 = blockIdx.x * GEMV_WARPS + warp;
  RowPf pf;
  if (p0 < npairs) prefetch_pair(head + (size_t)2 * p0 * K, head + (size_t)min(2 * p0 + 1, V - 1) * K, K, pf);
  pdl_wait();
  block_rmsnorm_to_smem(x, nw, K, eps, xs, red);
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  const int stride = gridDim.x * GEMV_WARPS;
  for (int p = p0; p < npairs; p += stride) {
    const int r0 = 2 * p, r1 = min(r0 + 1, V - 1);
    RowPf nxt;
    if (p + stride < npairs)
      prefetch_pair(head + (size_t)2 * (p + stride) * K, head + (size_t)min(2 * (p + stride) + 1, V - 1) * K, K, nxt);
    float a0, a1;
    warp_dot2_pf(head + (size_t)r0 * K, head + (size_t)r1 * K, xs, K, pf, a0, a1);
    pf = nxt;
    if (lane == 0) {
      if (logits) {
        logits[r0] = a0;
        if (r1 != r0) logits[r1] = a1;
      }
      if (a0 > best || (a0 == best && r0 < bidx)) { best = a0; bidx = r0; }
      if (a1 > best || (a1 == best && r1 < bidx)) { best = a1; bidx = r1; }
    }
  }
  if (!d_argmax) return;
  if (lane == 0) {
    wbest[warp] = best;
    wbidx[warp] = bidx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = wbest[0];
    int bi = wbidx[0];
    for (int w = 1; w < GEMV_WARPS; ++w)
      if (wbest[w] > b || (wbest[w] == b && wbidx[w] < bi)) { b = wbest[w]; bi = wbidx[w]; }
    pval[blockIdx.x] = b;
    pidx[blockIdx.x] = bi;
    __threadfence();
    const unsigned prev = atomicAdd(&st->counters[CNT_ARGMAX], 1u);
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  // The last CTA merges the per-CTA (value, index) partials: each thread folds
  // a strided subset, then a block reduction; ties keep the lower index.
  __threadfence();
  float b = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) {
    const float v = __ldcg(pval + i);
    const int vi = __ldcg(pidx + i);
    if (v > b || (v == b && vi < bi)) { b = v; bi = vi; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, b, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > b || (ov == b && oi < bi)) { b = ov; bi = oi; }
  }
  __syncthreads();
  if (lane == 0) {
    wbest[warp] = b;
    wbidx[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < GEMV_WARPS; ++w)
      if (wbest[w] > wbest[0] || (wbest[w] == wbest[0] && wbidx[w] < wbidx[0])) { wbest[0] = wbest[w]; wbidx[0] = wbidx[w]; }
    *d_argmax = wbidx[0];
    st->counters[CNT_ARGMAX] = 0u;
  }
}

// ---------------------------------------------------------------------------
// Standalone attention (dec_attend): position and counters live in a caller
// scratch area instead of the handle's step state.

__global__ void k_attend_setup(DeviceState* st, int32_t pos, int nkv) {
  if (threadIdx.x == 0) {
    st->pos = pos;
    st->err = 0u;
  }
  for (int g = threadIdx.x; g < nkv; g += blockDim.x) st->counters[CNT_ATTN + g] = 0u;
}

void launch_attend(const float* q, const void* kc, const void* vc, int nq, int nkv, int hd, int max_seq,
                   int sliding, int kv_dtype, int pos, int nsplit, DeviceState* st, float* part, float* out,
                   cudaStream_t s) {
  k_attend_setup<<<1, 128, 0, s>>>(st, pos, nkv);
  const dim3 grid(nkv, nsplit);
#define DEC_ATTEND_LAUNCH(KV, HD)                                                                    \
  k_flash_decode<KV, HD><<<grid, FD_THREADS, 0, s>>>(q, (const KV*)kc, (const KV*)vc, nq, nkv, max_seq, \
                                                     sliding, st, part, out)
  if (kv_dtype == DEC_BF16) {
    if (hd == 64) DEC_ATTEND_LAUNCH(__nv_bfloat16, 64);
    else if (hd == 128) DEC_ATTEND_LAUNCH(__nv_bfloat16, 128);
    else DEC_ATTEND_LAUNCH(__nv_bfloat16, 16);
  } else {
    if (hd == 64) DEC_ATTEND_LAUNCH(float, 64);
    else if (hd == 128) DEC_ATTEND_LAUNCH(float, 128);
    else DEC_ATTEND_LAUNCH(float, 16);
  }
#undef DEC_ATTEND_LAUNCH
}

// ---------------------------------------------------------------------------
// Host launchers

static inline int gemv_grid(int tasks) {
  int g = (tasks + GEMV_WARPS - 1) / GEMV_WARPS;
  const int cap = device_sm_count() * 8;
  return g < 1 ? 1 : (g > cap ? cap : g);
}

template <typename F>
static void set_smem(F* kern, size_t bytes) {
  if (bytes > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Launch with programmatic stream serialization: the kernel may start while
// its predecessor on the stream runs and orders itself with pdl_wait().
template <typename... KArgs, typename... Args>
static void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

const void* set_step_kernel() { return reinterpret_cast<const void*>(&k_set_step); }

void launch_set_step(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos) {
  k_set_step<<<1, 128, 0, s>>>(m.s.st, d_token, token, pos, m.cfg.vocab, m.s.inv_freq,
                               m.cfg.head_dim / 2, m.s.rope_tab);
  count_launch(m);
}

template <typename W>
static void lmhead(const Model& m, cudaStream_t s, const float* x, float* logits, int32_t* d_argmax) {
  const dec_config& c = m.cfg;
  const Scratch& S = m.s;
  const size_t sm_h = (64 + MAX_EXPERTS + (size_t)c.hidden) * sizeof(float);
  auto kern = k_norm_lmhead<W>;
  set_smem(kern, sm_h);
  timer_begin(m, DEC_K_LMHEAD, s);
  launch_pdl(kern, dim3(m.lm_grid), dim3(GEMV_THREADS), sm_h, s, x, m.out_norm, c.rms_eps, (const W*)m.head,
             c.hidden, c.vocab, logits, d_argmax, S.amax_val, S.amax_idx, S.st);
  timer_end(m, DEC_K_LMHEAD, s);
  count_launch(m);
}

void launch_lmhead(const Model& m, cudaStream_t s, const float* x, float* logits, int32_t* d_argmax) {
  if (m.cfg.weight_dtype == DEC_BF16) lmhead<__nv_bfloat16>(m, s, x, logits, d_argmax);
  else lmhead<float>(m, s, x, logits, d_argmax);
}

// Split partials are merged by every output-projection CTA when they are
// small, else once per kv head by the attention kernel's last CTA.
static bool merge_in_attention(const Model& m) {
  const size_t bytes = (size_t)m.cfg.n_heads * m.nsplit * (m.cfg.head_dim + 2) * sizeof(float);
  return m.nsplit > 1 && bytes > 64 * 1024;
}

template <typename KV, int HD>
static void attn_decode(const Model& m, cudaStream_t s, const LayerPtrs& L) {
  const dec_config& c = m.cfg;
  const size_t smb = AdLayout<KV, HD>::bytes(c.n_heads / c.n_kv_heads);
  auto kern = k_attn_decode<KV, HD>;
  set_smem(kern, smb);
  launch_pdl(kern, dim3(c.n_kv_heads, m.nsplit), dim3(AD_THREADS), smb, s, (const float*)m.s.q,
             (const KV*)L.kc, (const KV*)L.vc, c.n_heads, c.n_kv_heads, c.max_seq, c.sliding_window, m.attn_sps,
             m.s.st, m.s.part, m.s.attn, merge_in_attention(m) ? 1 : 0);
}

// One decode step: step state + RoPE row, then every layer, then the head.
// The first kernel orders fully after earlier stream work; every later one is
// a programmatic dependent of its predecessor.
template <typename W, typename KV>
static void decode_body(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos,
                        float* logits, int32_t* d_argmax) {
  const dec_config& c = m.cfg;
  const int h = c.hidden, hd = c.head_dim, qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  const Scratch& S = m.s;
  launch_set_step(m, s, d_token, token, pos);
  const size_t sm_h = (64 + MAX_EXPERTS + (size_t)h) * sizeof(float);
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerPtrs& L = m.layers[l];
    {
      auto kern = k_norm_qkv<W, KV>;
      set_smem(kern, sm_h);
      timer_begin(m, DEC_K_QKV, s);
      launch_pdl(kern, dim3(gemv_grid((qd + 2 * kd) / 2)), dim3(GEMV_THREADS), sm_h, s, (const float*)S.x,
                 l == 0 ? (const W*)m.tok_embd : (const W*)nullptr, S.x, L.attn_norm, c.rms_eps,
                 (const W*)L.wqkv, L.bqkv, h, qd, kd, hd, (const float2*)S.rope_tab, (const DeviceState*)S.st,
                 c.max_seq, c.sliding_window, S.q, (KV*)L.kc, (KV*)L.vc);
      timer_end(m, DEC_K_QKV, s);
      count_launch(m);
    }
    timer_begin(m, DEC_K_ATTN, s);
    if (hd == 64) attn_decode<KV, 64>(m, s, L);
    else if (hd == 128) attn_decode<KV, 128>(m, s, L);
    else attn_decode<KV, 16>(m, s, L);
    timer_end(m, DEC_K_ATTN, s);
    count_launch(m);
    {
      const size_t smb = (64 + (size_t)qd + (size_t)c.n_heads * m.nsplit) * sizeof(float);
      auto kern = k_gemv_accum<W>;
      set_smem(kern, smb);
      timer_begin(m, DEC_K_OPROJ, s);
      const bool merge = m.nsplit > 1 && !merge_in_attention(m);
      launch_pdl(kern, dim3(gemv_grid((h + 1) / 2)), dim3(GEMV_THREADS), smb, s, (const float*)S.attn,
                 (const W*)L.wo, h, qd, (const int32_t*)nullptr, (const float*)nullptr, 1, S.x,
                 merge ? (const float*)S.part : (const float*)nullptr, m.nsplit, hd);
      timer_end(m, DEC_K_OPROJ, s);
      count_launch(m);
    }
    const int f = c.ffn;
    if (c.n_experts > 0) {
      const int k = c.n_experts_used;
      {
        auto kern = k_moe_router<W>;
        set_smem(kern, sm_h);
        timer_begin(m, DEC_K_ROUTER, s);
        launch_pdl(kern, dim3(1), dim3(GEMV_THREADS), sm_h, s, (const float*)S.x, L.ffn_norm, c.rms_eps,
                   (const W*)L.router, h, c.n_experts, k, S.nbuf, S.ids, S.wts, (const DeviceState*)S.st,
                   m.trace_ids, m.trace_logits, m.trace_cap, l);
        timer_end(m, DEC_K_ROUTER, s);
        count_launch(m);
      }
      {
        auto kern = k_gateup<W>;
        set_smem(kern, sm_h);
        timer_begin(m, DEC_K_GATEUP, s);
        launch_pdl(kern, dim3(gemv_grid(k * f)), dim3(GEMV_THREADS), sm_h, s, (const float*)nullptr,
                   (const float*)nullptr, 0.f, (const float*)S.nbuf, (const W*)L.w_gateup, h, f,
                   (const int32_t*)S.ids, k, S.act);
        timer_end(m, DEC_K_GATEUP, s);
        count_launch(m);
      }
      {
        const size_t smb = (64 + (size_t)k * f) * sizeof(float);
        auto kern = k_gemv_accum<W>;
        set_smem(kern, smb);
        timer_begin(m, DEC_K_DOWN, s);
        launch_pdl(kern, dim3(gemv_grid((h + 1) / 2)), dim3(GEMV_THREADS), smb, s, (const float*)S.act,
                   (const W*)L.w_down, h, f, (const int32_t*)S.ids, (const float*)S.wts, k, S.x,
                   (const float*)nullptr, 0, 0);
        timer_end(m, DEC_K_DOWN, s);
        count_launch(m);
      }
    } else {
      {
        auto kern = k_gateup<W>;
        set_smem(kern, sm_h);
        timer_begin(m, DEC_K_GATEUP, s);
        launch_pdl(kern, dim3(gemv_grid(f)), dim3(GEMV_THREADS), sm_h, s, (const float*)S.x, L.ffn_norm,
                   c.rms_eps, (const float*)nullptr, (const W*)L.w_gateup, h, f, (const int32_t*)nullptr, 1,
                   S.act);
        timer_end(m, DEC_K_GATEUP, s);
        count_launch(m);
      }
      {
        const size_t smb = (64 + (size_t)f) * sizeof(float);
        auto kern = k_gemv_accum<W>;
        set_smem(kern, smb);
        timer_begin(m, DEC_K_DOWN, s);
        launch_pdl(kern, dim3(gemv_grid((h + 1) / 2)), dim3(GEMV_THREADS), smb, s, (const float*)S.act,
                   (const W*)L.w_down, h, f, (const int32_t*)nullptr, (const float*)nullptr, 1, S.x,
                   (const float*)nullptr, 0, 0);
        timer_end(m, DEC_K_DOWN, s);
        count_launch(m);
      }
    }
  }
  if (logits || d_argmax) lmhead<W>(m, s, S.x, logits, d_argmax);
}

void launch_decode_body(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos,
                        float* logits, int32_t* d_argmax) {
  const bool wb = m.cfg.weight_dtype == DEC_BF16, kb = m.cfg.kv_dtype == DEC_BF16;
  if (wb && kb) decode_body<__nv_bfloat16, __nv_bfloat16>(m, s, d_token, token, pos, logits, d_argmax);
  else if (wb) decode_body<__nv_bfloat16, float>(m, s, d_token, token, pos, logits, d_argmax);
  else if (kb) decode_body<float, __nv_bfloat16>(m, s, d_token, token, pos, logits, d_argmax);
  else decode_body<float, float>(m, s, d_token, token, pos, logits, d_argmax);
}

}  // namespace dec
