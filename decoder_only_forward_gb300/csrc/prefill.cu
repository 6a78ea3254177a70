// Single-pass prefill (sipllm "Transformer forward pass", Single-pass prefill;
// rml "The decoder", Forward with n tokens): each layer runs once over all n
// rows of the chunk, positions ascending, so position t's K/V exists before any
// later query reads it.  Per layer: RMSNorm rows -> QKV GEMM (+bias, RoPE, K/V
// rows) -> causal GQA attention -> O GEMM (+residual) -> RMSNorm rows -> SwiGLU
// GEMMs (+residual) or MoE routing + grouped expert GEMMs + combine.  Only the
// last row gets the final norm and LM head.
#include <math.h>

#include "prefill_common.cuh"

namespace dec {

// ---------------------------------------------------------------------------
// Row kernels

template <typename W>
__global__ void k_embed_rows(const W* __restrict__ E, const int32_t* __restrict__ tokens, int h,
                             float* __restrict__ X) {
  const int t = blockIdx.x;
  const W* row = E + (size_t)tokens[t] * h;
  for (int i = threadIdx.x; i < h; i += blockDim.x) X[(size_t)t * h + i] = to_f32(row[i]);
}

// (cos, sin) of every rotary pair for positions start..start+n-1, in fp64 then
// rounded (rml "The decoder", One forward pass, step 3: once per position).
__global__ void k_rope_rows(const double* __restrict__ inv_freq, int half, int start, int n,
                            float2* __restrict__ tab) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n * half) return;
  const int t = i / half, p = i % half;
  double sn, cs;
  sincos((double)(start + t) * inv_freq[p], &sn, &cs);
  tab[i] = make_float2((float)cs, (float)sn);
}

// Batched decode setup: each row's sequence, position and K/V row (passed by
// value), its token id (an id outside [0, vocab) becomes 0 and raises
// ERR_TOKEN) and the (cos, sin) table of the row's own position.
__global__ void k_rows_setup(const __grid_constant__ RowsMeta meta, int B, const int32_t* __restrict__ d_tokens,
                             int32_t host_token, int vocab, const double* __restrict__ inv_freq, int half, int32_t* __restrict__ tokens,
                             int32_t* __restrict__ b_seq, int32_t* __restrict__ b_pos, int32_t* __restrict__ b_rows,
                             float2* __restrict__ tab, DeviceState* st, const double* __restrict__ inv_local,
                             float2* __restrict__ tab_local) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B) {
    int t = d_tokens ? d_tokens[i] : host_token;
    if (t < 0 || t >= vocab) {
      raise_error(st, ERR_TOKEN, 0);
      t = 0;
    }
    tokens[i] = t;
    b_seq[i] = meta.seq[i];
    b_pos[i] = meta.pos[i];
    b_rows[i] = meta.rows[i];
  }
  if (i < B * half) {
    const int r = i / half, p = i % half;
    double sn, cs;
    sincos((double)meta.pos[r] * inv_freq[p], &sn, &cs);
    tab[i] = make_float2((float)cs, (float)sn);
    if (tab_local) {   // the local layers' base (per-layer RoPE)
      sincos((double)meta.pos[r] * inv_local[p], &sn, &cs);
      tab_local[i] = make_float2((float)cs, (float)sn);
    }
  }
}

// out[r] = argmax over logits row r (ties -> lower id), one CTA per row.
__global__ void __launch_bounds__(1024) k_argmax_rows(const float* __restrict__ logits, int V,
                                                      int32_t* __restrict__ out) {
  __shared__ float bv[32];
  __shared__ int bi[32];
  const float* x = logits + (size_t)blockIdx.x * V;
  float best = -INFINITY;
  int idx = 0x7fffffff;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float v = x[i];
    if (v > best) {   // ascending i per thread: the first maximum is kept
      best = v;
      idx = i;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > best || (ov == best && oi < idx)) {
      best = ov;
      idx = oi;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    bv[warp] = best;
    bi[warp] = idx;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    best = lane < nw ? bv[lane] : -INFINITY;
    idx = lane < nw ? bi[lane] : 0x7fffffff;
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ov > best || (ov == best && oi < idx)) {
        best = ov;
        idx = oi;
      }
    }
    if (lane == 0) out[blockIdx.x] = idx == 0x7fffffff ? 0 : idx;
  }
}

// A[t] = X[t] / sqrt(mean(X[t]^2) + eps) * w, one CTA per row.
__global__ void __launch_bounds__(256) k_rmsnorm_rows(const float* __restrict__ X, const float* __restrict__ w,
                                                      float eps, int h, RowOut out) {
  __shared__ float red[33];
  const int t = blockIdx.x;
  const float* x = X + (size_t)t * h;
  // 16-byte loads and 4-wide stores when the rows allow it (few rows: latency-bound).
  const bool vec = (h & 3) == 0 && ((reinterpret_cast<uintptr_t>(w) & 15) == 0);
  float ss = 0.f;
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int i = threadIdx.x; i < h / 4; i += blockDim.x) {
      const float4 v = x4[i];
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
  } else {
    for (int i = threadIdx.x; i < h; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  }
  ss = warp_sum(ss);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[32] / (float)h + eps);
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    for (int i = threadIdx.x; i < h / 4; i += blockDim.x) {
      const float4 v = x4[i], g = w4[i];
      row_store4(out, (size_t)t * h + 4 * i,
                 make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w));
    }
  } else {
    for (int i = threadIdx.x; i < h; i += blockDim.x) row_store(out, (size_t)t * h + i, x[i] * inv * w[i]);
  }
}

// ---------------------------------------------------------------------------
// SIMT GEMM: C[M,N] = A[M,K] . B[N,K]^T with fp32 accumulation, 64x64 tiles.
// Serves f32 weights (and any shape); the tcgen05 kernel serves bf16.
// Grouped: blockIdx.z = group g, rows [off[g], off[g+1]), B advanced by g*N*K.

template <typename TA, typename TB>
__global__ void __launch_bounds__(256) k_gemm_simt(const TA* __restrict__ A, const TB* __restrict__ B, int M,
                                                   int N, int K, GemmEpi e) {
  constexpr int BM = 64, BN = 64, BK = 32;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  int row0 = 0, rows = M;
  const TB* Bg = B;
  if (e.group_offset) {
    const int g = blockIdx.z;
    row0 = e.group_offset[g];
    rows = e.group_offset[g + 1] - row0;
    Bg = B + (size_t)g * N * K;
  }
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  if (m0 >= rows) return;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += 256) {
      const int r = i / BK, c = i % BK;
      const int gr = m0 + r, gc = k0 + c;
      As[c][r] = (gr < rows && gc < K) ? to_f32(A[(size_t)(row0 + gr) * K + gc]) : 0.f;
    }
    for (int i = tid; i < BN * BK; i += 256) {
      const int r = i / BK, c = i % BK;
      const int gr = n0 + r, gc = k0 + c;
      Bs[c][r] = (gr < N && gc < K) ? to_f32(Bg[(size_t)gr * K + gc]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    if (r >= rows) continue;
    epi_pair(e, row0 + r, n0 + tx * 4, acc[i][0], acc[i][1]);
    epi_pair(e, row0 + r, n0 + tx * 4 + 2, acc[i][2], acc[i][3]);
  }
}

// ---------------------------------------------------------------------------
// Causal GQA attention over the chunk (SIMT): a warp per query row, 32 keys
// at a time (lane j scores key j, then the warp folds the tile into its online
// softmax state; rml Attend).  Keys of query position p are [lo, p] with lo = 0
// or p - W + 1; key position j is read from row (j - base_pos) of K/V.

template <typename KV, int HD>
__global__ void __launch_bounds__(256) k_attn_prefill_simt(
    const float* __restrict__ Q, const KV* __restrict__ Ks, const KV* __restrict__ Vs, int base_pos, int nq,
    int nkv, int start, int n, int sliding, RowOut O) {
  constexpr int WARPS = 8, TILE = 32, DPL = (HD + 31) / 32;
  __shared__ float ks[TILE][HD + 1];
  __shared__ float vs[TILE][HD];
  __shared__ float qs[WARPS][HD];
  const int h = blockIdx.y, g = (h * nkv) / nq;
  const int kd = nkv * HD, qd = nq * HD;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * WARPS;
  const int t = t0 + warp;
  const bool active = t < n;
  const int pos = start + t;
  const int lo = sliding > 0 ? max(0, pos - sliding + 1) : 0;
  const float scale = 1.0f / sqrtf((float)HD);
  if (active)
    for (int d = lane; d < HD; d += 32) qs[warp][d] = Q[(size_t)t * qd + h * HD + d] * scale;
  // Key range of the whole CTA.
  const int tl = min(t0 + WARPS, n) - 1;
  const int kmin = sliding > 0 ? max(0, start + t0 - sliding + 1) : 0;
  const int kmax = start + tl;
  float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;
  for (int j0 = kmin; j0 <= kmax; j0 += TILE) {
    const int nt = min(TILE, kmax - j0 + 1);
    __syncthreads();
    for (int i = threadIdx.x; i < nt * HD; i += blockDim.x) {
      const int r = i / HD, d = i % HD;
      const size_t off = (size_t)(j0 + r - base_pos) * kd + (size_t)g * HD + d;
      ks[r][d] = to_f32(Ks[off]);
      vs[r][d] = to_f32(Vs[off]);
    }
    __syncthreads();
    if (!active) continue;
    const int j = j0 + lane;
    const bool valid = lane < nt && j >= lo && j <= pos;
    float s = -INFINITY;
    if (valid) {
      s = 0.f;
#pragma unroll 8
      for (int d = 0; d < HD; ++d) s = fmaf(qs[warp][d], ks[lane][d], s);
    }
    const float tmax = warp_max(s);
    if (tmax == -INFINITY) continue;
    const float mnew = fmaxf(m, tmax);
    const float corr = __expf(m - mnew);
    const float p = valid ? __expf(s - mnew) : 0.f;
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] *= corr;
    for (int jj = 0; jj < nt; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const int d = lane + 32 * i;
        if (d < HD) o[i] = fmaf(pj, vs[jj][d], o[i]);
      }
    }
    m = mnew;
  }
  if (!active) return;
  const float inv = 1.0f / l;
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    const int d = lane + 32 * i;
    if (d < HD) row_store(O, (size_t)t * qd + h * HD + d, o[i] * inv);
  }
}

// ---------------------------------------------------------------------------
// K/V ring <-> linear rows, for chunks whose positions wrap the ring.

template <typename KV>
__global__ void k_kv_gather(const KV* __restrict__ ring_k, const KV* __restrict__ ring_v, const KvPaging pg, int seq,
                            int max_seq, int kd, int h0, int count, KV* __restrict__ lin_k, KV* __restrict__ lin_v) {
  const size_t total = (size_t)count * kd;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / kd), c = (int)(i % kd);
    const size_t src = (size_t)kv_phys_row(pg, seq, (h0 + r) % max_seq) * kd + c;
    lin_k[i] = ring_k[src];
    lin_v[i] = ring_v[src];
  }
}

template <typename KV>
__global__ void k_kv_commit(const KV* __restrict__ lin_k, const KV* __restrict__ lin_v, int lin_row0, int start,
                            int t_first, int n, int max_seq, int kd, KV* __restrict__ ring_k, KV* __restrict__ ring_v,
                            const KvPaging pg, int seq) {
  const size_t total = (size_t)(n - t_first) * kd;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = t_first + (int)(i / kd), c = (int)(i % kd);
    const size_t dst = (size_t)kv_phys_row(pg, seq, (start + t) % max_seq) * kd + c;
    const size_t src = (size_t)(lin_row0 + t) * kd + c;
    ring_k[dst] = lin_k[src];
    ring_v[dst] = lin_v[src];
  }
}

// ---------------------------------------------------------------------------
// MoE for n rows: routing per row (fp32 RMSNorm, router logits, top-k by
// repeated selection with ties to the lower id, weights renormalised over the
// selection), a stable counting sort of (row, slot) by expert, grouped expert
// GEMMs, then a combine in slot order (Pantheon Mixture of Experts; rml
// Mixture of experts; zLLM moe/prefill grouping).

template <typename W>
__global__ void __launch_bounds__(256) k_router_rows(const float* __restrict__ X, const float* __restrict__ nw,
                                                     float eps, const W* __restrict__ router, int h, int E, int k,
                                                     int32_t* __restrict__ ids, float* __restrict__ wts, int start,
                                                     int32_t* __restrict__ trace_ids, float* __restrict__ trace_logits,
                                                     int trace_cap, int layer) {
  extern __shared__ float sm[];
  float* red = sm;
  float* logits = sm + 64;
  float* xs = sm + 64 + MAX_EXPERTS;
  const int t = blockIdx.x;
  const float* x = X + (size_t)t * h;
  float ss = 0.f;
  for (int i = threadIdx.x; i < h; i += blockDim.x) {
    const float v = x[i];
    xs[i] = v;
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < 8 ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[32] / (float)h + eps);
  for (int i = threadIdx.x; i < h; i += blockDim.x) xs[i] = xs[i] * inv * nw[i];
  __syncthreads();
  constexpr int V = Chunk<W>::N;
  for (int e = warp; e < E; e += 8) {
    const W* row = router + (size_t)e * h;
    float a = 0.f;
    for (int c = lane; c < h / V; c += 32) {
      float wv[V];
      Chunk<W>::widen(ld_stream16(row + (size_t)c * V), wv);
#pragma unroll
      for (int q = 0; q < V; ++q) a = fmaf(wv[q], xs[c * V + q], a);
    }
    a = warp_sum(a);
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
        for (int q = 0; q < j; ++q) taken |= (sel[q] == e);
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
      ids[(size_t)t * k + j] = sel[j];
      wts[(size_t)t * k + j] = p[j] / tot;
    }
    if (trace_ids) {
      const size_t row = (size_t)layer * trace_cap + ((start + t) % trace_cap);
      for (int j = 0; j < k; ++j) trace_ids[row * k + j] = sel[j];
      for (int e = 0; e < E; ++e) trace_logits[row * E + e] = logits[e];
    }
  }
}

// Stable counting sort of the n*k (row, slot) entries by expert: offsets[E+1],
// rows_sorted[pos] = entry, inv[entry] = pos.  One CTA; entries in row order.
__global__ void __launch_bounds__(256) k_moe_plan(const int32_t* __restrict__ ids, int entries, int E,
                                                  int32_t* __restrict__ offsets, int32_t* __restrict__ rows_sorted,
                                                  int32_t* __restrict__ inv) {
  __shared__ int cnt[MAX_EXPERTS + 1];
  __shared__ int base[MAX_EXPERTS + 1];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < entries; i += blockDim.x) atomicAdd(&cnt[ids[i]], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      base[e] = acc;
      offsets[e] = acc;
      acc += cnt[e];
    }
    offsets[E] = acc;
  }
  __syncthreads();
  // Stable placement: each expert's entries keep row order.  A warp per expert
  // scans the entries with a ballot so the order is the entry order.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = warp; e < E; e += blockDim.x >> 5) {
    int pos = base[e];
    for (int i0 = 0; i0 < entries; i0 += 32) {
      const int i = i0 + lane;
      const bool mine = i < entries && ids[i] == e;
      const unsigned mask = __ballot_sync(0xffffffffu, mine);
      if (mine) {
        const int p = pos + __popc(mask & ((1u << lane) - 1u));
        rows_sorted[p] = i;
        inv[i] = p;
      }
      pos += __popc(mask);
    }
  }
}

// out[p] = A[row of entry p] for every sorted position p (rows of `words`
// 32-bit words; one call per plane).
__global__ void k_gather_rows(const uint32_t* __restrict__ A, const int32_t* __restrict__ rows_sorted, int k,
                              int total, int words, uint32_t* __restrict__ out) {
  const int p = blockIdx.x;
  if (p >= total) return;
  const int t = rows_sorted[p] / k;
  for (int i = threadIdx.x; i < words; i += blockDim.x) out[(size_t)p * words + i] = A[(size_t)t * words + i];
}

// X[t] += sum_{j in selection order} w[t,j] * Y[inv[t*k+j]]
__global__ void k_moe_combine(const float* __restrict__ Y, const int32_t* __restrict__ inv,
                              const float* __restrict__ wts, int k, int h, float* __restrict__ X) {
  const int t = blockIdx.x;
  for (int c = threadIdx.x; c < h; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j) acc = fmaf(wts[(size_t)t * k + j], Y[(size_t)inv[(size_t)t * k + j] * h + c], acc);
    X[(size_t)t * h + c] += acc;
  }
}

// ---------------------------------------------------------------------------
// QK-norm and sandwich norms (rml "The decoder", One forward pass steps 4, 6)

// QK-norm then RoPE of one row's q (blockIdx.y = 0) or k (1): RMSNorm of each
// head with the shared [hd] weight (mode 1) or of the whole row (mode 2), then
// the adjacent-pair rotation of each head with the row's (cos, sin) table.  q
// is read from q_src and written to q_dst (the same rows or another buffer);
// k is rewritten in place at row k_rows[t] (or k_row0 + t) of k_base.
__global__ void __launch_bounds__(128) k_qk_norm_rope(const float* q_src, float* q_dst, float* k_base,
                                                      const int32_t* __restrict__ k_rows, int k_row0, int nq,
                                                      int nkv, int hd, int mode, const float* __restrict__ q_w,
                                                      const float* __restrict__ k_w, float eps,
                                                      const float2* __restrict__ rope) {
  __shared__ float red[5];
  const int t = blockIdx.x, is_k = blockIdx.y;
  const int heads = is_k ? nkv : nq, len = heads * hd;
  const float* src = is_k ? k_base + (size_t)(k_rows ? k_rows[t] : k_row0 + t) * len : q_src + (size_t)t * len;
  float* dst = is_k ? const_cast<float*>(src) : q_dst + (size_t)t * len;
  const float* w = is_k ? k_w : q_w;
  const float2* cs = rope + (size_t)t * (hd / 2);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float inv_row = 0.f;
  if (mode == 2) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < len; i += blockDim.x) ss = fmaf(src[i], src[i], ss);
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) red[4] = red[0] + red[1] + red[2] + red[3];
    __syncthreads();
    inv_row = 1.0f / sqrtf(red[4] / (float)len + eps);
  }
  // A warp per head: lane i takes pairs i, i + 32, ...
  for (int h = warp; h < heads; h += blockDim.x / 32) {
    const float* x = src + (size_t)h * hd;
    float inv = inv_row;
    if (mode == 1) {
      float ss = 0.f;
      for (int d = lane; d < hd; d += 32) ss = fmaf(x[d], x[d], ss);
      inv = 1.0f / sqrtf(warp_sum(ss) / (float)hd + eps);
    }
    const float* wh = mode == 1 ? w : w + (size_t)h * hd;
    float2 out[2];
    int np = 0;
    for (int i = lane; i < hd / 2; i += 32) {
      const float a = x[2 * i] * inv * wh[2 * i], b = x[2 * i + 1] * inv * wh[2 * i + 1];
      const float2 c = cs[i];
      out[np++] = make_float2(a * c.x - b * c.y, a * c.y + b * c.x);
    }
    __syncwarp();   // every lane has read the head before any writes it back
    np = 0;
    for (int i = lane; i < hd / 2; i += 32) {
      dst[(size_t)h * hd + 2 * i] = out[np].x;
      dst[(size_t)h * hd + 2 * i + 1] = out[np].y;
      ++np;
    }
  }
}

// f32 rows -> bf16 (hi, lo) planes (lo plane at plane_stride elements).
__global__ void k_rows_to_planes(const float* __restrict__ src, size_t n, __nv_bfloat16* __restrict__ hi,
                                 size_t plane_stride) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = src[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    hi[plane_stride + i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// X[t] += Z[t] / sqrt(mean(Z[t]^2) + eps) * w, one CTA per row.
__global__ void __launch_bounds__(256) k_rmsnorm_add_rows(float* __restrict__ X, const float* __restrict__ Z,
                                                          const float* __restrict__ w, float eps, int h) {
  __shared__ float red[33];
  const int t = blockIdx.x;
  const float* z = Z + (size_t)t * h;
  float ss = 0.f;
  for (int i = threadIdx.x; i < h; i += blockDim.x) ss = fmaf(z[i], z[i], ss);
  ss = warp_sum(ss);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[32] / (float)h + eps);
  for (int i = threadIdx.x; i < h; i += blockDim.x) X[(size_t)t * h + i] += z[i] * inv * w[i];
}

// ---------------------------------------------------------------------------
// Driver

// An activation row buffer: f32 rows (f32 weights) or bf16 hi/lo planes of
// `rows` x `cols` (bf16 weights, for the tensor-core GEMMs).
struct Act {
  void* base;
  bool split;
  int rows, cols;
  RowOut out() const {
    RowOut o;
    o.hi = base;
    o.lo = split ? reinterpret_cast<__nv_bfloat16*>(base) + (size_t)rows * cols : nullptr;
    o.f32 = split ? 0 : 1;
    return o;
  }
  const void* lo() const { return split ? reinterpret_cast<const __nv_bfloat16*>(base) + (size_t)rows * cols : nullptr; }
};

template <typename TW>
static cudaError_t gemm(const Model& m, cudaStream_t s, const Act& a, const TW* B, int M, int N, int K,
                        const GemmEpi& e, int groups, int max_rows, const QMat& q = QMat{nullptr, nullptr}) {
  cudaError_t err = cudaSuccess;
  timer_begin(m, DEC_K_PF_GEMM, s);
  if (q.codes) {
    // 8-bit weights, expanded a matrix at a time (every group's rows): bf16 models
    // multiply the weight's hi and lo planes separately (each against the
    // activation's hi and lo planes) and sum the two products before the
    // epilogue; f32 models expand to f32 for the SIMT GEMM.
    const size_t rows_b = (size_t)groups * N;
    if (std::is_same<TW, __nv_bfloat16>::value) {
      __nv_bfloat16* hi = reinterpret_cast<__nv_bfloat16*>(m.s.deq);
      __nv_bfloat16* lo = hi + rows_b * K;
      err = launch_weight_dequant_hilo(q, rows_b, K, hi, lo, s);
      GemmEpi ep = e;
      ep.mode = EPI_STORE;
      ep.n_out = N;
      for (int pl = 0; pl < 2 && err == cudaSuccess; ++pl) {
        ep.out_f32 = m.s.q8part + (size_t)pl * M * N;
        err = launch_gemm_tc(a.base, a.lo(), a.rows, pl ? lo : hi, M, N, K, ep, groups, max_rows, m.s.kpart,
                             m.s.kpart_bytes, m.s.st, s);
      }
      if (err == cudaSuccess) err = launch_sum_planes_epi(m.s.q8part, 2, M, N, e, s);
      count_launch(m, 4);
    } else {
      float* wf = reinterpret_cast<float*>(m.s.deq);
      err = launch_weight_dequant_f32(q, rows_b, K, wf, s);
      dim3 grid((max_rows + 63) / 64, (N + 63) / 64, groups);
      k_gemm_simt<float, float><<<grid, 256, 0, s>>>((const float*)a.base, wf, M, N, K, e);
      count_launch(m, 1);
    }
  } else if (std::is_same<TW, __nv_bfloat16>::value) {
    err = launch_gemm_tc(a.base, a.lo(), a.rows, B, M, N, K, e, groups, max_rows, m.s.kpart, m.s.kpart_bytes, m.s.st,
                         s);
  } else {
    dim3 grid((max_rows + 63) / 64, (N + 63) / 64, groups);
    k_gemm_simt<float, TW><<<grid, 256, 0, s>>>((const float*)a.base, B, M, N, K, e);
  }
  timer_end(m, DEC_K_PF_GEMM, s);
  count_launch(m);
  return err;
}

template <typename KV>
static cudaError_t attention(const Model& m, cudaStream_t s, const KV* Ks, const KV* Vs, int base_pos, int start, int n,
                      RowOut O) {
  const dec_config& c = m.cfg;
  dim3 grid((n + 7) / 8, c.n_heads);
  const float* Q = m.s.Q;
  if (std::is_same<KV, float>::value && m.s.at.Kb) {
    // Tensor cores: K and V^T planes of the key columns some query can see,
    // then the flash-attention kernel over 128-row query tiles.
    const int kd = c.n_kv_heads * c.head_dim;
    int c0 = c.sliding_window > 0 ? start - c.sliding_window + 1 : 0;
    c0 = c0 > base_pos ? c0 - base_pos : 0;
    cudaError_t err = launch_kv_split(reinterpret_cast<const float*>(Ks), reinterpret_cast<const float*>(Vs), kd,
                                      c0 & ~63, start + n - base_pos, m.s.at, s);
    timer_begin(m, DEC_K_PF_ATTN, s);
    const cudaError_t e2 = launch_attn_prefill_tc(m.s.at, n, start, base_pos, c.n_heads, c.n_kv_heads, c.head_dim,
                                                  c.sliding_window, O, m.s.st, s);
    timer_end(m, DEC_K_PF_ATTN, s);
    count_launch(m, 2);
    return err != cudaSuccess ? err : e2;
  }
  timer_begin(m, DEC_K_PF_ATTN, s);
  if (c.head_dim == 64)
    k_attn_prefill_simt<KV, 64><<<grid, 256, 0, s>>>(Q, Ks, Vs, base_pos, c.n_heads, c.n_kv_heads, start, n,
                                                    c.sliding_window, O);
  else if (c.head_dim == 128)
    k_attn_prefill_simt<KV, 128><<<grid, 256, 0, s>>>(Q, Ks, Vs, base_pos, c.n_heads, c.n_kv_heads, start, n,
                                                     c.sliding_window, O);
  else
    k_attn_prefill_simt<KV, 16><<<grid, 256, 0, s>>>(Q, Ks, Vs, base_pos, c.n_heads, c.n_kv_heads, start, n,
                                                    c.sliding_window, O);
  timer_end(m, DEC_K_PF_ATTN, s);
  count_launch(m);
  return cudaSuccess;
}

// FFN half of a layer over n rows, residual in m.s.X: RMSNorm -> SwiGLU GEMMs
// (+residual), or router softmax / top-k -> rows grouped by expert -> grouped
// expert GEMMs -> weighted combine (+residual).  start: position of row 0 for
// the router trace; trace = false records nothing.
template <typename TW>
static cudaError_t ffn_rows(const Model& m, cudaStream_t s, const LayerPtrs& L, int l, int n, int start, bool trace) {
  const dec_config& c = m.cfg;
  const Scratch& S = m.s;
  cudaError_t err = cudaSuccess;
  auto chk = [&err](cudaError_t e) {
    if (err == cudaSuccess) err = e;
  };
  const int h = c.hidden, f = c.ffn;
  const bool split = std::is_same<TW, __nv_bfloat16>::value;
  const Act a_h{S.A, split, n, h};
  const Act act{S.ACT, split, n, f};
  if (c.n_experts == 0) {
    k_rmsnorm_rows<<<n, 256, 0, s>>>(S.X, L.ffn_norm, c.rms_eps, h, a_h.out());
    count_launch(m);
    GemmEpi e1{};
    e1.mode = EPI_SWIGLU;
    e1.n_out = 2 * f;
    e1.act = act.base;
    e1.act_bf16 = split;
    e1.act_lo = act.out().lo;
    chk(gemm<TW>(m, s, a_h, (const TW*)L.w_gateup, n, 2 * f, h, e1, 1, n, L.q_gateup));
    GemmEpi e2{};
    // Sandwich norms: the block output goes to Z and is normalised into x.
    e2.mode = c.sandwich_norms ? EPI_STORE : EPI_RESID;
    e2.n_out = h;
    e2.out_f32 = c.sandwich_norms ? S.Z : S.X;
    chk(gemm<TW>(m, s, act, (const TW*)L.w_down, n, h, f, e2, 1, n, L.q_down));
    if (c.sandwich_norms) {
      k_rmsnorm_add_rows<<<n, 256, 0, s>>>(S.X, S.Z, L.post_ffn_norm, c.rms_eps, h);
      count_launch(m);
    }
    return err;
  }
  const int k = c.n_experts_used, E = c.n_experts, entries = n * k;
  const Act a_sort{S.Asort, split, entries, h};
  const Act act_sort{S.ACT, split, entries, f};
  const size_t smr = (64 + MAX_EXPERTS + (size_t)h) * sizeof(float);
  if (smr > 48 * 1024)
    cudaFuncSetAttribute(k_router_rows<TW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smr);
  k_router_rows<TW><<<n, 256, smr, s>>>(S.X, L.ffn_norm, c.rms_eps, (const TW*)L.router, h, E, k, S.pf_ids,
                                        S.pf_wts, start, trace ? m.trace_ids : nullptr,
                                        trace ? m.trace_logits : nullptr, m.trace_cap, l);
  k_moe_plan<<<1, 256, 0, s>>>(S.pf_ids, entries, E, S.pf_offset, S.pf_rows, S.pf_inv);
  k_rmsnorm_rows<<<n, 256, 0, s>>>(S.X, L.ffn_norm, c.rms_eps, h, a_h.out());
  count_launch(m, 3);
  if (split) {
    const int words = h / 2;  // bf16 row of h elements
    k_gather_rows<<<entries, 128, 0, s>>>((const uint32_t*)a_h.base, S.pf_rows, k, entries, words,
                                          (uint32_t*)a_sort.base);
    k_gather_rows<<<entries, 128, 0, s>>>((const uint32_t*)a_h.lo(), S.pf_rows, k, entries, words,
                                          (uint32_t*)a_sort.lo());
    count_launch(m, 2);
  } else {
    k_gather_rows<<<entries, 128, 0, s>>>((const uint32_t*)a_h.base, S.pf_rows, k, entries, h,
                                          (uint32_t*)a_sort.base);
    count_launch(m);
  }
  GemmEpi e1{};
  e1.mode = EPI_SWIGLU;
  e1.n_out = 2 * f;
  e1.act = act_sort.base;
  e1.act_bf16 = split;
  e1.act_lo = act_sort.out().lo;
  e1.group_offset = S.pf_offset;
  chk(gemm<TW>(m, s, a_sort, (const TW*)L.w_gateup, entries, 2 * f, h, e1, E, n, L.q_gateup));
  GemmEpi e2{};
  e2.mode = EPI_STORE;
  e2.n_out = h;
  e2.out_f32 = S.Y;
  e2.group_offset = S.pf_offset;
  chk(gemm<TW>(m, s, act_sort, (const TW*)L.w_down, entries, h, f, e2, E, n, L.q_down));
  if (c.sandwich_norms) {
    cudaMemsetAsync(S.Z, 0, sizeof(float) * (size_t)n * h, s);
    k_moe_combine<<<n, 256, 0, s>>>(S.Y, S.pf_inv, S.pf_wts, k, h, S.Z);
    k_rmsnorm_add_rows<<<n, 256, 0, s>>>(S.X, S.Z, L.post_ffn_norm, c.rms_eps, h);
    count_launch(m, 2);
  } else {
    k_moe_combine<<<n, 256, 0, s>>>(S.Y, S.pf_inv, S.pf_wts, k, h, S.X);
    count_launch(m);
  }
  return err;
}

// Attention output projection over n rows: x += Wo.o, or with sandwich norms
// x += rmsnorm(Wo.o) * w_post.
template <typename TW>
static cudaError_t oproj_rows(const Model& m, cudaStream_t s, const LayerPtrs& L, int n, const Act& a_q) {
  const dec_config& c = m.cfg;
  const Scratch& S = m.s;
  const int h = c.hidden, qd = c.n_heads * c.head_dim;
  GemmEpi e{};
  e.mode = c.sandwich_norms ? EPI_STORE : EPI_RESID;
  e.n_out = h;
  e.out_f32 = c.sandwich_norms ? S.Z : S.X;
  const cudaError_t err = gemm<TW>(m, s, a_q, (const TW*)L.wo, n, h, qd, e, 1, n, L.q_wo);
  if (c.sandwich_norms) {
    k_rmsnorm_add_rows<<<n, 256, 0, s>>>(S.X, S.Z, L.post_attn_norm, c.rms_eps, h);
    count_launch(m);
  }
  return err;
}

// QK-norm + RoPE after a QKV GEMM that wrote unrotated q (f32 rows in S.Q) and
// k (f32 rows at k_base).  planes: the rotated q goes to the bf16 (hi, lo)
// planes of the tensor-core attention (through S.A, free between the GEMM and
// the attention), else back into S.Q.
static void qk_norm_rows(const Model& m, cudaStream_t s, const LayerPtrs& L, int n, float* k_base,
                         const int32_t* k_rows, int k_row0, bool planes, const float2* rope) {
  const dec_config& c = m.cfg;
  const Scratch& S = m.s;
  const int qd = c.n_heads * c.head_dim;
  float* q_dst = planes ? (float*)S.A : S.Q;
  k_qk_norm_rope<<<dim3(n, 2), 128, 0, s>>>(S.Q, q_dst, k_base, k_rows, k_row0, c.n_heads, c.n_kv_heads,
                                            c.head_dim, c.qk_norm, L.q_norm, L.k_norm, c.rms_eps, rope);
  count_launch(m);
  if (planes) {
    k_rows_to_planes<<<device_sm_count(), 256, 0, s>>>((const float*)S.A, (size_t)n * qd, S.at.Qb, (size_t)S.at.qcap * qd);
    count_launch(m);
  }
}

// Sequence seq's ring of one layer (ring sets hold n_seqs rings back to back).
template <typename KV>
static KV* seq_ring(const Model& m, void* layer_ring, int seq) {
  return reinterpret_cast<KV*>(reinterpret_cast<char*>(layer_ring) + (size_t)seq * m.ring_bytes);
}

template <typename TW, typename KV>
static cudaError_t prefill_chunk(const Model& m, cudaStream_t s, int seq, int n, int start, float* logits,
                                 int32_t* d_argmax) {
  const dec_config& c = m.cfg;
  cudaError_t err = cudaSuccess;
  auto chk = [&err](cudaError_t e) {
    if (err == cudaSuccess) err = e;
  };
  const Scratch& S = m.s;
  const int h = c.hidden, hd = c.head_dim, qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  const int half = hd / 2;
  // bf16 weights: activations reach the tensor cores as bf16 (hi, lo) pairs;
  // f32 weights: f32 rows for the SIMT GEMM.  Both keep ~fp32 activations.
  const bool split = std::is_same<TW, __nv_bfloat16>::value;
  k_embed_rows<TW><<<n, 128, 0, s>>>((const TW*)m.tok_embd, S.tokens, h, S.X);
  k_rope_rows<<<(n * half + 255) / 256, 256, 0, s>>>(S.inv_freq, half, start, n, S.rope_tab);
  count_launch(m, 2);
  if (S.rope_tab_local) {
    k_rope_rows<<<(n * half + 255) / 256, 256, 0, s>>>(S.inv_freq_local, half, start, n, S.rope_tab_local);
    count_launch(m);
  }

  // Ring slots equal positions unless this chunk can overwrite history it reads.
  // An int8 cache always takes the linear f32 rows: history read back from the
  // ring, the chunk's rows quantised and read back before attention.
  const bool i8 = c.kv_dtype == DEC_I8;
  const bool paged = m.paging.table != nullptr;
  const bool direct = !i8 && !paged && (c.sliding_window == 0 || start + n <= c.max_seq);
  const int h0 = direct || c.sliding_window == 0 ? 0
                 : (start - c.sliding_window + 1 > 0 ? start - c.sliding_window + 1 : 0);
  const int hist = start - h0;

  const Act a_h{S.A, split, n, h};      // normalised rows
  const Act a_q{S.A, split, n, qd};     // attention output rows
  const bool qkn = c.qk_norm != 0;

  for (int l = 0; l < c.n_layers; ++l) {
    const LayerPtrs& L = m.layers[l];
    KV* kc = seq_ring<KV>(m, L.kc, seq);
    KV* vc = seq_ring<KV>(m, L.vc, seq);
    k_rmsnorm_rows<<<n, 256, 0, s>>>(S.X, L.attn_norm, c.rms_eps, h, a_h.out());
    count_launch(m);
    KV* kdst = direct ? kc : (KV*)S.KVlin_k;
    KV* vdst = direct ? vc : (KV*)S.KVlin_v;
    if (!direct && hist > 0) {
      if (i8) launch_kv_gather_i8(c, L.kc, L.vc, m.paging, seq, h0, hist, (float*)kdst, (float*)vdst, s);
      else k_kv_gather<KV><<<device_sm_count(), 256, 0, s>>>((const KV*)L.kc, (const KV*)L.vc, m.paging, seq, c.max_seq, kd, h0,
                                               hist, kdst, vdst);
      count_launch(m);
    }
    {
      GemmEpi e{};
      e.mode = EPI_QKV;
      e.n_out = qd + 2 * kd;
      e.bias = L.bqkv;
      e.rope = layer_rope_global(c, l) ? S.rope_tab : S.rope_tab_local;
      e.qd = qd;
      e.kd = kd;
      e.hd = hd;
      // Rotated queries: bf16 (hi, lo) planes for the tensor-core attention,
      // else f32 rows.  With QK-norm the epilogue leaves q and k unrotated
      // (f32) and qk_norm_rows normalises and rotates them.
      const bool q_planes = std::is_same<KV, float>::value && S.at.Kb;
      e.q_out = q_planes && !qkn ? (void*)S.at.Qb : (void*)S.Q;
      e.q_bf16 = q_planes && !qkn;
      e.q_lo = q_planes && !qkn ? S.at.Qb + (size_t)S.at.qcap * qd : nullptr;
      const float2* rope = e.rope;
      if (qkn) e.rope = nullptr;
      e.k_dst = kdst;
      e.v_dst = vdst;
      e.kv_bf16 = std::is_same<KV, __nv_bfloat16>::value;
      e.kv_row0 = direct ? start : hist;
      chk(gemm<TW>(m, s, a_h, (const TW*)L.wqkv, n, qd + 2 * kd, h, e, 1, n, L.q_wqkv));
      if (qkn) qk_norm_rows(m, s, L, n, (float*)kdst, nullptr, e.kv_row0, q_planes, rope);
    }
    const int t_first = n > c.max_seq ? n - c.max_seq : 0;
    if (i8) {
      // Codes of the rows whose slot survives the chunk go to the ring; every
      // row's read-back replaces it in the linear rows, so attention sees what
      // the cache holds.
      float* lk = (float*)kdst + (size_t)hist * kd;
      float* lv = (float*)vdst + (size_t)hist * kd;
      launch_kv_quant(c, lk, lv, n, nullptr, m.paging, seq, start, t_first, L.kc, L.vc, lk, lv, s);
      count_launch(m);
    }
    chk(attention<KV>(m, s, kdst, vdst, direct ? 0 : h0, start, n, a_q.out()));
    if (!direct && !i8) {
      k_kv_commit<KV><<<device_sm_count(), 256, 0, s>>>(kdst, vdst, hist, start, t_first, n, c.max_seq, kd, (KV*)L.kc, (KV*)L.vc,
                                          m.paging, seq);
      count_launch(m);
    }
    chk(oproj_rows<TW>(m, s, L, n, a_q));
    chk(ffn_rows<TW>(m, s, L, l, n, start, seq == 0));
  }
  if ((logits || d_argmax) && m.q_head.codes) {
    // 8-bit untied head: the last row through the row GEMM, then its argmax.
    const Act a1{S.A, split, 1, h};
    k_rmsnorm_rows<<<1, 256, 0, s>>>(S.X + (size_t)(n - 1) * h, m.out_norm, c.rms_eps, h, a1.out());
    count_launch(m);
    float* lg = logits ? logits : S.q8part + (S.q8part_bytes / 4 - (size_t)c.vocab);
    GemmEpi eh{};
    eh.mode = EPI_STORE;
    eh.n_out = c.vocab;
    eh.out_f32 = lg;
    chk(gemm<TW>(m, s, a1, (const TW*)m.head, 1, c.vocab, h, eh, 1, 1, m.q_head));
    if (d_argmax) {
      k_argmax_rows<<<1, 1024, 0, s>>>(lg, c.vocab, d_argmax);
      count_launch(m);
    }
  } else if (logits || d_argmax) {
    launch_lmhead(m, s, S.X + (size_t)(n - 1) * h, logits, d_argmax);
  }
  return err;
}

cudaError_t launch_prefill_chunk(const Model& m, cudaStream_t s, int seq, int n, int start, float* logits,
                                 int32_t* d_argmax) {
  // An int8 cache runs on f32 linear rows (KV = float here).
  const bool wb = m.cfg.weight_dtype == DEC_BF16, kb = m.cfg.kv_dtype == DEC_BF16;
  if (wb && kb) return prefill_chunk<__nv_bfloat16, __nv_bfloat16>(m, s, seq, n, start, logits, d_argmax);
  if (wb) return prefill_chunk<__nv_bfloat16, float>(m, s, seq, n, start, logits, d_argmax);
  if (kb) return prefill_chunk<float, __nv_bfloat16>(m, s, seq, n, start, logits, d_argmax);
  return prefill_chunk<float, float>(m, s, seq, n, start, logits, d_argmax);
}

// ---------------------------------------------------------------------------
// Batched decode (Pantheon "Llama Forward Pass", Batched Multi-Sequence
// Decode): B rows, row b one token of sequence b_seq[b] at position b_pos[b].
// The projections, FFN/MoE and LM head are the prefill GEMMs over the B rows
// (each weight matrix read once per step for every row); RoPE uses each row's
// own position; the QKV epilogue writes row b's K/V into row b_rows[b] of the
// layer's ring set (its sequence's ring, slot of its position); attention is
// per row over its own sequence (attn_rows.cu).  No kernel mixes rows except
// through per-row-independent arithmetic, so a row's result does not depend
// on the batch.

template <typename TW, typename KV>
static cudaError_t decode_rows(const Model& m, cudaStream_t s, int B, float* logits, int32_t* d_argmax) {
  const dec_config& c = m.cfg;
  cudaError_t err = cudaSuccess;
  auto chk = [&err](cudaError_t e) {
    if (err == cudaSuccess) err = e;
  };
  const Scratch& S = m.s;
  const int h = c.hidden, hd = c.head_dim, qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  const bool split = std::is_same<TW, __nv_bfloat16>::value;
  k_embed_rows<TW><<<B, 128, 0, s>>>((const TW*)m.tok_embd, S.tokens, h, S.X);
  count_launch(m);
  const Act a_h{S.A, split, B, h};
  const Act a_q{S.A, split, B, qd};
  const int nsplit = attn_rows_splits(c);
  const bool i8 = c.kv_dtype == DEC_I8;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerPtrs& L = m.layers[l];
    k_rmsnorm_rows<<<B, 256, 0, s>>>(S.X, L.attn_norm, c.rms_eps, h, a_h.out());
    count_launch(m);
    {
      GemmEpi e{};
      e.mode = EPI_QKV;
      e.n_out = qd + 2 * kd;
      e.bias = L.bqkv;
      e.rope = layer_rope_global(c, l) ? S.rope_tab : S.rope_tab_local;
      e.qd = qd;
      e.kd = kd;
      e.hd = hd;
      e.q_out = S.Q;
      // int8 cache: f32 K/V rows to the linear scratch, quantised into the
      // rings below; else straight into each row's ring.
      e.k_dst = i8 ? S.KVlin_k : L.kc;
      e.v_dst = i8 ? S.KVlin_v : L.vc;
      e.kv_bf16 = std::is_same<KV, __nv_bfloat16>::value;
      e.kv_rows = i8 ? nullptr : S.b_rows;
      const float2* rope = e.rope;
      if (c.qk_norm) e.rope = nullptr;
      chk(gemm<TW>(m, s, a_h, (const TW*)L.wqkv, B, qd + 2 * kd, h, e, 1, B, L.q_wqkv));
      if (c.qk_norm) qk_norm_rows(m, s, L, B, (float*)e.k_dst, e.kv_rows, 0, false, rope);
    }
    if (i8) {
      launch_kv_quant(c, (const float*)S.KVlin_k, (const float*)S.KVlin_v, B, S.b_rows, m.paging, 0, 0, 0, L.kc,
                      L.vc, nullptr, nullptr, s);
      count_launch(m);
    }
    timer_begin(m, DEC_K_ATTN, s);
    launch_attn_rows(c, S.Q, L.kc, L.vc, m.paging, S.b_seq, S.b_pos, B, nsplit, S.b_part, a_q.out(), s);
    timer_end(m, DEC_K_ATTN, s);
    count_launch(m, 2);
    chk(oproj_rows<TW>(m, s, L, B, a_q));
    chk(ffn_rows<TW>(m, s, L, l, B, 0, false));
  }
  // Final RMSNorm and the LM head over every row.
  k_rmsnorm_rows<<<B, 256, 0, s>>>(S.X, m.out_norm, c.rms_eps, h, a_h.out());
  count_launch(m);
  {
    GemmEpi e{};
    e.mode = EPI_STORE;
    e.n_out = c.vocab;
    e.out_f32 = logits;
    chk(gemm<TW>(m, s, a_h, (const TW*)m.head, B, c.vocab, h, e, 1, B, m.q_head));
  }
  if (d_argmax) {
    k_argmax_rows<<<B, 1024, 0, s>>>(logits, c.vocab, d_argmax);
    count_launch(m);
  }
  return err;
}

cudaError_t launch_decode_rows(const Model& m, cudaStream_t s, int B, float* logits, int32_t* d_argmax) {
  const bool wb = m.cfg.weight_dtype == DEC_BF16, kb = m.cfg.kv_dtype == DEC_BF16;
  if (wb && kb) return decode_rows<__nv_bfloat16, __nv_bfloat16>(m, s, B, logits, d_argmax);
  if (wb) return decode_rows<__nv_bfloat16, float>(m, s, B, logits, d_argmax);
  if (kb) return decode_rows<float, __nv_bfloat16>(m, s, B, logits, d_argmax);
  return decode_rows<float, float>(m, s, B, logits, d_argmax);
}

static int rows_setup_blocks(const Model& m, int B) {
  const int half = m.cfg.head_dim / 2;
  const int n = B * half > B ? B * half : B;
  return (n + 255) / 256;
}

cudaError_t launch_rows_setup(const Model& m, cudaStream_t s, const RowsMeta& meta, const int32_t* d_tokens,
                              int32_t host_token, int B) {
  const Scratch& S = m.s;
  k_rows_setup<<<rows_setup_blocks(m, B), 256, 0, s>>>(meta, B, d_tokens, host_token, m.cfg.vocab, S.inv_freq,
                                                       m.cfg.head_dim / 2, S.tokens, S.b_seq, S.b_pos, S.b_rows,
                                                       S.rope_tab, S.st, S.inv_freq_local, S.rope_tab_local);
  count_launch(m);
  return cudaGetLastError();
}

cudaError_t update_rows_setup_node(cudaGraphExec_t g, cudaGraphNode_t node, const Model& m, const RowsMeta& meta,
                                   const int32_t* d_tokens, int32_t host_token, int B) {
  const Scratch& S = m.s;
  int vocab = m.cfg.vocab, half = m.cfg.head_dim / 2;
  const double* inv = S.inv_freq;
  int32_t *tokens = S.tokens, *bs = S.b_seq, *bp = S.b_pos, *br = S.b_rows;
  float2* tab = S.rope_tab;
  DeviceState* st = S.st;
  const double* invl = S.inv_freq_local;
  float2* tabl = S.rope_tab_local;
  void* args[] = {const_cast<RowsMeta*>(&meta), &B, &d_tokens, &host_token, &vocab, &inv, &half, &tokens, &bs, &bp,
                  &br, &tab, &st, &invl, &tabl};
  cudaKernelNodeParams p = {};
  p.func = reinterpret_cast<void*>(k_rows_setup);
  p.gridDim = dim3(rows_setup_blocks(m, B));
  p.blockDim = dim3(256);
  p.sharedMemBytes = 0;
  p.kernelParams = args;
  p.extra = nullptr;
  return cudaGraphExecKernelNodeSetParams(g, node, &p);
}

}  // namespace dec
