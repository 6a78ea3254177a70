// C ABI of libdec.so: validation, workspace plan, handle state, decode graph.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <string>
#include <vector>

#include "paging.h"
#include "runtime.h"

using namespace dec;

struct dec_handle {
  Model m;
  std::vector<LayerPtrs> layers;
  cudaStream_t stream;
  std::vector<int32_t> lens;   // positions held per sequence (host bookkeeping)
  RowsMeta meta;        // rows of the current batched decode step
  PageAllocator pages;  // paged cache: host copy of the page table and the free pages
  PageSet pset;
  std::string err;
  // decode graph, captured for one (logits, d_argmax) pair
  cudaGraphExec_t graph = nullptr;
  cudaGraph_t graph_src = nullptr;        // kept for the setup node's parameter updates
  cudaGraphNode_t graph_step_node = nullptr;
  float* graph_logits = nullptr;
  int32_t* graph_argmax = nullptr;
  int graph_timed_pairs = 0;
  int64_t graph_kernels = 0;
  int64_t launches = 0;
  Timing timing;
  std::vector<cudaEvent_t> events;
  // batched decode graph, captured for one (batch, tokens, logits, argmax)
  cudaGraphExec_t bgraph = nullptr;
  cudaGraph_t bgraph_src = nullptr;
  cudaGraphNode_t bgraph_setup = nullptr;
  int bgraph_batch = 0;
  const int32_t* bgraph_tokens = nullptr;
  float* bgraph_logits = nullptr;
  int32_t* bgraph_argmax = nullptr;
  int bgraph_timed_pairs = 0;
  int64_t bgraph_kernels = 0;
  bool use_graph = true;
  int fused_mode = 1;   // DEC_FUSED_*
};

static void drop_graph(dec_handle* h) {
  if (h->graph) cudaGraphExecDestroy(h->graph);
  if (h->graph_src) cudaGraphDestroy(h->graph_src);
  h->graph = nullptr;
  h->graph_src = nullptr;
  h->graph_step_node = nullptr;
  if (h->bgraph) cudaGraphExecDestroy(h->bgraph);
  if (h->bgraph_src) cudaGraphDestroy(h->bgraph_src);
  h->bgraph = nullptr;
  h->bgraph_src = nullptr;
  h->bgraph_setup = nullptr;
}

static void timing_start(dec_handle* h) { h->timing.n = 0; }
static void timing_finish(dec_handle* h) { h->timing.n_done = h->timing.n; }

static std::atomic<int> g_sm_count[64];

int dec::device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 1;
  }
  g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

static thread_local std::string g_create_error;

void dec::set_global_error(const char* msg) { g_create_error = msg; }

static dec_status fail(dec_handle* h, dec_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  else g_create_error = buf;
  return st;
}

static size_t dsize(int32_t dt) { return dt == DEC_BF16 ? 2 : 4; }

// Row r of wqkv (and entry r of bqkv) <- the row that holds dim src(d) of the
// same head, for q and k rows: src(2i) = i, src(2i+1) = i + rd/2 for i < rd/2,
// src(d) = d beyond the rotary width rd; v rows are copied unchanged.
__global__ void k_permute_qk_rows(const uint4* __restrict__ w, const float* __restrict__ b, int qd, int kd, int hd,
                                  int rd, int row_chunks, uint4* __restrict__ wdst, float* __restrict__ bdst) {
  const int r = blockIdx.x;
  int src = r;
  if (r < qd + kd) {
    const int d = (r < qd ? r : r - qd) % hd;
    const int sd = d < rd ? ((d & 1) ? (d >> 1) + rd / 2 : (d >> 1)) : d;
    src = r - d + sd;
  }
  for (int i = threadIdx.x; i < row_chunks; i += blockDim.x)
    wdst[(size_t)r * row_chunks + i] = w[(size_t)src * row_chunks + i];
  if (b && bdst && threadIdx.x == 0) bdst[r] = b[src];
}

// dst[i] = src[i - d + src(d)], d = i % hd: a per-head vector (a QK-norm weight)
// in the permuted dim order of the kHalf q/k rows.
__global__ void k_permute_head_vector(const float* __restrict__ src, int n, int hd, int rd, float* __restrict__ dst) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int d = i % hd;
  const int sd = d < rd ? ((d & 1) ? (d >> 1) + rd / 2 : (d >> 1)) : d;
  dst[i] = src[i - d + sd];
}

void dec::launch_permute_head_vector(const dec_config& c, const float* src, int n, float* dst, cudaStream_t s) {
  const int rd = c.rope_dim ? c.rope_dim : c.head_dim;
  k_permute_head_vector<<<(n + 255) / 256, 256, 0, s>>>(src, n, c.head_dim, rd, dst);
}

void dec::launch_permute_qk_rows(const dec_config& c, const void* w, const float* b, void* wdst, float* bdst,
                                 cudaStream_t s) {
  const int qd = c.n_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
  const int rd = c.rope_dim ? c.rope_dim : c.head_dim;
  const int chunks = (int)((size_t)c.hidden * dsize(c.weight_dtype) / 16);
  k_permute_qk_rows<<<qd + 2 * kd, 128, 0, s>>>((const uint4*)w, b, qd, kd, c.head_dim, rd, chunks, (uint4*)wdst,
                                                bdst);
}

static bool validate(const dec_config* c, std::string& why) {
  char b[256];
  auto bad = [&](const char* m) { why = m; return false; };
  if (!c) return bad("config is NULL");
  if (c->n_layers <= 0 || c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
      c->head_dim <= 0 || c->ffn <= 0 || c->vocab <= 0 || c->max_seq <= 0)
    return bad("every size must be positive");
  if (c->n_heads % c->n_kv_heads != 0) return bad("n_heads must be a multiple of n_kv_heads");
  if (c->head_dim % 2 != 0) return bad("head_dim must be even (RoPE rotates pairs)");
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return bad("rms_eps and rope_theta must be positive");
  if (c->weight_dtype != DEC_F32 && c->weight_dtype != DEC_BF16) return bad("weight_dtype must be DEC_F32 or DEC_BF16");
  if (c->kv_dtype != DEC_F32 && c->kv_dtype != DEC_BF16 && c->kv_dtype != DEC_I8)
    return bad("kv_dtype must be DEC_F32, DEC_BF16 or DEC_I8");
  if (c->n_experts < 0 || c->n_experts_used < 0) return bad("expert counts must be >= 0");
  if (c->n_experts == 0 && c->n_experts_used != 0) return bad("n_experts_used must be 0 for a dense FFN");
  if (c->n_experts > 0 && (c->n_experts_used < 1 || c->n_experts_used > c->n_experts))
    return bad("experts used must lie in [1, n_experts]");
  if (c->sliding_window < 0 || c->max_tokens < 0) return bad("sliding_window and max_tokens must be >= 0");
  if (c->sliding_window > 0 && c->max_seq > c->sliding_window)
    return bad("under a sliding window max_seq = min(sliding_window, n_ctx) cannot exceed the window");
  if (c->rope_half != 0 && c->rope_half != 1) return bad("rope_half must be 0 or 1");
  if (c->rope_dim < 0 || c->rope_dim > c->head_dim || c->rope_dim % 2 != 0)
    return bad("rope_dim must be even and in [0, head_dim] (0 = head_dim)");
  if (c->n_seqs < 0 || c->n_seqs > 65536) return bad("n_seqs must be in [0, 65536] (0 = 1)");
  if (c->qk_norm < 0 || c->qk_norm > 2) return bad("qk_norm must be 0 (off), 1 (per head) or 2 (whole row)");
  if (c->qk_norm && c->kv_dtype == DEC_BF16) return bad("qk_norm needs a DEC_F32 or DEC_I8 cache");
  if (c->sandwich_norms != 0 && c->sandwich_norms != 1) return bad("sandwich_norms must be 0 or 1");
  if (!(c->rope_theta_local >= 0.f) || c->rope_global_every < 0)
    return bad("rope_theta_local and rope_global_every must be >= 0");
  if (c->page_size < 0 || (c->page_size > 0 && (c->page_size < 16 || (c->page_size & (c->page_size - 1)))))
    return bad("page_size must be 0 or a power of two >= 16");
  if (c->page_size > 0 && c->n_pages < 1) return bad("a paged cache needs n_pages >= 1");
  if (c->n_pages < 0) return bad("n_pages must be >= 0");
  if (c->weight_quant != 0 && c->weight_quant != 1) return bad("weight_quant must be 0 or 1");
  if (c->weight_quant && (c->hidden % 32 || c->ffn % 32 || (c->n_heads * c->head_dim) % 32))
    return bad("8-bit weights need hidden, ffn and n_heads*head_dim multiples of 32 (one scale per 32 columns)");
  if (c->rope_llama3 && !(c->rope_factor > 0.f && c->rope_low_freq_factor > 0.f &&
                          c->rope_high_freq_factor > c->rope_low_freq_factor && c->rope_orig_ctx > 0))
    return bad("llama3 RoPE scaling needs factor > 0, 0 < low < high, orig_ctx > 0");
  // Limits of this implementation.
  if (c->head_dim != 16 && c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 16, 64 or 128");
  if (c->n_heads / c->n_kv_heads > MAX_GROUP) return bad("at most 16 query heads per kv head");
  if (c->n_kv_heads > MAX_KV_HEADS) return bad("at most 192 kv heads");
  if (c->n_experts > MAX_EXPERTS) return bad("at most 256 experts");
  if (c->n_experts_used > MAX_EXPERTS_USED) return bad("at most 8 experts per token");
  const size_t ws = dsize(c->weight_dtype), ks = c->kv_dtype == DEC_I8 ? 1 : dsize(c->kv_dtype);
  if ((c->hidden * ws) % 16 || (c->ffn * ws) % 16 || ((size_t)c->n_heads * c->head_dim * ws) % 16)
    return bad("hidden, ffn and n_heads*head_dim rows must be whole 16-byte chunks");
  if ((c->head_dim * ks) % 16) return bad("head_dim rows of the KV cache must be whole 16-byte chunks");
  const size_t k_slots = c->n_experts ? (size_t)c->n_experts_used : 1;
  const size_t smem_floats_max = (200 * 1024) / 4 - 64 - MAX_EXPERTS;
  if ((size_t)c->hidden > smem_floats_max || (size_t)c->n_heads * c->head_dim > smem_floats_max ||
      k_slots * c->ffn > smem_floats_max) {
    snprintf(b, sizeof b, "vectors held in shared memory exceed %zu floats", smem_floats_max);
    return bad(b);
  }
  return true;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

WsPlan dec::plan_workspace(const dec_config& c) {
  WsPlan p{};
  const int T = c.max_tokens > 0 ? c.max_tokens : c.max_seq;
  p.max_tokens = T;
  const int hd = c.head_dim, qd = c.n_heads * hd, kd = c.n_kv_heads * hd;
  const int k = c.n_experts ? c.n_experts_used : 1;
  // Decode attention: split s owns slots [s*sps, (s+1)*sps), sps a multiple
  // of 64 keys, at most 64 splits per kv head.
  const int chunks = (c.max_seq + 63) / 64;
  const int per = (chunks + 63) / 64;
  p.attn_sps = 64 * per;
  const int nsplit = (c.max_seq + p.attn_sps - 1) / p.attn_sps;
  p.nsplit = nsplit;
  const size_t ws = dsize(c.weight_dtype), ks = dsize(c.kv_dtype);
  const size_t a_elem = 4;  // prefill activation rows: f32 (or a bf16 hi/lo pair of the same size)
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + (bytes ? bytes : 1), 256); return o; };
  p.st = take(sizeof(DeviceState));
  p.inv_freq = take(sizeof(double) * (hd / 2));
  p.rope_tab = take(sizeof(float2) * (size_t)T * (hd / 2));
  p.x = take(4 * (size_t)c.hidden);
  p.q = take(4 * (size_t)qd);
  p.attn = take(4 * (size_t)qd);
  p.act = take(4 * (size_t)k * c.ffn);
  p.nbuf = take(4 * (size_t)c.hidden);
  p.ids = take(4 * (size_t)MAX_EXPERTS_USED);
  p.wts = take(4 * (size_t)MAX_EXPERTS_USED);
  p.part = take(4 * (size_t)c.n_heads * nsplit * (hd + 2));
  p.amax_val = take(4 * (size_t)LM_GRID_MAX);
  p.amax_idx = take(4 * (size_t)LM_GRID_MAX);
  p.tokens = take(4 * (size_t)T);
  size_t amax = c.hidden;
  if ((size_t)qd > amax) amax = qd;
  if ((size_t)c.ffn > amax) amax = c.ffn;
  p.X = take(4 * (size_t)T * c.hidden);
  p.A = take(a_elem * (size_t)T * amax);
  p.Q = take(4 * (size_t)T * qd);
  p.KVlin_k = take(ks * (size_t)(c.max_seq + T) * kd);
  p.KVlin_v = take(ks * (size_t)(c.max_seq + T) * kd);
  p.pf_ids = take(4 * (size_t)T * k);
  p.pf_wts = take(4 * (size_t)T * k);
  p.pf_count = take(4 * (size_t)(c.n_experts + 1));
  p.pf_offset = take(4 * (size_t)(c.n_experts + 2));
  p.pf_rows = take(4 * (size_t)T * k);
  p.pf_inv = take(4 * (size_t)T * k);
  p.Asort = take(c.n_experts ? a_elem * (size_t)T * k * c.hidden : 0);
  p.Y = take(c.n_experts ? 4 * (size_t)T * k * c.hidden : 0);
  p.ACT = take(a_elem * (size_t)T * k * c.ffn);
  // Tensor-core prefill attention: K planes and V^T planes (bf16 hi, lo) of up
  // to max_seq + T key columns; the Q planes reuse the f32 Q rows.
  const bool at = attn_tc_supported(c);
  p.at_kcap = at ? c.max_seq + T : 0;
  p.at_vt_ld = at ? (int)align_up((size_t)(c.max_seq + T), 8) : 0;
  p.at_Kb = take(2 * 2 * (size_t)p.at_kcap * kd);
  p.at_Vt = take(2 * 2 * (size_t)kd * p.at_vt_ld);
  // kHalf RoPE: per-head row-permuted copies of the q/k rows (and biases) of wqkv.
  const size_t qkv_rows = (size_t)qd + 2 * kd;
  p.wqkv_perm = take(c.rope_half ? (size_t)c.n_layers * qkv_rows * c.hidden * ws : 0);
  p.bqkv_perm = take(c.rope_half && c.qkv_bias ? (size_t)c.n_layers * qkv_rows * 4 : 0);
  p.mk_maps = take(mk_maps_bytes(c));
  // Batched decode: per-row metadata and the attention split partials.
  const int bmax = T < MAX_BATCH ? T : MAX_BATCH;
  p.b_seq = take(4 * (size_t)MAX_BATCH);
  p.b_pos = take(4 * (size_t)MAX_BATCH);
  p.b_rows = take(4 * (size_t)MAX_BATCH);
  p.b_part = take(4 * (size_t)bmax * c.n_heads * AR_MAX_SPLIT * (hd + 2));
  // Split-K partials of the tensor-core GEMMs (bf16 weights): room for 8 splits
  // of one 128-row tile of the widest GEMM, at most 128 MB; a GEMM takes only
  // the splits that fit.
  size_t nmax = (size_t)qd + 2 * kd;
  if ((size_t)c.hidden > nmax) nmax = c.hidden;
  if (2 * (size_t)c.ffn > nmax) nmax = 2 * (size_t)c.ffn;
  if ((size_t)c.vocab > nmax) nmax = c.vocab;
  p.kpart_bytes = c.weight_dtype == DEC_BF16 ? 8 * 128 * nmax * 4 : 0;
  if (p.kpart_bytes > ((size_t)128 << 20)) p.kpart_bytes = (size_t)128 << 20;
  p.kpart = take(p.kpart_bytes);
  p.Z = take(c.sandwich_norms ? 4 * (size_t)T * c.hidden : 0);
  const bool local = c.rope_theta_local > 0.f;
  p.inv_freq_local = take(local ? sizeof(double) * (hd / 2) : 0);
  p.rope_tab_local = take(local ? sizeof(float2) * (size_t)T * (hd / 2) : 0);
  // kHalf with QK-norm: the norm weights follow the permuted q/k dims.
  const size_t qn = c.qk_norm == 2 ? (size_t)qd : (size_t)hd, kn = c.qk_norm == 2 ? (size_t)kd : (size_t)hd;
  p.qk_perm = take(c.qk_norm && c.rope_half ? 4 * (size_t)c.n_layers * (qn + kn) : 0);
  // 8-bit weights: codes + scales of every quantised matrix, one expanded matrix
  // for the row GEMMs, and the two planes' products before their epilogue.
  {
    const size_t E1 = c.n_experts ? (size_t)c.n_experts : 1;
    const size_t mats[5][2] = {{qkv_rows, (size_t)c.hidden}, {(size_t)c.hidden, (size_t)qd},
                               {E1 * 2 * c.ffn, (size_t)c.hidden}, {E1 * c.hidden, (size_t)c.ffn},
                               {c.tied_embedding ? 0 : (size_t)c.vocab, (size_t)c.hidden}};
    size_t q8 = 0, big = 0;
    for (int i = 0; i < 5; ++i) {
      const size_t n = mats[i][0] * mats[i][1];
      q8 += (i < 4 ? (size_t)c.n_layers : 1) * (align_up(n, 256) + align_up(n / 32 * 4, 256));
      if (n > big) big = n;
    }
    const size_t kk = c.n_experts ? (size_t)c.n_experts_used : 1;
    size_t mn = (size_t)T * qkv_rows;
    mn = std::max(mn, (size_t)T * c.hidden);
    mn = std::max(mn, (size_t)T * kk * 2 * c.ffn);
    mn = std::max(mn, (size_t)T * kk * c.hidden);
    mn = std::max(mn, (size_t)bmax * c.vocab);   // the head: one row per batched sequence
    const bool wq = c.weight_quant != 0;
    p.q8_bytes = wq ? q8 : 0;
    p.q8 = take(p.q8_bytes);
    p.deq_bytes = wq ? 4 * big : 0;
    p.deq = take(p.deq_bytes);
    // (+ one logits row for the prefill's untied head when only the argmax is asked for)
    p.q8part_bytes = wq ? 2 * 4 * mn + 4 * (size_t)c.vocab : 0;
    p.q8part = take(p.q8part_bytes);
  }
  // Persistent decode with a fused FFN: every down projection transposed
  // ([expert][ffn][hidden], bf16) and the per-CTA partial sums of its product.
  {
    const bool ft = mk_ffn_fused_layout(c);
    const size_t E1 = c.n_experts ? (size_t)c.n_experts : 1;
    p.wdown_t = take(ft ? (size_t)c.n_layers * E1 * c.ffn * c.hidden * 2 : 0);
    p.fpart = take(ft ? (size_t)MK_MAX_NB * c.hidden * 4 : 0);
  }
  p.kv_cur = take(decode_kv_i8_persistent(c) || decode_qkn_persistent(c) ? 2 * 4 * (size_t)kd : 0);
  // KV rings: [layer][K, V][seq][ring_rows][n_kv*hd], ring_rows = max_seq
  // rounded up to 64 rows so every ring starts 256-byte aligned.
  p.n_seqs = c.n_seqs > 0 ? c.n_seqs : 1;
  p.ring_rows = (int)align_up((size_t)c.max_seq, 64);
  p.ring_bytes = (size_t)kv_row_layout(c).bytes * p.ring_rows;
  p.pages_per_seq = c.page_size > 0 ? (c.max_seq + c.page_size - 1) / c.page_size : 0;
  p.page_table = take(c.page_size > 0 ? 4 * (size_t)p.n_seqs * p.pages_per_seq : 0);
  p.kv = off;
  if (c.page_size > 0) {
    // Arena of pages, each [layer][K, V][page_size rows]; one layer's K base is
    // kv + layer * 2 * page_size rows, pages 2 * n_layers * page_size rows apart.
    p.kv_layer_bytes = (size_t)kv_row_layout(c).bytes * c.page_size;   // one K (or V) block of a page
    off += (size_t)c.n_pages * 2 * c.n_layers * p.kv_layer_bytes;
  } else {
    p.kv_layer_bytes = p.ring_bytes * p.n_seqs;
    off += 2 * p.kv_layer_bytes * c.n_layers;
  }
  p.total = off;
  return p;
}

extern "C" {

dec_status dec_config_validate(const dec_config* cfg, char* msg, size_t msg_len) {
  std::string why;
  const bool ok = validate(cfg, why);
  if (msg && msg_len) {
    snprintf(msg, msg_len, "%s", ok ? "ok" : why.c_str());
  }
  return ok ? DEC_OK : DEC_EINVAL;
}

size_t dec_workspace_bytes(const dec_config* cfg) {
  std::string why;
  if (!validate(cfg, why)) return 0;
  return plan_workspace(*cfg).total;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

dec_status dec_create(const dec_config* cfg, const dec_weights* w, void* workspace,
                      size_t workspace_bytes, void* cuda_stream, dec_handle** out) {
  std::string why;
  if (!out) return fail(nullptr, DEC_EINVAL, "out is NULL");
  *out = nullptr;
  if (!validate(cfg, why)) return fail(nullptr, DEC_EINVAL, "invalid config: %s", why.c_str());
  if (!w || !w->tok_embd || !w->out_norm || !w->layers) return fail(nullptr, DEC_EINVAL, "weights missing");
  if (!cfg->tied_embedding && !w->lm_head) return fail(nullptr, DEC_EINVAL, "untied config needs lm_head");
  if (!workspace) return fail(nullptr, DEC_EINVAL, "workspace is NULL");
  if (((uintptr_t)workspace & 255u) != 0) return fail(nullptr, DEC_EINVAL, "workspace must be 256-byte aligned");
  const WsPlan p = plan_workspace(*cfg);
  if (workspace_bytes < p.total)
    return fail(nullptr, DEC_ENOMEM, "workspace has %zu bytes, needs %zu", workspace_bytes, p.total);
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dec_layer_weights& L = w->layers[l];
    if (!L.attn_norm || !L.wqkv || !L.wo || !L.ffn_norm || !L.w_gateup || !L.w_down)
      return fail(nullptr, DEC_EINVAL, "layer %d: a required weight is NULL", l);
    if (cfg->qkv_bias && !L.bqkv) return fail(nullptr, DEC_EINVAL, "layer %d: qkv_bias set but bqkv is NULL", l);
    if (cfg->n_experts > 0 && !L.router) return fail(nullptr, DEC_EINVAL, "layer %d: MoE layer needs router", l);
    if (cfg->qk_norm && (!L.q_norm || !L.k_norm))
      return fail(nullptr, DEC_EINVAL, "layer %d: qk_norm set but q_norm / k_norm is NULL", l);
    if (cfg->sandwich_norms && (!L.post_attn_norm || !L.post_ffn_norm))
      return fail(nullptr, DEC_EINVAL, "layer %d: sandwich_norms set but a post norm is NULL", l);
    if (!aligned16(L.wqkv) || !aligned16(L.wo) || !aligned16(L.w_gateup) || !aligned16(L.w_down) ||
        (L.router && !aligned16(L.router)))
      return fail(nullptr, DEC_EINVAL, "layer %d: weight matrices must be 16-byte aligned", l);
  }
  if (!aligned16(w->tok_embd) || (w->lm_head && !aligned16(w->lm_head)))
    return fail(nullptr, DEC_EINVAL, "embedding / head must be 16-byte aligned");

  dec_handle* h = new (std::nothrow) dec_handle();
  if (!h) return fail(nullptr, DEC_EINVAL, "out of host memory");
  h->stream = (cudaStream_t)cuda_stream;
  h->lens.assign(p.n_seqs, 0);
  if (cfg->page_size > 0) {
    h->pages.init(p.n_seqs, cfg->max_seq, cfg->page_size, cfg->n_pages, cfg->sliding_window > 0);
  }
  Model& m = h->m;
  m.cfg = *cfg;
  if (m.cfg.max_tokens == 0) m.cfg.max_tokens = p.max_tokens;
  m.ws = workspace;
  m.ws_bytes = workspace_bytes;
  m.nsplit = p.nsplit;
  m.attn_sps = p.attn_sps;
  m.n_seqs = p.n_seqs;
  m.ring_rows = p.ring_rows;
  m.ring_bytes = p.ring_bytes;
  m.paging = KvPaging{};
  m.paging.ring_rows = p.ring_rows;
  if (cfg->page_size > 0) {
    m.paging.table = (const int32_t*)((char*)workspace + p.page_table);
    m.paging.pages_per_seq = p.pages_per_seq;
    m.paging.page = cfg->page_size;
    m.paging.stride_rows = 2LL * cfg->n_layers * cfg->page_size;
  }
  // LM head: two CTAs per SM, each warp walking its row pairs with the next
  // pair's loads in flight.
  int lg = (cfg->vocab / 2 + 7) / 8;
  const int sms = device_sm_count();
  if (lg > 2 * sms) lg = 2 * sms;
  m.lm_grid = lg < 1 ? 1 : (lg > LM_GRID_MAX ? LM_GRID_MAX : lg);
  m.tok_embd = w->tok_embd;
  m.out_norm = (const float*)w->out_norm;
  m.head = cfg->tied_embedding ? w->tok_embd : w->lm_head;
  m.trace_ids = nullptr;
  m.trace_logits = nullptr;
  m.trace_cap = 1;
  m.mk_stamps = nullptr;
  m.timing = &h->timing;
  m.launches = &h->launches;
  char* base = (char*)workspace;
  Scratch& S = m.s;
  S.st = (DeviceState*)(base + p.st);
  S.inv_freq = (double*)(base + p.inv_freq);
  S.rope_tab = (float2*)(base + p.rope_tab);
  S.x = (float*)(base + p.x);
  S.q = (float*)(base + p.q);
  S.attn = (float*)(base + p.attn);
  S.act = (float*)(base + p.act);
  S.nbuf = (float*)(base + p.nbuf);
  S.ids = (int32_t*)(base + p.ids);
  S.wts = (float*)(base + p.wts);
  S.part = (float*)(base + p.part);
  S.amax_val = (float*)(base + p.amax_val);
  S.amax_idx = (int32_t*)(base + p.amax_idx);
  S.tokens = (int32_t*)(base + p.tokens);
  S.X = (float*)(base + p.X);
  S.A = base + p.A;
  S.Q = (float*)(base + p.Q);
  S.KVlin_k = base + p.KVlin_k;
  S.KVlin_v = base + p.KVlin_v;
  S.pf_ids = (int32_t*)(base + p.pf_ids);
  S.pf_wts = (float*)(base + p.pf_wts);
  S.pf_count = (int32_t*)(base + p.pf_count);
  S.pf_offset = (int32_t*)(base + p.pf_offset);
  S.pf_rows = (int32_t*)(base + p.pf_rows);
  S.pf_inv = (int32_t*)(base + p.pf_inv);
  S.Asort = base + p.Asort;
  S.Y = (float*)(base + p.Y);
  S.ACT = base + p.ACT;
  S.at.Qb = (__nv_bfloat16*)S.Q;
  S.at.qcap = p.max_tokens;
  S.at.Kb = p.at_kcap ? (__nv_bfloat16*)(base + p.at_Kb) : nullptr;
  S.at.kcap = p.at_kcap;
  S.at.Vt = p.at_kcap ? (__nv_bfloat16*)(base + p.at_Vt) : nullptr;
  S.at.vt_ld = p.at_vt_ld;
  S.b_seq = (int32_t*)(base + p.b_seq);
  S.b_pos = (int32_t*)(base + p.b_pos);
  S.b_rows = (int32_t*)(base + p.b_rows);
  S.b_part = (float*)(base + p.b_part);
  S.kpart = p.kpart_bytes ? (float*)(base + p.kpart) : nullptr;
  S.kpart_bytes = p.kpart_bytes;
  S.Z = cfg->sandwich_norms ? (float*)(base + p.Z) : nullptr;
  S.inv_freq_local = cfg->rope_theta_local > 0.f ? (double*)(base + p.inv_freq_local) : nullptr;
  S.rope_tab_local = cfg->rope_theta_local > 0.f ? (float2*)(base + p.rope_tab_local) : nullptr;
  h->layers.resize(cfg->n_layers);
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dec_layer_weights& L = w->layers[l];
    LayerPtrs& d = h->layers[l];
    d.attn_norm = (const float*)L.attn_norm;
    d.wqkv = L.wqkv;
    d.bqkv = cfg->qkv_bias ? (const float*)L.bqkv : nullptr;
    d.wo = L.wo;
    d.ffn_norm = (const float*)L.ffn_norm;
    d.w_gateup = L.w_gateup;
    d.w_down = L.w_down;
    d.router = cfg->n_experts > 0 ? L.router : nullptr;
    d.kc = base + p.kv + (size_t)(2 * l) * p.kv_layer_bytes;       // paged: page 0's blocks of layer l
    d.vc = base + p.kv + (size_t)(2 * l + 1) * p.kv_layer_bytes;
    d.q_norm = cfg->qk_norm ? (const float*)L.q_norm : nullptr;
    d.k_norm = cfg->qk_norm ? (const float*)L.k_norm : nullptr;
    d.post_attn_norm = cfg->sandwich_norms ? (const float*)L.post_attn_norm : nullptr;
    d.post_ffn_norm = cfg->sandwich_norms ? (const float*)L.post_ffn_norm : nullptr;
    d.q_wqkv = d.q_wo = d.q_gateup = d.q_down = QMat{nullptr, nullptr};
    d.w_down_t = nullptr;
  }
  S.fpart = nullptr;
  S.kv_cur = decode_kv_i8_persistent(*cfg) || decode_qkn_persistent(*cfg) ? (float*)(base + p.kv_cur) : nullptr;
  if (mk_ffn_fused_layout(*cfg)) {
    // The persistent step's fused FFN reads each layer's down projection transposed.
    const size_t E1 = cfg->n_experts ? (size_t)cfg->n_experts : 1;
    const size_t lbytes = E1 * cfg->ffn * cfg->hidden * 2;
    cudaError_t te = cudaSuccess;
    for (int l = 0; l < cfg->n_layers && te == cudaSuccess; ++l) {
      LayerPtrs& d = h->layers[l];
      char* dst = base + p.wdown_t + (size_t)l * lbytes;
      te = launch_transpose_bf16(d.w_down, cfg->hidden, cfg->ffn, (int)E1, dst, h->stream);
      d.w_down_t = dst;
    }
    if (te != cudaSuccess) {
      delete h;
      return fail(nullptr, DEC_ECUDA, "down-projection transpose: %s", cudaGetErrorString(te));
    }
    S.fpart = (float*)(base + p.fpart);
  }
  if (cfg->rope_half) {
    // kHalf pairs (i, i + d/2) become adjacent pairs (2i, 2i+1) on q/k rows
    // permuted per head: every kernel rotates adjacent pairs, and attention,
    // which only forms q . k, is unchanged by the common permutation.
    const size_t qkv_rows = (size_t)cfg->n_heads * cfg->head_dim + 2 * (size_t)cfg->n_kv_heads * cfg->head_dim;
    const size_t row_bytes = (size_t)cfg->hidden * dsize(cfg->weight_dtype);
    for (int l = 0; l < cfg->n_layers; ++l) {
      LayerPtrs& d = h->layers[l];
      char* wdst = base + p.wqkv_perm + (size_t)l * qkv_rows * row_bytes;
      float* bdst = d.bqkv ? (float*)(base + p.bqkv_perm) + (size_t)l * qkv_rows : nullptr;
      launch_permute_qk_rows(*cfg, d.wqkv, d.bqkv, wdst, bdst, h->stream);
      d.wqkv = wdst;
      d.bqkv = bdst;
      if (cfg->qk_norm) {
        const size_t qn = cfg->qk_norm == 2 ? (size_t)cfg->n_heads * cfg->head_dim : (size_t)cfg->head_dim;
        const size_t kn = cfg->qk_norm == 2 ? (size_t)cfg->n_kv_heads * cfg->head_dim : (size_t)cfg->head_dim;
        float* qdst = (float*)(base + p.qk_perm) + (size_t)l * (qn + kn);
        launch_permute_head_vector(*cfg, d.q_norm, (int)qn, qdst, h->stream);
        launch_permute_head_vector(*cfg, d.k_norm, (int)kn, qdst + qn, h->stream);
        d.q_norm = qdst;
        d.k_norm = qdst + qn;
      }
    }
  }
  m.layers = h->layers.data();
  m.wq8 = cfg->weight_quant != 0;
  m.q_head = QMat{nullptr, nullptr};
  S.deq = nullptr;
  S.deq_bytes = 0;
  S.q8part = nullptr;
  S.q8part_bytes = 0;
  if (m.wq8) {
    // Quantise every projection (after any kHalf row permutation) into the workspace.
    char* q = base + p.q8;
    const bool wb = cfg->weight_dtype == DEC_BF16;
    cudaError_t qe = cudaSuccess;
    auto carve = [&](size_t rows, size_t cols, const void* src) {
      QMat r;
      r.codes = (const int8_t*)q;
      q += align_up(rows * cols, 256);
      r.scales = (const float*)q;
      q += align_up(rows * cols / 32 * 4, 256);
      const cudaError_t e = launch_weight_quant(src, wb, rows, (int)cols, (int8_t*)r.codes, (float*)r.scales,
                                                h->stream);
      if (qe == cudaSuccess) qe = e;
      return r;
    };
    const size_t hd_ = cfg->hidden, qd_ = (size_t)cfg->n_heads * cfg->head_dim;
    const size_t kd_ = (size_t)cfg->n_kv_heads * cfg->head_dim, f_ = cfg->ffn;
    const size_t E1 = cfg->n_experts ? (size_t)cfg->n_experts : 1;
    for (int l = 0; l < cfg->n_layers; ++l) {
      LayerPtrs& d = h->layers[l];
      d.q_wqkv = carve(qd_ + 2 * kd_, hd_, d.wqkv);
      d.q_wo = carve(hd_, qd_, d.wo);
      d.q_gateup = carve(E1 * 2 * f_, hd_, d.w_gateup);
      d.q_down = carve(E1 * hd_, f_, d.w_down);
    }
    if (!cfg->tied_embedding) m.q_head = carve((size_t)cfg->vocab, hd_, m.head);
    if (qe != cudaSuccess) {
      delete h;
      return fail(nullptr, DEC_ECUDA, "weight quantisation: %s", cudaGetErrorString(qe));
    }
    S.deq = base + p.deq;
    S.deq_bytes = p.deq_bytes;
    S.q8part = p.q8part_bytes ? (float*)(base + p.q8part) : nullptr;
    S.q8part_bytes = p.q8part_bytes;
  }
  {
    m.mk_maps = mk_maps_bytes(*cfg) ? (void*)(base + p.mk_maps) : nullptr;
    int dev = 0, sms = 0;
    cudaError_t e2 = cudaGetDevice(&dev);
    if (e2 == cudaSuccess) e2 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e2 != cudaSuccess) {
      delete h;
      return fail(nullptr, DEC_ECUDA, "CUDA error at create: %s", cudaGetErrorString(e2));
    }
    mk_prepare(m, sms);
    cudaGetLastError();  // a configuration the persistent kernel cannot take is not an error
    // Small models are bound by the latency of ~150 dependent phases per token,
    // where the per-layer kernels overlapped by programmatic dependent launch
    // are faster (SmolLM2-135M, 0.27 GB per token); from about half a GB per
    // token the persistent kernel's weight rings win (Qwen2.5-0.5B, ~1 GB:
    // 1030 vs 715 tok/s decode on GB300).
    size_t wbytes = (size_t)cfg->vocab * cfg->hidden * (cfg->tied_embedding ? 1 : 2);
    const size_t qd = (size_t)cfg->n_heads * cfg->head_dim, kd = (size_t)cfg->n_kv_heads * cfg->head_dim;
    const size_t kslots = cfg->n_experts ? cfg->n_experts_used : 1;
    wbytes += (size_t)cfg->n_layers * ((qd + 2 * kd) * cfg->hidden + cfg->hidden * qd + 3 * kslots * cfg->ffn * cfg->hidden);
    wbytes *= cfg->weight_dtype == DEC_BF16 ? 2 : 4;
    h->fused_mode = wbytes >= (size_t)512 << 20 ? DEC_FUSED_GRID : DEC_FUSED_OFF;
    // 8-bit weights: the per-layer decode kernels read bf16/f32 rows only, so the
    // persistent step is the fast path whenever it can run.
    if (m.wq8) h->fused_mode = DEC_FUSED_GRID;
  }

  // RoPE frequencies inv_i = theta^(-2i/hd), llama3-scaled when enabled
  // (rml "The decoder", Rotary embeddings), computed once in double.
  // Pairs beyond the rotary width keep frequency 0: a rotation by angle 0 (cos 1,
  // sin 0) leaves them exactly as they are (partial rotary).
  const int rdim = cfg->rope_dim ? cfg->rope_dim : cfg->head_dim;
  std::vector<double> inv(cfg->head_dim / 2, 0.0);
  for (int i = 0; i < rdim / 2; ++i) {
    double f = pow((double)cfg->rope_theta, -2.0 * i / rdim);
    if (cfg->rope_llama3) {
      const double wl = 2.0 * M_PI / f, orig = cfg->rope_orig_ctx;
      const double lo = cfg->rope_low_freq_factor, hi = cfg->rope_high_freq_factor, fac = cfg->rope_factor;
      if (wl < orig / hi) {
      } else if (wl > orig / lo) {
        f = f / fac;
      } else {
        const double sm = (orig / wl - lo) / (hi - lo);
        f = (1.0 - sm) * f / fac + sm * f;
      }
    }
    inv[i] = f;
  }
  cudaError_t e = cudaMemcpy(S.inv_freq, inv.data(), inv.size() * sizeof(double), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && S.inv_freq_local) {
    // Local layers: the same rotary width, their own base, no llama3 scaling.
    std::vector<double> invl(cfg->head_dim / 2, 0.0);
    for (int i = 0; i < rdim / 2; ++i) invl[i] = pow((double)cfg->rope_theta_local, -2.0 * i / rdim);
    e = cudaMemcpy(S.inv_freq_local, invl.data(), invl.size() * sizeof(double), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMemset(S.st, 0, sizeof(DeviceState));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete h;
    return fail(nullptr, DEC_ECUDA, "CUDA error at create: %s", cudaGetErrorString(e));
  }
  *out = h;
  return DEC_OK;
}

static dec_status cuda_check(dec_handle* h, const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  return DEC_OK;
}

// Position rules shared by prefill and decode (rml "The decoder", One forward
// pass, step 1; Pantheon Sliding Window).
static dec_status check_positions(dec_handle* h, int32_t seq, int32_t n, int32_t start_pos) {
  const dec_config& c = h->m.cfg;
  if (n <= 0) return fail(h, DEC_EINVAL, "empty input");
  const int32_t len = h->lens[seq];
  if (start_pos < 0 || start_pos > len)
    return fail(h, DEC_EINVAL, "start_pos %d outside [0, %d]", start_pos, len);
  if (c.sliding_window > 0 && c.max_seq == c.sliding_window) {
    if (len > c.max_seq && start_pos < len)
      return fail(h, DEC_EINVAL, "cannot rewind to %d: the ring has overwritten positions below %d",
                  start_pos, len - c.max_seq);
  } else if ((int64_t)start_pos + n > c.max_seq) {
    return fail(h, DEC_ERANGE, "cache full: start_pos %d + n %d > max_seq %d", start_pos, n, c.max_seq);
  }
  return DEC_OK;
}

// Paged cache: the pages that writing positions [p0, p0 + n) of each sequence
// needs and does not hold yet, all or none (DEC_ENOMEM leaves everything as it
// was), then written into the device table on the stream.
static dec_status reserve_pages(dec_handle* h, const int32_t* seqs, const int32_t* p0s, int count, int32_t n) {
  const dec_config& c = h->m.cfg;
  if (c.page_size <= 0) return DEC_OK;
  std::vector<std::pair<int, int>> taken;   // (table index, page)
  if (!h->pages.reserve(seqs, p0s, count, n, taken))
    return fail(h, DEC_ENOMEM, "paged cache: all %d pages are in use", c.n_pages);
  PageSet& ps = h->pset;
  for (size_t i = 0; i < taken.size(); i += 256) {
    ps.n = (int)std::min<size_t>(256, taken.size() - i);
    for (int j = 0; j < ps.n; ++j) {
      ps.idx[j] = taken[i + j].first;
      ps.val[j] = taken[i + j].second;
    }
    launch_set_pages(const_cast<int32_t*>(h->m.paging.table), ps, h->stream);
  }
  return cuda_check(h, "page table update");
}

static void release_pages(dec_handle* h, int32_t seq) {
  if (h->m.cfg.page_size > 0) h->pages.release(seq);
}

dec_status dec_prefill_seq(dec_handle* h, int32_t seq, const int32_t* tokens, int32_t n, int32_t start_pos,
                           float* logits, int32_t* d_argmax) {
  if (!h) return DEC_EINVAL;
  if (seq < 0 || seq >= h->m.n_seqs) return fail(h, DEC_EINVAL, "sequence %d outside [0, %d)", seq, h->m.n_seqs);
  if (!tokens && n > 0) return fail(h, DEC_EINVAL, "tokens is NULL");
  dec_status st = check_positions(h, seq, n, start_pos);
  if (st != DEC_OK) return st;
  for (int32_t i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->m.cfg.vocab)
      return fail(h, DEC_EINVAL, "token %d at index %d outside [0, %d)", tokens[i], i, h->m.cfg.vocab);
  st = reserve_pages(h, &seq, &start_pos, 1, n);
  if (st != DEC_OK) return st;
  const int T = h->m.cfg.max_tokens;
  timing_start(h);
  for (int32_t done = 0; done < n; done += T) {
    const int chunk = (n - done) < T ? (n - done) : T;
    cudaError_t e = cudaMemcpyAsync(h->m.s.tokens, tokens + done, sizeof(int32_t) * chunk,
                                    cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return fail(h, DEC_ECUDA, "token copy: %s", cudaGetErrorString(e));
    const bool last = done + chunk == n;
    e = launch_prefill_chunk(h->m, h->stream, seq, chunk, start_pos + done, last ? logits : nullptr,
                             last ? d_argmax : nullptr);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(h, DEC_ECUDA, "prefill launch setup: %s", cudaGetErrorString(e));
    }
    st = cuda_check(h, "prefill launch");
    if (st != DEC_OK) return st;
  }
  timing_finish(h);
  h->lens[seq] = start_pos + n;
  return DEC_OK;
}

dec_status dec_prefill(dec_handle* h, const int32_t* tokens, int32_t n, int32_t start_pos, float* logits,
                       int32_t* d_argmax) {
  return dec_prefill_seq(h, 0, tokens, n, start_pos, logits, d_argmax);
}

// Points the captured step-setup node at this step's token and position.
static cudaError_t set_step_node(dec_handle* h, const int32_t* d_token, int32_t token, int32_t pos) {
  DeviceState* st = h->m.s.st;
  int32_t vocab = h->m.cfg.vocab;
  const double* inv = h->m.s.inv_freq;
  int half = h->m.cfg.head_dim / 2;
  float2* tab = h->m.s.rope_tab;
  void* args[] = {&st, &d_token, &token, &pos, &vocab, &inv, &half, &tab};
  cudaKernelNodeParams p = {};
  p.func = const_cast<void*>(set_step_kernel());
  p.gridDim = dim3(1);
  p.blockDim = dim3(128);
  p.sharedMemBytes = 0;
  p.kernelParams = args;
  p.extra = nullptr;
  return cudaGraphExecKernelNodeSetParams(h->graph, h->graph_step_node, &p);
}

// One decode step.  On a non-default stream the whole step (setup, every layer,
// head) is one CUDA graph, captured once per (logits, argmax) pair; per step
// only the setup node's token/position change.
static dec_status run_rows(dec_handle* h, int32_t batch, const int32_t* seqs, const int32_t* positions,
                           const int32_t* d_tokens, int32_t host_token, float* logits, int32_t* d_argmax);

static dec_status run_decode_step(dec_handle* h, const int32_t* d_token, int32_t token, int32_t pos,
                                  float* logits, int32_t* d_argmax) {
  const bool cluster = h->fused_mode == DEC_FUSED_CLUSTER && h->m.mk_cluster > 0;
  const bool fused = h->m.mk_ok && (cluster || h->fused_mode == DEC_FUSED_GRID);
  if (decode_needs_rows(h->m.cfg) ||
      ((h->m.wq8 || h->m.cfg.kv_dtype == DEC_I8 || h->m.cfg.qk_norm != 0 || h->m.cfg.rope_theta_local > 0.f) &&
       !fused)) {
    // Sandwich norms, the row-long QK-norm and the int8 caches the persistent step
    // does not read run on the row kernels: one row, sequence 0; so do 8-bit weights,
    // int8 caches, QK-norm and the per-layer RoPE base when the persistent step is
    // not taken (the per-layer decode kernels implement none of them).
    const int32_t seq0 = 0;
    return run_rows(h, 1, &seq0, &pos, d_token, token, logits, d_argmax);
  }
  if (fused) {
    timing_start(h);
    launch_decode_mk(h->m, h->stream, d_token, token, pos, logits, d_argmax, cluster);
    timing_finish(h);
    return cuda_check(h, "decode launch");
  }
  if (h->stream == nullptr || !h->use_graph) {
    timing_start(h);
    launch_decode_body(h->m, h->stream, d_token, token, pos, logits, d_argmax);
    timing_finish(h);
    return cuda_check(h, "decode launch");
  }
  if (!h->graph || h->graph_logits != logits || h->graph_argmax != d_argmax) {
    drop_graph(h);
    cudaError_t e = cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) return fail(h, DEC_ECUDA, "begin capture: %s", cudaGetErrorString(e));
    timing_start(h);
    const int64_t before = h->launches;
    launch_decode_body(h->m, h->stream, d_token, token, pos, logits, d_argmax);
    h->graph_kernels = h->launches - before;
    h->launches = before;
    h->graph_timed_pairs = h->timing.n;
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(h->stream, &g);
    if (e != cudaSuccess) return fail(h, DEC_ECUDA, "end capture: %s", cudaGetErrorString(e));
    h->graph_src = g;
    cudaGraphNode_t roots[4];
    size_t nroots = 4;
    e = cudaGraphGetRootNodes(g, roots, &nroots);
    if (e != cudaSuccess || nroots != 1) {
      drop_graph(h);
      return fail(h, DEC_ECUDA, "decode graph: expected one root node (%s)", cudaGetErrorString(e));
    }
    h->graph_step_node = roots[0];
    e = cudaGraphInstantiate(&h->graph, g, 0);
    if (e != cudaSuccess) {
      drop_graph(h);
      return fail(h, DEC_ECUDA, "graph instantiate: %s", cudaGetErrorString(e));
    }
    h->graph_logits = logits;
    h->graph_argmax = d_argmax;
  }
  cudaError_t e = set_step_node(h, d_token, token, pos);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "graph step update: %s", cudaGetErrorString(e));
  e = cudaGraphLaunch(h->graph, h->stream);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "graph launch: %s", cudaGetErrorString(e));
  h->timing.n = h->graph_timed_pairs;
  h->launches += h->graph_kernels;
  timing_finish(h);
  return DEC_OK;
}

dec_status dec_decode(dec_handle* h, int32_t token, int32_t pos, float* logits) {
  if (!h) return DEC_EINVAL;
  dec_status st = check_positions(h, 0, 1, pos);
  if (st != DEC_OK) return st;
  if (token < 0 || token >= h->m.cfg.vocab)
    return fail(h, DEC_EINVAL, "token %d outside [0, %d)", token, h->m.cfg.vocab);
  st = run_decode_step(h, nullptr, token, pos, logits, nullptr);
  if (st != DEC_OK) return st;
  h->lens[0] = pos + 1;
  return DEC_OK;
}

dec_status dec_decode_dev(dec_handle* h, const int32_t* d_token, int32_t pos, float* logits,
                          int32_t* d_argmax) {
  if (!h) return DEC_EINVAL;
  if (!d_token) return fail(h, DEC_EINVAL, "d_token is NULL");
  dec_status st = check_positions(h, 0, 1, pos);
  if (st != DEC_OK) return st;
  st = run_decode_step(h, d_token, 0, pos, logits, d_argmax);
  if (st != DEC_OK) return st;
  h->lens[0] = pos + 1;
  return DEC_OK;
}

dec_status dec_kv_reset(dec_handle* h) { return dec_kv_reset_seq(h, 0); }

dec_status dec_kv_reset_seq(dec_handle* h, int32_t seq) {
  if (!h) return DEC_EINVAL;
  if (seq < 0 || seq >= h->m.n_seqs) return fail(h, DEC_EINVAL, "sequence %d outside [0, %d)", seq, h->m.n_seqs);
  h->lens[seq] = 0;
  release_pages(h, seq);
  return DEC_OK;
}

int32_t dec_pages_free(const dec_handle* h) {
  if (!h || h->m.cfg.page_size <= 0) return -1;
  return (int32_t)h->pages.free_count();
}

dec_status dec_kv_slot(const dec_handle* h, int32_t layer, int32_t seq, int32_t slot, void** k, void** v) {
  if (!h || !k || !v || layer < 0 || layer >= h->m.cfg.n_layers || seq < 0 || seq >= h->m.n_seqs || slot < 0 ||
      slot >= h->m.cfg.max_seq)
    return DEC_EINVAL;
  const KvPaging& pg = h->m.paging;
  long long row;
  if (h->m.cfg.page_size > 0) {
    const int32_t page = h->pages.page_of(seq, slot);
    if (page < 0) return DEC_EINVAL;
    row = page * pg.stride_rows + slot % pg.page;
  } else {
    row = (long long)seq * pg.ring_rows + slot;
  }
  const size_t rb = (size_t)kv_row_layout(h->m.cfg).bytes;
  *k = (char*)h->m.layers[layer].kc + (size_t)row * rb;
  *v = (char*)h->m.layers[layer].vc + (size_t)row * rb;
  return DEC_OK;
}

int32_t dec_length(const dec_handle* h) { return dec_length_seq(h, 0); }

int32_t dec_length_seq(const dec_handle* h, int32_t seq) {
  if (!h || seq < 0 || seq >= h->m.n_seqs) return -1;
  return h->lens[seq];
}

// Enqueues one step of the row kernels for rows already validated: one CUDA
// graph per (batch, token source, logits, argmax) on a non-default stream.
static dec_status run_rows(dec_handle* h, int32_t batch, const int32_t* seqs, const int32_t* positions,
                           const int32_t* d_tokens, int32_t host_token, float* logits, int32_t* d_argmax) {
  const dec_config& c = h->m.cfg;
  RowsMeta& meta = h->meta;
  const dec_status ps = reserve_pages(h, seqs, positions, batch, 1);
  if (ps != DEC_OK) return ps;
  for (int32_t i = 0; i < batch; ++i) {
    const int32_t p = positions[i];
    const int32_t slot = c.sliding_window > 0 ? p % c.max_seq : p;
    meta.seq[i] = seqs[i];
    meta.pos[i] = p;
    if (c.page_size > 0) {
      const KvPaging& pg = h->m.paging;
      meta.rows[i] = (int32_t)(h->pages.page_of(seqs[i], slot) * pg.stride_rows + slot % pg.page);
    } else {
      meta.rows[i] = seqs[i] * h->m.ring_rows + slot;
    }
  }
  if (h->stream == nullptr || !h->use_graph) {
    timing_start(h);
    cudaError_t e = launch_rows_setup(h->m, h->stream, meta, d_tokens, host_token, batch);
    if (e == cudaSuccess) e = launch_decode_rows(h->m, h->stream, batch, logits, d_argmax);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(h, DEC_ECUDA, "batched decode launch: %s", cudaGetErrorString(e));
    }
    const dec_status st = cuda_check(h, "batched decode launch");
    if (st != DEC_OK) return st;
    timing_finish(h);
    return DEC_OK;
  }
  if (!h->bgraph || h->bgraph_batch != batch || h->bgraph_tokens != d_tokens || h->bgraph_logits != logits ||
      h->bgraph_argmax != d_argmax) {
    if (h->bgraph) cudaGraphExecDestroy(h->bgraph);
    if (h->bgraph_src) cudaGraphDestroy(h->bgraph_src);
    h->bgraph = nullptr;
    h->bgraph_src = nullptr;
    cudaError_t e = cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) return fail(h, DEC_ECUDA, "begin capture: %s", cudaGetErrorString(e));
    timing_start(h);
    const int64_t before = h->launches;
    cudaError_t le = launch_rows_setup(h->m, h->stream, meta, d_tokens, host_token, batch);
    if (le == cudaSuccess) le = launch_decode_rows(h->m, h->stream, batch, logits, d_argmax);
    h->bgraph_kernels = h->launches - before;
    h->launches = before;
    h->bgraph_timed_pairs = h->timing.n;
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(h->stream, &g);
    if (le != cudaSuccess || e != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      cudaGetLastError();
      return fail(h, DEC_ECUDA, "batched decode capture: %s", cudaGetErrorString(le != cudaSuccess ? le : e));
    }
    h->bgraph_src = g;
    cudaGraphNode_t roots[4];
    size_t nroots = 4;
    e = cudaGraphGetRootNodes(g, roots, &nroots);
    if (e != cudaSuccess || nroots != 1) {
      drop_graph(h);
      return fail(h, DEC_ECUDA, "batched decode graph: expected one root node (%s)", cudaGetErrorString(e));
    }
    h->bgraph_setup = roots[0];
    e = cudaGraphInstantiate(&h->bgraph, g, 0);
    if (e != cudaSuccess) {
      drop_graph(h);
      return fail(h, DEC_ECUDA, "batched graph instantiate: %s", cudaGetErrorString(e));
    }
    h->bgraph_batch = batch;
    h->bgraph_tokens = d_tokens;
    h->bgraph_logits = logits;
    h->bgraph_argmax = d_argmax;
  }
  cudaError_t e = update_rows_setup_node(h->bgraph, h->bgraph_setup, h->m, meta, d_tokens, host_token, batch);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "batched graph update: %s", cudaGetErrorString(e));
  e = cudaGraphLaunch(h->bgraph, h->stream);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "batched graph launch: %s", cudaGetErrorString(e));
  h->timing.n = h->bgraph_timed_pairs;
  h->launches += h->bgraph_kernels;
  timing_finish(h);
  return DEC_OK;
}

// One step of `batch` sequences through the row kernels; every argument is
// checked before anything is enqueued.
dec_status dec_decode_batch(dec_handle* h, int32_t batch, const int32_t* seqs, const int32_t* positions,
                            const int32_t* d_tokens, float* logits, int32_t* d_argmax) {
  if (!h) return DEC_EINVAL;
  const dec_config& c = h->m.cfg;
  const int bmax = c.max_tokens < MAX_BATCH ? c.max_tokens : MAX_BATCH;
  if (batch < 1 || batch > bmax) return fail(h, DEC_EINVAL, "batch %d outside [1, %d]", batch, bmax);
  if (!seqs || !positions || !d_tokens || !logits)
    return fail(h, DEC_EINVAL, "seqs, positions, d_tokens and logits must not be NULL");
  std::vector<char> seen(h->m.n_seqs, 0);
  for (int32_t i = 0; i < batch; ++i) {
    const int32_t q = seqs[i];
    if (q < 0 || q >= h->m.n_seqs)
      return fail(h, DEC_EINVAL, "row %d: sequence %d outside [0, %d)", i, q, h->m.n_seqs);
    if (seen[q]) return fail(h, DEC_EINVAL, "row %d: sequence %d appears twice in the batch", i, q);
    seen[q] = 1;
    const dec_status st = check_positions(h, q, 1, positions[i]);
    if (st != DEC_OK) return st;
  }
  const dec_status st = run_rows(h, batch, seqs, positions, d_tokens, 0, logits, d_argmax);
  if (st != DEC_OK) return st;
  for (int32_t i = 0; i < batch; ++i) h->lens[seqs[i]] = positions[i] + 1;
  return DEC_OK;
}

int64_t dec_launch_count(const dec_handle* h) { return h ? h->launches : -1; }

dec_status dec_phase_stamps(dec_handle* h, uint64_t* d_stamps, int32_t capacity) {
  if (!h) return DEC_EINVAL;
  const int need = h->m.cfg.n_layers * 6 + 2;
  if (d_stamps && capacity < need) return fail(h, DEC_EINVAL, "phase stamps need %d entries", need);
  h->m.mk_stamps = reinterpret_cast<unsigned long long*>(d_stamps);
  return DEC_OK;
}

dec_status dec_set_fused(dec_handle* h, int32_t mode) {
  if (!h) return DEC_EINVAL;
  if (mode < DEC_FUSED_OFF || mode > DEC_FUSED_CLUSTER) return fail(h, DEC_EINVAL, "unknown schedule %d", mode);
  h->fused_mode = mode;
  return DEC_OK;
}

int32_t dec_fused_mode(const dec_handle* h) {
  if (!h) return -1;
  if (h->fused_mode == DEC_FUSED_CLUSTER && h->m.mk_ok && h->m.mk_cluster > 0) return DEC_FUSED_CLUSTER;
  if (h->fused_mode == DEC_FUSED_GRID && h->m.mk_ok) return DEC_FUSED_GRID;
  return DEC_FUSED_OFF;
}

int32_t dec_ffn_fused(const dec_handle* h) {
  if (!h) return -1;
  const int32_t mode = dec_fused_mode(h);
  if (mode == DEC_FUSED_OFF) return 0;
  return mk_ffn_fused_ok(h->m, mode == DEC_FUSED_CLUSTER ? h->m.mk_cluster : h->m.mk_nb) ? 1 : 0;
}

int32_t dec_fused_available(const dec_handle* h, int32_t mode) {
  if (!h) return 0;
  if (mode == DEC_FUSED_OFF) return 1;
  if (mode == DEC_FUSED_GRID) return h->m.mk_ok ? 1 : 0;
  if (mode == DEC_FUSED_CLUSTER) return h->m.mk_ok && h->m.mk_cluster > 0 ? h->m.mk_cluster : 0;
  return 0;
}

dec_status dec_set_graph(dec_handle* h, int32_t enable) {
  if (!h) return DEC_EINVAL;
  h->use_graph = enable != 0;
  drop_graph(h);
  return DEC_OK;
}

dec_status dec_kv_layer(const dec_handle* h, int32_t layer, void** k, void** v) {
  return dec_kv_layer_seq(h, layer, 0, k, v);
}

dec_status dec_kv_layer_seq(const dec_handle* h, int32_t layer, int32_t seq, void** k, void** v) {
  if (!h || !k || !v || layer < 0 || layer >= h->m.cfg.n_layers || seq < 0 || seq >= h->m.n_seqs ||
      h->m.cfg.page_size > 0)
    return DEC_EINVAL;
  *k = (char*)h->m.layers[layer].kc + (size_t)seq * h->m.ring_bytes;
  *v = (char*)h->m.layers[layer].vc + (size_t)seq * h->m.ring_bytes;
  return DEC_OK;
}

dec_status dec_set_trace(dec_handle* h, int32_t* d_ids, float* d_logits, int32_t capacity) {
  if (!h) return DEC_EINVAL;
  if ((d_ids == nullptr) != (d_logits == nullptr)) return fail(h, DEC_EINVAL, "pass both trace buffers or neither");
  if (d_ids && capacity <= 0) return fail(h, DEC_EINVAL, "trace capacity must be positive");
  h->m.trace_ids = d_ids;
  h->m.trace_logits = d_logits;
  h->m.trace_cap = d_ids ? capacity : 1;
  drop_graph(h);  // the captured graph holds the old trace pointers
  return DEC_OK;
}

dec_status dec_check(dec_handle* h) {
  if (!h) return DEC_EINVAL;
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "stream: %s", cudaGetErrorString(e));
  unsigned words[2];
  e = cudaMemcpy(words, &h->m.s.st->err, sizeof words, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "state read: %s", cudaGetErrorString(e));
  if (words[0]) {
    cudaMemset(&h->m.s.st->err, 0, sizeof words);
    if (words[0] & ERR_TIMEOUT) {
      // A wait that gave up leaves its barrier or last-CTA counter part-way; the
      // stream is idle now, so every counter starts again from zero.
      cudaMemset(h->m.s.st->counters, 0, sizeof h->m.s.st->counters);
      return fail(h, DEC_ETIMEOUT, "a bounded device wait timed out (site %u)", words[1]);
    }
    if (words[0] & ERR_LAYOUT)
      return fail(h, DEC_ECUDA, "a kernel's shared-memory window was not aligned for its tiles (site %u)",
                  words[1]);
    return fail(h, DEC_EINVAL, "a device-side token was outside [0, vocab)");
  }
  return DEC_OK;
}

dec_status dec_selftest_wait_timeout(dec_handle* h, int32_t limit_us) {
  if (!h) return DEC_EINVAL;
  if (limit_us < 1 || limit_us > 100000) return fail(h, DEC_EINVAL, "limit_us must be in [1, 100000]");
  cudaError_t e = launch_wait_selftest(h->m, h->stream, (uint64_t)limit_us * 1000u, DEC_SITE_SELFTEST);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "self-test launch: %s", cudaGetErrorString(e));
  return DEC_OK;
}

dec_status dec_timing_enable(dec_handle* h, int32_t kernel_class, int32_t max_launches) {
  if (!h) return DEC_EINVAL;
  if (kernel_class < 0 || max_launches < 0) return fail(h, DEC_EINVAL, "bad timing arguments");
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return fail(h, DEC_ECUDA, "stream: %s", cudaGetErrorString(e));
  for (cudaEvent_t ev : h->events) cudaEventDestroy(ev);
  h->events.clear();
  h->timing = Timing();
  if (kernel_class > 0 && max_launches > 0) {
    h->events.resize(2 * (size_t)max_launches);
    for (auto& ev : h->events) {
      e = cudaEventCreate(&ev);
      if (e != cudaSuccess) return fail(h, DEC_ECUDA, "event create: %s", cudaGetErrorString(e));
    }
    h->timing.cls = kernel_class;
    h->timing.max = max_launches;
    h->timing.ev = h->events.data();
  }
  drop_graph(h);
  return DEC_OK;
}

dec_status dec_timing_read(dec_handle* h, float* total_ms, int32_t* launches) {
  if (!h || !total_ms || !launches) return DEC_EINVAL;
  float tot = 0.f;
  const int n = h->timing.n_done;
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(h->timing.ev[2 * i + 1]);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, h->timing.ev[2 * i], h->timing.ev[2 * i + 1]);
    if (e != cudaSuccess) return fail(h, DEC_ECUDA, "event read: %s", cudaGetErrorString(e));
    tot += ms;
  }
  *total_ms = tot;
  *launches = n;
  return DEC_OK;
}

void dec_destroy(dec_handle* h) {
  if (!h) return;
  drop_graph(h);
  for (cudaEvent_t ev : h->events) cudaEventDestroy(ev);
  delete h;
}

const char* dec_last_error(const dec_handle* h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

}  // extern "C"
