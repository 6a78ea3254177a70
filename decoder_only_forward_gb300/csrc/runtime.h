// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <type_traits>

#include "../../include/dec.h"
#include "common.cuh"

namespace dec {

// Where the K (or V) row of (sequence, slot) lives, in rows from a layer's K
// (or V) base: contiguous rings (table == nullptr) keep each sequence's
// ring_rows rows together; a paged cache (rml "The decoder", KV cache: pages of
// `page` positions out of one arena) looks the slot's page up in the
// sequence's page table, pages being stride_rows rows apart.
struct KvPaging {
  const int32_t* table;   // device [n_seqs][pages_per_seq] physical page ids, or nullptr
  int pages_per_seq;
  int page;               // slots per page
  long long stride_rows;  // rows between consecutive pages of one layer's K: 2 * n_layers * page
  int ring_rows;          // contiguous rings: rows per sequence
};
__host__ __device__ inline long long kv_phys_row(const KvPaging& pg, int seq, int slot) {
  if (!pg.table) return (long long)seq * pg.ring_rows + slot;
  return (long long)pg.table[seq * pg.pages_per_seq + slot / pg.page] * pg.stride_rows + slot % pg.page;
}

// Per-layer pointers as the persistent decode kernel reads them (device table).
struct MkLayer {
  const float* attn_norm;
  const void* wqkv;
  const float* bqkv;
  const void* wo;
  const float* ffn_norm;
  const void* w_gateup;
  const void* w_down;
  const void* router;
  void* kc;
  void* vc;
  const float* q_norm;   // per-head QK-norm weights [head_dim] (nullable)
  const float* k_norm;
  int rope_local;        // 1: this layer rotates with the local base (per-layer RoPE base)
};

// An 8-bit projection matrix (weight_quant = 1): int8 codes [rows][cols] and one
// f32 scale per 32 columns [rows][cols / 32]; the weight is float32(code * scale).
struct QMat {
  const int8_t* codes;   // nullptr: the matrix is used as given
  const float* scales;
};

struct LayerPtrs {
  const float* attn_norm;
  const void* wqkv;
  const float* bqkv;   // nullable
  const void* wo;
  const float* ffn_norm;
  const void* w_gateup;
  const void* w_down;
  const void* router;  // nullable (dense)
  void* kc;            // this layer's K ring [max_seq][n_kv*hd]
  void* vc;            // this layer's V ring
  const float* q_norm;  // QK-norm weights (nullable)
  const float* k_norm;
  const float* post_attn_norm;  // sandwich norms (nullable)
  const float* post_ffn_norm;
  QMat q_wqkv, q_wo, q_gateup, q_down;   // weight_quant = 1: the quantised projections
  const void* w_down_t;  // persistent decode, fused FFN: w_down transposed, [expert][ffn][hidden] (nullable)
};

// bf16 (hi, lo) operand planes of the tensor-core prefill attention; plane
// 1 (lo) follows plane 0 (hi) at the stated capacity.
struct AttnTcPlanes {
  __nv_bfloat16* Qb;    // [2][qcap][nq*hd] rotated queries (aliases Scratch::Q)
  int qcap;
  __nv_bfloat16* Kb;    // [2][kcap][n_kv*hd] keys as rows, column = position - base
  int kcap;
  __nv_bfloat16* Vt;    // [2][n_kv*hd][vt_ld] values transposed
  int vt_ld;
};

// Device scratch carved out of the caller's workspace (see plan_workspace).
struct Scratch {
  DeviceState* st;
  double* inv_freq;     // [hd/2] RoPE frequencies (llama3-scaled if enabled)
  float2* rope_tab;     // [max(1,max_tokens)][hd/2] (cos, sin) per position of the current call
  double* inv_freq_local;  // the local layers' frequencies (per-layer base), else nullptr
  float2* rope_tab_local;  // their (cos, sin) rows, else nullptr
  float* x;             // [h] decode residual
  float* q;             // [nq*hd]
  float* attn;          // [nq*hd]
  float* act;           // [k_slots*ffn]
  float* nbuf;          // [h] normalised FFN input (MoE)
  int32_t* ids;         // [k] selected experts (decode)
  float* wts;           // [k]
  float* part;          // [nq][nsplit][hd+2] split-K partials
  float* amax_val;      // [LM_GRID_MAX]
  int32_t* amax_idx;    // [LM_GRID_MAX]
  int32_t* tokens;      // [max_tokens] prefill token ids on the device
  // prefill buffers (rows = max_tokens)
  float* X;             // [T][h] residual rows
  void* A;              // [T][max(h, nq*hd, ffn)] GEMM A operand (bf16, or f32 for f32 weights)
  float* Q;             // [T][nq*hd] rotated queries
  void* KVlin_k;        // [max_seq + T][n_kv*hd] linear K for a wrapping append (kv dtype)
  void* KVlin_v;
  int32_t* pf_ids;      // [T][k] routing per row
  float* pf_wts;        // [T][k]
  int32_t* pf_count;    // [E] rows per expert
  int32_t* pf_offset;   // [E+1]
  int32_t* pf_rows;     // [T*k] (row*k + slot) grouped by expert
  int32_t* pf_inv;      // [T*k] sorted position of entry row*k + slot
  void* Asort;          // [T*k][h] normalised rows gathered by expert (MoE)
  float* Y;             // [T*k][h] per-(row, slot) expert outputs (MoE)
  void* ACT;            // [T*k][ffn] gate/up output rows (A operand of down)
  AttnTcPlanes at;      // at.Kb == nullptr: this configuration takes the SIMT attention
  // batched decode (rows = sequences of one step)
  int32_t* b_seq;       // [MAX_BATCH] sequence of each row
  int32_t* b_pos;       // [MAX_BATCH] position of each row
  int32_t* b_rows;      // [MAX_BATCH] K/V row of each row: seq * ring_rows + slot(pos)
  float* b_part;        // [MAX_BATCH][nq][AR_MAX_SPLIT][hd+2] attention split partials
  float* kpart;         // split-K partial sums of the tensor-core GEMMs
  size_t kpart_bytes;
  float* Z;             // [T][h] block output before its post norm (sandwich norms)
  // weight_quant = 1: one matrix expanded for the row GEMMs (bf16 hi, lo planes, or
  // f32 for f32 models) and the two planes' products before their shared epilogue.
  void* deq;
  size_t deq_bytes;
  float* q8part;
  size_t q8part_bytes;
  float* fpart;         // persistent decode, fused FFN: [MK_MAX_NB][h] per-CTA down partials (nullable)
  float* kv_cur;        // persistent decode, int8 cache or QK-norm: [2][n_kv*hd] f32 K and V of the current position
};

constexpr int LM_GRID_MAX = 1024;
constexpr int MAX_EXPERTS = 256;
constexpr int MAX_EXPERTS_USED = 8;
constexpr int MAX_KV_HEADS = 192;
constexpr int MAX_GROUP = 16;     // query heads per kv head
constexpr int NUM_COUNTERS = 256;
constexpr int MAX_BATCH = 256;    // rows of one batched decode step (also <= max_tokens)
constexpr int AR_MAX_SPLIT = 16;  // key splits per kv head in batched decode attention
constexpr int MK_MAX_NB = 256;    // CTAs of the persistent decode step with a fused FFN

// Optional CUDA-event pairs recorded around every launch of one kernel class
// (dec_timing_enable); also captured into the decode graph.
struct Timing {
  int cls = 0;
  int max = 0;
  int n = 0;              // pairs recorded by the current call
  int n_done = 0;         // pairs recorded by the last completed call
  cudaEvent_t* ev = nullptr;
};

struct Model {
  dec_config cfg;
  Timing* timing;       // nullable
  int64_t* launches;    // host counter of kernel launches
  LayerPtrs* layers;    // host array [n_layers]
  const void* tok_embd;
  const float* out_norm;
  const void* head;     // tok_embd when tied
  Scratch s;
  int nsplit;           // split-K CTAs per kv head in decode attention
  int attn_sps;         // KV slots owned by one split
  size_t mk_smem;       // its dynamic shared memory
  int mk_nb;            // its grid (one CTA per SM)
  bool mk_ok;           // the persistent kernel fits this configuration
  int mk_cluster;       // CTAs of its one-cluster schedule (0: the GPU cannot place such a cluster)
  void* mk_maps;        // its weight tensor maps (bf16 weights; device, in the workspace)
  unsigned long long* mk_stamps;  // nullable phase timestamps (dec_phase_stamps)
  int lm_grid;          // CTAs of the LM head kernel
  int32_t* trace_ids;   // nullable
  float* trace_logits;  // nullable
  int trace_cap;
  void* ws;             // workspace base
  size_t ws_bytes;
  KvPaging paging;      // K/V row addressing (device page table when paged)
  int n_seqs;           // sequences whose KV rings the workspace holds
  int ring_rows;        // rows of one sequence's ring (max_seq rounded up to 64)
  size_t ring_bytes;    // bytes of one sequence's K (or V) ring of one layer
  int num_sms;
  bool wq8;             // weight_quant = 1
  QMat q_head;          // the quantised LM head (untied), else no codes
};

// Workspace plan: byte offsets of every region; total size.
struct WsPlan {
  size_t st, inv_freq, rope_tab, x, q, attn, act, nbuf, ids, wts, part, amax_val, amax_idx, tokens;
  size_t X, A, Q, KVlin_k, KVlin_v, pf_ids, pf_wts, pf_count, pf_offset, pf_rows, pf_inv, Asort, Y, ACT;
  size_t at_Kb, at_Vt;
  int at_kcap, at_vt_ld;  // 0: no tensor-core prefill attention for this configuration
  size_t wqkv_perm, bqkv_perm;  // kHalf RoPE: q/k rows permuted per head
  size_t mk_maps;       // its weight tensor maps
  size_t b_seq, b_pos, b_rows, b_part;  // batched decode
  size_t kpart, kpart_bytes;            // split-K partials
  size_t Z;                             // sandwich block outputs
  size_t inv_freq_local, rope_tab_local;  // per-layer RoPE base
  size_t page_table;                      // paged cache: [n_seqs][pages_per_seq] int32
  int pages_per_seq;
  size_t qk_perm;                       // kHalf + QK-norm: permuted norm weights
  size_t q8, q8_bytes;                  // weight_quant: codes and scales of every quantised matrix
  size_t deq, deq_bytes, q8part, q8part_bytes;
  size_t wdown_t, fpart;                // fused decode FFN: transposed down projections, partials
  size_t kv_cur;                        // persistent decode, int8 cache: the current K/V rows in f32
  size_t kv;            // start of the KV rings: [layer][K, V][seq][ring_rows][n_kv*hd]
  size_t kv_layer_bytes; // one layer's K (or V) rings of every sequence
  size_t ring_bytes;    // one sequence's ring
  int ring_rows;
  int n_seqs;
  size_t total;
  int nsplit;
  int attn_sps;
  int max_tokens;
};

WsPlan plan_workspace(const dec_config& c);

// Inside stream capture an event record must be an external node to be
// timeable after the graph runs; outside capture a plain record is used.
inline void record_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else cudaEventRecord(ev, s);
}
inline void timer_begin(const Model& m, int cls, cudaStream_t s) {
  Timing* t = m.timing;
  if (t && t->cls == cls && t->n < t->max) record_event(t->ev[2 * t->n], s);
}
inline void timer_end(const Model& m, int cls, cudaStream_t s) {
  Timing* t = m.timing;
  if (t && t->cls == cls && t->n < t->max) {
    record_event(t->ev[2 * t->n + 1], s);
    ++t->n;
  }
}

// decode.cu
void launch_set_step(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos);
// One whole decode step: the setup kernel (token, position, RoPE row) first.
void launch_decode_body(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos,
                        float* logits, int32_t* d_argmax);
// Host handle of the setup kernel (for updating its node in a captured graph).
const void* set_step_kernel();

// int8 K/V rows (kv_int8.cu): [scales: kd/G f32, padded to 16 B][codes: kd
// int8, padded to 16 B], G the largest power of two dividing head_dim, <= 32.
struct KvRowLayout {
  int bytes;      // one ring row
  int code_off;   // bytes before the codes (the scales' area)
  int group;      // channels per scale
};
// int8 caches at head_dim 128 with bf16 weights decode on the persistent step
// (a head's group scales are one 16-byte block there, a whole TMA stride); the
// per-layer decode kernels do not read int8 rows.
inline bool decode_kv_i8_persistent(const dec_config& c) {
  return c.kv_dtype == DEC_I8 && c.head_dim == 128 && c.weight_dtype == DEC_BF16 && !c.weight_quant;
}
// Models whose decode runs the row kernels (one row per step): the persistent
// step and the per-layer decode kernels implement none of these.
// Per-head QK-norm (one shared head_dim weight) decodes on the persistent step at
// head_dim 64 / 128 with bf16 weights and an f32 cache: the attention task normalises
// and rotates its heads' q and the current k itself (the QKV phase leaves them raw).
// The row-long norm needs a whole row's sum and stays on the row kernels.
inline bool decode_qkn_persistent(const dec_config& c) {
  return c.qk_norm == 1 && c.kv_dtype == DEC_F32 && c.weight_dtype == DEC_BF16 && !c.weight_quant &&
         (c.head_dim == 64 || c.head_dim == 128);
}
inline bool decode_needs_rows(const dec_config& c) {
  return (c.kv_dtype == DEC_I8 && !decode_kv_i8_persistent(c)) || (c.qk_norm != 0 && !decode_qkn_persistent(c)) ||
         c.sandwich_norms != 0 || c.page_size > 0;
}
// Whether layer l rotates with the global base (every layer without a local base).
inline bool layer_rope_global(const dec_config& c, int l) {
  if (!(c.rope_theta_local > 0.f)) return true;
  return c.rope_global_every > 0 && (l + 1) % c.rope_global_every == 0;
}
inline int kv_group_size(int hd) {
  int g = 1;
  while (g < 32 && hd % (2 * g) == 0) g *= 2;
  return g;
}
inline KvRowLayout kv_row_layout(const dec_config& c) {
  const int kd = c.n_kv_heads * c.head_dim;
  if (c.kv_dtype != DEC_I8) return KvRowLayout{kd * (c.kv_dtype == DEC_BF16 ? 2 : 4), 0, 1};
  const int g = kv_group_size(c.head_dim);
  const int sb = (kd / g * 4 + 15) / 16 * 16;
  return KvRowLayout{sb + (kd + 15) / 16 * 16, sb, g};
}
// f32 rows -> int8 ring rows: row r to dst_rows[r] (rows from the layer base),
// or to the row of (seq, slot of position pos0 + r) under pg; rows below t_first
// are not stored; rt_k/rt_v (nullable) get the values read back.  planes: 2 =
// K and V, 1 = K only.
void launch_kv_quant(const dec_config& c, const float* src_k, const float* src_v, int n, const int32_t* dst_rows,
                     const KvPaging& pg, int seq, int pos0, int t_first, void* ring_k, void* ring_v, float* rt_k,
                     float* rt_v, cudaStream_t s, int planes = 2);
// int8 rows of positions h0 .. h0+count-1 of sequence seq -> f32 rows.
void launch_kv_gather_i8(const dec_config& c, const void* ring_k, const void* ring_v, const KvPaging& pg, int seq,
                         int h0, int count, float* lin_k, float* lin_v, cudaStream_t s);
// Paged cache: table[idx[i]] = val[i] for the n entries (at most 256 per launch).
struct PageSet {
  int n;
  int32_t idx[256];
  int32_t val[256];
};
void launch_set_pages(int32_t* table, const PageSet& ps, cudaStream_t s);

// Streaming multiprocessors of the current device, queried once per device (1 when
// no device can be queried).  Grid sizes follow it rather than a fixed part.
int device_sm_count();

// 8-bit projection weights (weight_int8.cu).
// Quantises rows [rows][cols] (cols % 32 == 0) of w (f32 or bf16) into codes and scales.
cudaError_t launch_weight_quant(const void* w, bool w_bf16, size_t rows, int cols, int8_t* codes, float* scales,
                                cudaStream_t s);
// Sum of `planes` f32 partial planes [planes][M][N] in order, then the GEMM epilogue e.
struct GemmEpi;
cudaError_t launch_sum_planes_epi(const float* part, int planes, int M, int N, const GemmEpi& e, cudaStream_t s);
// Expands rows [rows][cols] of q into bf16 (hi, lo) planes (hi + lo ~ code * s), or into f32.
cudaError_t launch_weight_dequant_hilo(const QMat& q, size_t rows, int cols, __nv_bfloat16* hi,
                                       __nv_bfloat16* lo, cudaStream_t s);
cudaError_t launch_weight_dequant_f32(const QMat& q, size_t rows, int cols, float* out, cudaStream_t s);

// Persistent single-kernel decode step (decode_mk.cu).
size_t mk_smem_bytes(const dec_config& c, int nsplit);
size_t mk_maps_bytes(const dec_config& c);
bool mk_prepare(Model& m, int num_sms);
// Whether the persistent step runs its FFN fused (one phase over ffn slices + partial sums) on nb CTAs.
bool mk_ffn_fused_ok(const Model& m, int nb);
// Whether a configuration gets the fused FFN's transposed down copy in its workspace.
bool mk_ffn_fused_layout(const dec_config& c);
// dst[b] = src[b]^T for `batch` bf16 matrices of rows x cols.
cudaError_t launch_transpose_bf16(const void* src, int rows, int cols, int batch, void* dst, cudaStream_t s);
// cluster: run on one thread-block cluster of m.mk_cluster CTAs, else over m.mk_nb CTAs (one per SM).
void launch_decode_mk(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos,
                      float* logits, int32_t* d_argmax, bool cluster);
// Bounded-wait self-test: one CTA in the persistent step's grid barrier with an
// arrival that never comes; the wait gives up after limit_ns and records the site.
cudaError_t launch_wait_selftest(const Model& m, cudaStream_t s, uint64_t limit_ns, unsigned site);
// Final RMSNorm + LM head (+ argmax) of one residual row x.
void launch_lmhead(const Model& m, cudaStream_t s, const float* x, float* logits, int32_t* d_argmax);

// prefill.cu
// Runs tokens (already in m.s.tokens[0..n)) at positions start..start+n-1; writes
// the last row's logits when logits != nullptr.  wrap_mode: K/V go through the
// linear scratch and are committed afterwards (needed once the ring may wrap).
// Returns the first launch-setup error (a tensor map the driver rejects, ...).
// seq: the sequence whose rings the chunk reads and writes.
cudaError_t launch_prefill_chunk(const Model& m, cudaStream_t s, int seq, int n, int start, float* logits,
                                 int32_t* d_argmax);
// One batched decode step over B rows: token ids in m.s.tokens, sequences,
// positions and K/V rows in m.s.b_seq / b_pos / b_rows (device).  Writes
// logits [B][vocab] and, when d_argmax is given, each row's argmax.
cudaError_t launch_decode_rows(const Model& m, cudaStream_t s, int B, float* logits, int32_t* d_argmax);
// Its setup: per-row sequence, position and K/V row into m.s.b_*, token ids
// from d_tokens (checked) and each row's RoPE (cos, sin).
struct RowsMeta {
  int32_t seq[MAX_BATCH];
  int32_t pos[MAX_BATCH];
  int32_t rows[MAX_BATCH];   // seq * ring_rows + slot(pos)
};
// d_tokens == nullptr: one row whose token is host_token.
cudaError_t launch_rows_setup(const Model& m, cudaStream_t s, const RowsMeta& meta, const int32_t* d_tokens,
                              int32_t host_token, int B);
// Points a captured setup node (of a graph captured for the same B) at new rows.
cudaError_t update_rows_setup_node(cudaGraphExec_t g, cudaGraphNode_t node, const Model& m, const RowsMeta& meta,
                                   const int32_t* d_tokens, int32_t host_token, int B);

struct RowOut;
// Batched decode attention (attn_rows.cu): rotated queries Q [B][nq*hd] f32,
// the layer's K/V bases kc/vc, rows addressed through pg.
int attn_rows_splits(const dec_config& c);
void launch_attn_rows(const dec_config& c, const float* Q, const void* kc, const void* vc, const KvPaging& pg,
                      const int32_t* seq, const int32_t* pos, int B, int nsplit, float* part, RowOut out,
                      cudaStream_t s);

inline void count_launch(const Model& m, int n = 1) { *m.launches += n; }

// Standalone attention over a KV ring (decode.cu).  st/part: scratch of
// attend_scratch_layout().
void launch_attend(const float* q, const void* kc, const void* vc, int nq, int nkv, int hd, int max_seq,
                   int sliding, int kv_dtype, int pos, int nsplit, DeviceState* st, float* part, float* out,
                   cudaStream_t s);

struct AttendLayout {
  int nsplit;
  size_t part_offset;   // bytes from the scratch base to the partials
  size_t total;         // bytes of scratch needed
};
// Checks the arguments of a standalone attention call; on success fills lay.
bool attend_check(const void* q, const void* k, const void* v, const void* out, int nq, int nkv, int hd,
                  int max_seq, int sliding, int kv_dtype, int pos, AttendLayout& lay, const char** why);

// Tensor-core GEMM (gemm_tc.cu); see prefill_common.cuh for GemmEpi.
struct GemmEpi;
// kpart (nullable): f32 scratch of kpart_bytes for split-K partial sums.
cudaError_t launch_gemm_tc(const void* a_hi, const void* a_lo, int a_rows, const void* b, int M, int N, int K,
                           const GemmEpi& e, int groups, int max_rows, float* kpart, size_t kpart_bytes,
                           DeviceState* st, cudaStream_t s);

struct RowOut;
// Tensor-core causal prefill attention (attn_tc.cu) over key columns
// [0, start + n - base_pos); head_dim 64 or 128.  launch_kv_split fills the K
// and V^T planes of rows [r0, r1) from f32 K/V row buffers.
cudaError_t launch_attn_prefill_tc(const AttnTcPlanes& pl, int n, int start, int base_pos, int nq, int nkv, int hd,
                                   int sliding, RowOut out, DeviceState* st, cudaStream_t s);
cudaError_t launch_kv_split(const float* K, const float* V, int kd, int r0, int r1, const AttnTcPlanes& pl,
                            cudaStream_t s);
// The tensor-core prefill attention reads f32 K/V rows: the f32 cache itself,
// or the f32 read-back of an int8 cache.
inline bool attn_tc_supported(const dec_config& c) {
  return c.kv_dtype != DEC_BF16 && (c.head_dim == 64 || c.head_dim == 128);
}

// Copies one layer's wqkv (and bqkv) with the q/k rows of every head permuted
// so that kHalf RoPE pairs (i, i + rope_dim/2) become adjacent (api.cu).
void launch_permute_qk_rows(const dec_config& c, const void* w, const float* b, void* wdst, float* bdst,
                            cudaStream_t s);
// A per-head vector (n = heads * hd) in the same permuted dim order.
void launch_permute_head_vector(const dec_config& c, const float* src, int n, float* dst, cudaStream_t s);

// Message returned by dec_last_error(NULL) (api.cu).
void set_global_error(const char* msg);

}  // namespace dec
