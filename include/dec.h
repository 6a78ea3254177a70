/*
 * dec.h -- C ABI of libdec.so: the decoder-only transformer forward pass over a
 * KV cache (single-pass prefill and one-token decode) on one NVIDIA GB300.
 *
 * What is computed, per layer, pre-norm (Pantheon "Llama Forward Pass",
 * Forward Pass Flow; rml "The decoder", One forward pass):
 *   RMSNorm -> Q/K/V projection (+ optional q/k/v bias) -> adjacent-pair RoPE
 *   (sipllm "Transformer forward pass", RoPE is adjacent-pair; optional llama3
 *   frequency scaling, rml Rotary embeddings) -> K/V written at pos (a circular
 *   buffer under a sliding window, Pantheon Sliding Window) -> causal GQA
 *   attention, query head h reading kv head h*n_kv/n_head (Pantheon Grouped
 *   Query Attention; rml Attend) -> output projection + residual -> RMSNorm ->
 *   SwiGLU FFN or router softmax / top-k / renormalise / weighted expert sum
 *   (Pantheon Mixture of Experts) + residual; then final RMSNorm and LM head.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device addresses on the handle's device;
 *     "host" are ordinary host addresses.  Nothing here takes torch types.
 *   - Ownership: the caller owns the weights, the workspace and every output
 *     buffer; the library never allocates device memory and never frees caller
 *     memory.  Weights and workspace must outlive the handle.
 *   - Work is enqueued on the handle's stream and the call returns; outputs are
 *     valid once that stream has been synchronised.
 *   - Argument errors are detected on the host before anything is enqueued or
 *     any state changes (rml "The decoder", One forward pass, step 1: "in every
 *     case nothing has changed yet").
 *   - Matrices are row-major [out, in] (each output's weights contiguous).
 */
#ifndef DEC_H
#define DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dec_status {
  DEC_OK = 0,
  DEC_EINVAL = 1,   /* bad argument: empty input, token outside [0,vocab), NULL, bad config, bad position */
  DEC_ERANGE = 2,   /* the cache is full (no sliding window and start_pos + n > max_seq) */
  DEC_ECUDA = 3,    /* a CUDA call failed; dec_last_error() has the CUDA message */
  DEC_ETIMEOUT = 4, /* a bounded device wait gave up; the kernel returned without finishing */
  DEC_ENOMEM = 5    /* the workspace is smaller than dec_workspace_bytes() */
} dec_status;

typedef enum dec_dtype {
  DEC_F32 = 0,
  DEC_BF16 = 1,
  DEC_I8 = 2   /* K/V cache only: int8 codes with one f32 scale per group of channels (rml "The decoder",
                  KV cache): the group is the largest power of two dividing head_dim, at most 32; each
                  group stored as round(x / s), s = max|x| / 127, in f32 with halves rounded away from
                  zero and codes in [-127, 127]; read back as code * s.  A ring row is the row's scales
                  (kd/group f32, padded to 16 bytes) then its codes (kd int8, padded to 16 bytes) */
} dec_dtype;

/*
 * Model configuration: sizes plus switches (rml "The decoder", The model
 * config).  Fixed layout with no build-dependent fields (Pantheon ABI note).
 */
typedef struct dec_config {
  int32_t n_layers;
  int32_t hidden;         /* h */
  int32_t n_heads;        /* query heads */
  int32_t n_kv_heads;     /* n_heads % n_kv_heads == 0 */
  int32_t head_dim;       /* even (RoPE rotates pairs) */
  int32_t ffn;            /* SwiGLU inner size (per expert for MoE) */
  int32_t vocab;
  int32_t n_experts;      /* 0 = dense FFN */
  int32_t n_experts_used; /* top-k, 1 <= k <= n_experts (0 when dense) */
  int32_t max_seq;        /* KV slots per layer; = min(sliding_window, n_ctx) under a window */
  int32_t sliding_window; /* 0 = full causal; else window W (W positions including the query) */
  int32_t max_tokens;     /* largest n of one dec_prefill call the workspace holds (0 = max_seq);
                             longer calls are processed in chunks of max_tokens */
  int32_t tied_embedding; /* 1: LM head = token embedding matrix */
  int32_t qkv_bias;       /* 1: bqkv present */
  int32_t weight_dtype;   /* DEC_F32 or DEC_BF16: projection, embedding, router, head matrices */
  int32_t kv_dtype;       /* DEC_F32, DEC_BF16 or DEC_I8: KV cache storage.  With DEC_I8, decode
                             (dec_decode, dec_decode_dev) runs the persistent schedules when head_dim
                             is 128 with bf16 weights and no weight_quant (the attention reads the
                             codes and scales, and quantises the new position's row itself); otherwise,
                             and under DEC_FUSED_OFF, and with sandwich_norms or qk_norm 2, it runs the
                             batched row kernels with one row */
  float rms_eps;
  float rope_theta;
  int32_t rope_llama3;    /* 1: llama3 frequency scaling with the four fields below */
  float rope_factor;
  float rope_low_freq_factor;
  float rope_high_freq_factor;
  int32_t rope_orig_ctx;
  int32_t rope_half;      /* which dimensions pair (rml "The decoder", Rotary embeddings): 0 = adjacent
                             (2i, 2i+1) (kInterleaved, llama.cpp order); 1 = (i, i + rope_dim/2)
                             (kHalf, rotate_half).  With 1, the library keeps a per-head row-permuted
                             copy of each layer's q/k weight rows and biases in the workspace, and
                             the K cache holds each head's dims in the adjacent order
                             (0, d/2, 1, d/2+1, ..., then the unrotated tail) */
  int32_t rope_dim;       /* rotary width: only the first rope_dim dims of a head turn, the rest
                             pass through (sipllm partial-rotary rope_rot); 0 = head_dim; even,
                             <= head_dim.  inv_freq_i = theta^(-2i/rope_dim) */
  int32_t n_seqs;         /* independent sequences whose KV rings the workspace holds (0 = 1): each
                             has its own positions and length.  dec_prefill / dec_decode /
                             dec_kv_reset act on sequence 0; dec_prefill_seq, dec_kv_reset_seq and
                             dec_decode_batch on any (Pantheon "Llama Forward Pass", Batched
                             Multi-Sequence Decode: a KV cache and position per sequence) */
  int32_t qk_norm;        /* QK-norm (rml "The decoder", One forward pass step 4): after the biases and
                             before RoPE, q and k are RMS-normalised with eps = rms_eps.  0 off; 1 per head
                             with one [head_dim] weight shared by the heads (q_norm, k_norm); 2 over the whole
                             q / k row with [n_heads*head_dim] / [n_kv_heads*head_dim] weights.  Not with a
                             DEC_BF16 cache (DEC_EINVAL).  Decode: mode 1 with bf16 weights, an f32 cache and
                             head_dim 64 / 128 runs the persistent schedules (the attention normalises and
                             rotates q and the new k); other cases, and DEC_FUSED_OFF, run the row kernels */
  int32_t sandwich_norms; /* 1: each block's output (attention after wo, FFN after the down projection or
                             the expert sum) is RMS-normalised with post_attn_norm / post_ffn_norm before
                             the residual add (rml "The decoder", One forward pass step 6) */
  float rope_theta_local; /* per-layer RoPE base (sipllm "Transformer forward pass", RoPE: Gemma 3): 0 = one
                             base; else local layers rotate with this base (no llama3 scaling) and every
                             rope_global_every-th layer, l with (l + 1) % rope_global_every == 0, with
                             rope_theta (0 = no global layer).  Decode takes the persistent schedules
                             (both tables per step) when the rest of the config allows; DEC_FUSED_OFF runs
                             the row kernels */
  int32_t rope_global_every;
  int32_t page_size;      /* 0: each sequence owns contiguous K/V rings of max_seq rows.  Else a paged cache
                             (rml "The decoder", KV cache): slots are grouped in pages of page_size positions
                             (a power of two >= 16); pages come from one arena of n_pages pages reserved up
                             front, each holding its span for every layer (rows ordered page, layer, K/V,
                             slot), and a sequence takes a page only when a position first lands in it, so
                             memory follows the sequences' lengths rather than n_seqs * max_seq.  Pages are
                             returned by dec_kv_reset / dec_kv_reset_seq.  A call that needs more pages than
                             are free fails with DEC_ENOMEM before anything changes.  Decode of a paged cache
                             runs the row kernels */
  int32_t n_pages;        /* pages in the arena (with page_size > 0) */
  int32_t weight_quant;   /* 0: projections used as given.  1: 8-bit projection weights (Pantheon "Llama Forward
                             Pass", weight modes: the projections stay quantised and are expanded a block at a
                             time): dec_create quantises Wq|Wk|Wv, Wo, gate/up, down (every expert) and an untied
                             LM head into the workspace, each row in groups of 32 input columns as
                             round(w / s) with s = max|w| / 127 (the int8 rule the pages give for the cache;
                             float32 arithmetic, round = halves away from zero, codes in [-127, 127]), and
                             every later call reads those codes and scales: the forward pass uses
                             float32(code * s).  Embeddings, norms, biases and the router stay as given.
                             hidden, ffn and n_heads * head_dim must be multiples of 32.  The projection
                             pointers are read by dec_create only */
} dec_config;

/*
 * Per-layer weight views (device).  Norm weights and biases are f32; the
 * matrices are weight_dtype.  Layouts:
 *   attn_norm, ffn_norm [hidden]
 *   wqkv      [(n_heads + 2*n_kv_heads)*head_dim, hidden]: rows Wq, then Wk, then Wv
 *   bqkv      [(n_heads + 2*n_kv_heads)*head_dim] or NULL (no bias)
 *   wo        [hidden, n_heads*head_dim]
 *   w_gateup  dense: [2*ffn, hidden] with gate row r at 2r and up row r at 2r+1;
 *             MoE:   [n_experts, 2*ffn, hidden], each expert interleaved the same way
 *   w_down    dense: [hidden, ffn];  MoE: [n_experts, hidden, ffn]
 *   router    MoE only: [n_experts, hidden]; NULL when dense
 */
typedef struct dec_layer_weights {
  const void *attn_norm, *wqkv, *bqkv, *wo, *ffn_norm, *w_gateup, *w_down, *router;
  const void *q_norm, *k_norm;                /* f32, with qk_norm (see dec_config); else NULL */
  const void *post_attn_norm, *post_ffn_norm; /* f32 [hidden], with sandwich_norms; else NULL */
} dec_layer_weights;

typedef struct dec_weights {
  const void *tok_embd;             /* [vocab, hidden] weight_dtype, device */
  const void *out_norm;             /* [hidden] f32, device */
  const void *lm_head;              /* [vocab, hidden] weight_dtype, device; NULL when tied */
  const dec_layer_weights *layers;  /* host array of n_layers entries (copied by dec_create) */
} dec_weights;

typedef struct dec_handle dec_handle;

/* Checks a configuration (rml "The decoder", ValidateConfig: positive sizes,
 * heads split evenly into kv groups, even head_dim, positive eps/theta/scales,
 * 1 <= experts used <= experts) plus this library's limits.  Host only, needs
 * no GPU.  Writes a message into msg (may be NULL).  Returns DEC_OK or DEC_EINVAL. */
dec_status dec_config_validate(const dec_config *cfg, char *msg, size_t msg_len);

/* Bytes of device workspace dec_create needs for cfg (KV cache plus all
 * scratch).  0 if cfg is invalid.  Host only.  For bf16 weights without
 * weight_quant whose hidden size is a multiple of 128 and ffn a multiple of 16,
 * this includes a transposed copy of every w_down ([expert][ffn][hidden], bf16,
 * the size of w_down itself) read by the persistent decode step's FFN phase, and
 * 256 * hidden floats of its partial sums. */
size_t dec_workspace_bytes(const dec_config *cfg);

/* Creates a handle.  workspace: device, >= dec_workspace_bytes(cfg) bytes,
 * 256-byte aligned, owned by the caller.  cuda_stream: a cudaStream_t (NULL =
 * legacy default stream).  Weights are validated for presence and 16-byte
 * alignment.  The weights must be complete when work on cuda_stream starts:
 * dec_create itself enqueues kernels that read them (8-bit quantisation, the
 * kHalf row permutation, the transposed w_down copy), so a caller that wrote
 * them on another stream makes cuda_stream wait for it first.  Errors:
 * DEC_EINVAL (config, NULL or misaligned pointers), DEC_ENOMEM (workspace too
 * small), DEC_ECUDA. */
dec_status dec_create(const dec_config *cfg, const dec_weights *weights, void *workspace,
                      size_t workspace_bytes, void *cuda_stream, dec_handle **out);

/* Single-pass prefill (sipllm "Transformer forward pass", Single-pass prefill;
 * rml Forward with n tokens): runs tokens[0..n) at positions start_pos.. through
 * every layer, each layer once for all positions, writes their K/V, and writes
 * the LAST position's logits.
 *   tokens: host, n ids in [0, vocab).  logits: device, [vocab] f32 (may be NULL
 *   to skip the head).  d_argmax: device int32 or NULL; when given, receives
 *   argmax(logits) (ties -> lower id), the first greedy token.
 *   start_pos <= current length; start_pos < length drops the later history.
 *   Under a sliding window, once positions have wrapped the ring, start_pos must
 *   equal the length (a rewind would need overwritten slots).
 * Errors: DEC_EINVAL (n <= 0, bad token, bad start_pos), DEC_ERANGE (no window
 * and start_pos + n > max_seq), DEC_ECUDA. */
dec_status dec_prefill(dec_handle *h, const int32_t *tokens, int32_t n, int32_t start_pos,
                       float *logits, int32_t *d_argmax);

/* One-token decode (sipllm Transformer::forward(token, pos)): identical in
 * meaning to dec_prefill(&token, 1, pos, logits), run with the decode kernels.
 * logits: device [vocab] f32. */
dec_status dec_decode(dec_handle *h, int32_t token, int32_t pos, float *logits);

/* Decode step whose token is read from device memory (greedy loops without a
 * host round trip).  d_token: device int32.  d_argmax: device int32 or NULL;
 * when given, receives argmax(logits) (ties -> lower id).  A token outside
 * [0, vocab) read from d_token is replaced by 0 and reported as DEC_EINVAL by
 * dec_check(). */
dec_status dec_decode_dev(dec_handle *h, const int32_t *d_token, int32_t pos, float *logits,
                          int32_t *d_argmax);

/* Empties the cache (length 0).  Slots are not cleared: the readable length
 * gates every read. */
dec_status dec_kv_reset(dec_handle *h);

/* Number of positions currently in the cache (host-side bookkeeping). */
int32_t dec_length(const dec_handle *h);

/* Sequence-addressed forms of dec_prefill, dec_kv_reset and dec_length:
 * seq in [0, n_seqs) selects whose KV rings are read and written; the rules of
 * the plain calls apply per sequence.  DEC_EINVAL for seq out of range
 * (dec_length_seq returns -1). */
dec_status dec_prefill_seq(dec_handle *h, int32_t seq, const int32_t *tokens, int32_t n, int32_t start_pos,
                           float *logits, int32_t *d_argmax);
dec_status dec_kv_reset_seq(dec_handle *h, int32_t seq);
int32_t dec_length_seq(const dec_handle *h, int32_t seq);

/* Batched decode: one step of `batch` independent sequences, row i being token
 * d_tokens[i] of sequence seqs[i] at position positions[i] (Pantheon "Llama
 * Forward Pass", Batched Multi-Sequence Decode: each sequence keeps its own KV
 * cache and position and attends only to its own keys; one weight read serves
 * every row, the throughput lever named under "Future work" of sipllm
 * "Transformer forward pass").  Projections, FFN/MoE and the LM head run as
 * tensor-core GEMMs over the rows (the prefill kernels).  A row's result is
 * bit-identical whatever the other rows, its place in the batch or the batch
 * size; against dec_decode it agrees to rounding (different kernels).
 *   batch: 1 <= batch <= min(max_tokens, 256).
 *   seqs, positions: host, batch entries; sequences distinct, in [0, n_seqs);
 *     each position obeys the dec_decode rules for its sequence.
 *   d_tokens: device, batch int32 ids in [0, vocab) (a device id outside is
 *     replaced by 0 and reported by dec_check as DEC_EINVAL).
 *   logits: device [batch][vocab] f32, row i for row i.
 *   d_argmax: device [batch] int32 or NULL: each row's argmax (ties -> lower id).
 * Errors (host-side, before anything is enqueued or any length changes):
 * DEC_EINVAL, DEC_ERANGE; DEC_ECUDA from a launch. */
dec_status dec_decode_batch(dec_handle *h, int32_t batch, const int32_t *seqs, const int32_t *positions,
                            const int32_t *d_tokens, float *logits, int32_t *d_argmax);

/* Device pointers to layer's K and V rings, each [max_seq][n_kv_heads][head_dim]
 * of kv_dtype (DEC_I8: max_seq rows of the int8 row format of dec_dtype);
 * position p lives in slot p % max_seq under a window, else slot p. */
dec_status dec_kv_layer(const dec_handle *h, int32_t layer, void **k, void **v);

/* The same for sequence seq in [0, n_seqs) (dec_kv_layer is sequence 0).
 * DEC_EINVAL for a paged cache (its rows are not contiguous: use dec_kv_slot). */
dec_status dec_kv_layer_seq(const dec_handle *h, int32_t layer, int32_t seq, void **k, void **v);

/* Device pointers to the K and V rows (n_kv_heads * head_dim elements of kv_dtype, or one
 * DEC_I8 row) of slot `slot` of sequence seq in layer `layer`, for either layout.
 * DEC_EINVAL for arguments out of range or a page the sequence does not hold. */
dec_status dec_kv_slot(const dec_handle *h, int32_t layer, int32_t seq, int32_t slot, void **k, void **v);

/* Paged cache: pages currently free in the arena (-1 for NULL or an unpaged cache). */
int32_t dec_pages_free(const dec_handle *h);

/* Optional MoE trace for testing: when d_ids/d_logits are non-NULL, every
 * later MoE layer records, for position p, its selected expert ids
 * (d_ids[(layer*capacity + p % capacity)*n_experts_used + j]) and router logits
 * (d_logits[(layer*capacity + p % capacity)*n_experts + e]).  Pass NULLs to stop.
 * Buffers are device memory owned by the caller. */
dec_status dec_set_trace(dec_handle *h, int32_t *d_ids, float *d_logits, int32_t capacity);

/* Decode step schedules (dec_set_fused). */
typedef enum dec_schedule {
  DEC_FUSED_OFF = 0,      /* per-layer kernels chained by programmatic dependent launch in a CUDA graph */
  DEC_FUSED_GRID = 1,     /* ONE persistent cooperative kernel per step over every SM: every layer and the
                             head, grid-wide barriers between phases, weights streamed by bulk copies */
  DEC_FUSED_CLUSTER = 2   /* the same persistent step on ONE thread-block cluster (up to 16 SMs), whose
                             phase barriers are shared-memory mbarriers across the cluster */
} dec_schedule;

/* Selects the decode step schedule.  A schedule the configuration or GPU cannot
 * take (see dec_fused_available) falls back to DEC_FUSED_OFF at each step.
 * dec_create picks DEC_FUSED_GRID when the weights read per token reach
 * 512 MB, else DEC_FUSED_OFF (small models: latency-bound).  Results agree to
 * rounding.  DEC_EINVAL for an unknown mode. */
dec_status dec_set_fused(dec_handle *h, int32_t mode);

/* Whether a schedule can run on this handle: 1 (DEC_FUSED_OFF, DEC_FUSED_GRID),
 * the cluster's CTA count (DEC_FUSED_CLUSTER), or 0.  The persistent schedules need
 * at most 128 layers (the layer table travels in the kernel's parameters), at most 8
 * query heads per kv head at head_dim 64 and 4 at head_dim 128, and a shared-memory
 * plan within the GPU's limit. */
int32_t dec_fused_available(const dec_handle *h, int32_t mode);

/* The schedule the next decode step takes (after any fallback); -1 for NULL. */
int32_t dec_fused_mode(const dec_handle *h);

/* Whether the next decode step runs its FFN as one phase over ffn slices plus a
 * partial-sum phase (1: a persistent schedule, bf16 weights without weight_quant,
 * hidden a multiple of 128, ffn a multiple of 16, at most 256 (slot, ffn) tasks per
 * CTA) or as a gate/up phase and a down phase (0); -1 for NULL. */
int32_t dec_ffn_fused(const dec_handle *h);

/* Measurement hook of the persistent decode step: when d_stamps (device,
 * >= 6*n_layers + 2 entries) is set, every later fused decode step writes the
 * GPU's nanosecond timer at its start ([0]) and after each of its phases
 * (QKV, attention, [merge], output projection, gate/up, down per layer; then
 * the head).  With the transposed w_down copy (see dec_workspace_bytes) the last
 * two phases of a layer are the whole FFN over each CTA's ffn slice (gate/up,
 * then that slice's share of the down projection) and the sum of those shares
 * into the residual.  NULL stops it. */
dec_status dec_phase_stamps(dec_handle *h, uint64_t *d_stamps, int32_t capacity);

/* Decode steps run as one captured CUDA graph by default (when the handle's
 * stream is not the legacy default stream).  enable = 0 launches the kernels
 * one by one instead (e.g. under a per-kernel profiler). */
dec_status dec_set_graph(dec_handle *h, int32_t enable);

/* Number of kernels this handle has launched so far (graph launches count
 * every kernel node), for measurement. */
int64_t dec_launch_count(const dec_handle *h);

/* Synchronises the handle's stream and reports device-side errors raised since
 * the last check: DEC_ETIMEOUT (a bounded wait gave up; the handle's barrier and
 * last-CTA counters are reset so later calls start clean), DEC_EINVAL (a device
 * token out of range), DEC_ECUDA (a CUDA error, or a kernel whose shared-memory
 * window was not aligned for its tile layout and did no work). */
dec_status dec_check(dec_handle *h);

/* Site number that dec_check names after dec_selftest_wait_timeout's wait ran out. */
#define DEC_SITE_SELFTEST 901

/* Self-test of the failure path of a bounded device wait (rml "The decoder", One
 * forward pass: errors come back as a status, the handle stays usable).  Enqueues on
 * the handle's stream one CTA that enters the persistent decode step's grid barrier
 * expecting two arrivals; the second never comes, so the wait gives up after
 * limit_us microseconds (1 .. 100000), records the timeout with site
 * DEC_SITE_SELFTEST and returns.  The next dec_check returns DEC_ETIMEOUT naming
 * that site, clears the error and resets the handle's barrier counters, after which
 * the handle decodes normally.  Errors: DEC_EINVAL (NULL handle, limit out of
 * range), DEC_ECUDA (launch failure). */
dec_status dec_selftest_wait_timeout(dec_handle *h, int32_t limit_us);

/* Kernel classes for dec_timing_enable. */
typedef enum dec_kernel_class {
  DEC_K_NONE = 0,
  DEC_K_QKV = 1,      /* decode: RMSNorm -> QKV GEMV -> RoPE -> KV write */
  DEC_K_ATTN = 2,     /* decode: split-K flash-decode attention */
  DEC_K_OPROJ = 3,    /* decode: output projection + residual */
  DEC_K_GATEUP = 4,   /* decode: RMSNorm -> gate/up GEMV -> silu(g)*u (dense or experts) */
  DEC_K_DOWN = 5,     /* decode: down projection (+ expert combine) + residual */
  DEC_K_LMHEAD = 6,   /* decode/prefill: final RMSNorm -> LM head (+ argmax) */
  DEC_K_ROUTER = 7,   /* decode: MoE router + top-k */
  DEC_K_PF_GEMM = 8,  /* prefill: projection GEMMs */
  DEC_K_PF_ATTN = 9,  /* prefill: causal attention */
  DEC_K_STEP = 10     /* decode: the whole step as one persistent kernel */
} dec_kernel_class;

/* Measurement hook: from the next call on, a CUDA event pair is recorded on
 * the handle's stream around each launch of kernel_class (at most
 * max_launches per call; the decode graph is re-captured to include them).
 * kernel_class 0 turns it off.  The library creates and owns the events. */
dec_status dec_timing_enable(dec_handle *h, int32_t kernel_class, int32_t max_launches);

/* Waits for the most recent call's events and returns the summed duration in
 * milliseconds and the number of timed launches of that call. */
dec_status dec_timing_read(dec_handle *h, float *total_ms, int32_t *launches);

/* Standalone attention of one query position over a KV ring: the split-K
 * flash-decode kernel of the decode step (rml "The decoder", Attend: one-pass
 * online softmax; Pantheon "Llama Forward Pass", Grouped Query Attention and
 * Sliding Window).  Query head h reads kv head h*n_kv_heads/n_heads over the
 * readable slots: min(pos+1, max_seq) under a window, else pos+1 (pos < max_seq).
 * A ring shorter than the window (max_seq < sliding_window) takes pos < max_seq only.
 *   q:   device [n_heads][head_dim] f32, already rotated.
 *   k,v: device rings [max_seq][n_kv_heads][head_dim] of kv_dtype.
 *   out: device [n_heads][head_dim] f32.
 *   scratch: device, >= dec_attend_scratch_bytes(...) bytes, 256-byte aligned,
 *   caller-owned; overwritten by the call.
 * Enqueued on cuda_stream.  Errors (host-side, before any launch): DEC_EINVAL,
 * DEC_ENOMEM (scratch too small), DEC_ECUDA.  Messages via dec_last_error(NULL). */
size_t dec_attend_scratch_bytes(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_seq);
dec_status dec_attend(const float *q, const void *k, const void *v, int32_t n_heads, int32_t n_kv_heads,
                      int32_t head_dim, int32_t max_seq, int32_t sliding_window, int32_t kv_dtype,
                      int32_t pos, float *out, void *scratch, size_t scratch_bytes, void *cuda_stream);

/* C = (A_hi + A_lo) . B^T on the tensor cores: the projection GEMM of the
 * prefill path (tcgen05, TMA, f32 accumulation in TMEM), callable alone.
 *   a_hi, a_lo: device [m][k] bf16 (a_lo may be NULL: A = A_hi); the pair
 *   carries an f32 activation as hi + lo.  b: device [n][k] bf16 (weights,
 *   row-major [out, in]).  c: device [m][n] f32.  k a multiple of 8, n even,
 *   operands 16-byte aligned.  Enqueued on cuda_stream.
 * Errors: DEC_EINVAL, DEC_ECUDA (messages via dec_last_error(NULL)). */
dec_status dec_gemm_bf16(const void *a_hi, const void *a_lo, const void *b, float *c, int32_t m, int32_t n,
                         int32_t k, void *cuda_stream);

/* dec_attend for callers that cannot allocate device memory (a plug-in whose
 * host framework's pooled allocator already owns the GPU's memory, or a
 * latency-critical path where cudaMalloc may not be called).  The pages have
 * no counterpart: this is an addition of this library.  Arguments and result
 * are those of dec_attend, without scratch: the scratch is a fixed 1 MiB array
 * in device memory inside libdec.so, held by every GPU that loads the library
 * until the process exits.  The call allocates nothing.
 *   - Sizes whose scratch exceeds 1 MiB (dec_attend_scratch_bytes() > 1 MiB)
 *     are rejected with DEC_EINVAL and a message.
 *   - The first call on a device looks up the array's device address on the
 *     current device (once per device and context: after cudaDeviceReset the
 *     next call looks it up again); make that first call before any stream
 *     capture.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and give undefined results.  The call
 *     resets what must start at zero itself. */
dec_status dec_attend_noalloc(const float *q, const void *k, const void *v, int32_t n_heads,
                              int32_t n_kv_heads, int32_t head_dim, int32_t max_seq,
                              int32_t sliding_window, int32_t kv_dtype, int32_t pos, float *out,
                              void *cuda_stream);

/* The 8-bit weight quantiser of weight_quant = 1, callable alone: w (device,
 * [rows][cols] of weight_dtype DEC_F32 or DEC_BF16, row-major) -> codes (device
 * int8 [rows][cols]) and scales (device f32 [rows][cols / 32]); cols a multiple
 * of 32.  Enqueued on cuda_stream.  Errors: DEC_EINVAL, DEC_ECUDA (messages via
 * dec_last_error(NULL)). */
dec_status dec_weight_quantize_int8(const void *w, int32_t weight_dtype, int64_t rows, int32_t cols, int8_t *codes,
                                    float *scales, void *cuda_stream);

/* The int8 K/V quantiser of the cache, callable alone: rows x (device,
 * [n_rows][n_kv_heads * head_dim] f32) -> out (device, n_rows rows of the
 * DEC_I8 row format: scales then codes, see dec_dtype).  head_dim a multiple
 * of 16, n_rows <= 65535.  Enqueued on cuda_stream.  Errors: DEC_EINVAL,
 * DEC_ECUDA (messages via dec_last_error(NULL)). */
dec_status dec_kv_quantize_int8(const float *x, int32_t n_rows, int32_t n_kv_heads, int32_t head_dim, void *out,
                                void *cuda_stream);

void dec_destroy(dec_handle *h);

/* Message of the last error on h (or of the last failed dec_create when h is NULL). */
const char *dec_last_error(const dec_handle *h);

#ifdef __cplusplus
}
#endif
#endif /* DEC_H */
