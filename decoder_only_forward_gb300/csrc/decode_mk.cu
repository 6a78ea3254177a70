// Persistent decode step: the whole one-token forward pass (every layer and
// the LM head) as ONE cooperative kernel with grid-wide barriers between its
// phases, so a step costs one launch instead of ~5 per layer.
//
// Roles inside each CTA (one CTA per SM):
//   warps 0-7  compute: phase prologues (RMSNorm, split merge), the dot
//              products of this CTA's weight rows, epilogues, attention tasks;
//   warps 8-15 producers: warp 8+w (one lane) feeds compute warp w.  Each walks the same
//              phase schedule and streams the rows its warp will reduce, in
//              pieces of up to 4 KB, into that warp's 4-stage shared-memory
//              ring with cp.async.bulk (TMA bulk copies, mbarrier completion).
//              It runs ahead across phases and grid barriers, so the HBM
//              weight stream does not wait for a barrier, and the compute
//              warps never synchronise with each other inside a GEMV phase.
//
// Phases per layer (Pantheon "Llama Forward Pass", Forward Pass Flow):
//   QKV    RMSNorm -> [q;k;v] rows (+bias) -> adjacent-pair RoPE -> K/V at the slot of pos
//   ATTN   (kv head, slot range) tasks: one-pass online softmax (rml Attend), partials per split
//  [MERGE] large split sets merged once per query head
//   OPROJ  split merge (small sets) -> x += Wo o
//   GATEUP RMSNorm -> silu(gate) * up (dense), or router -> top-k -> renormalise (MoE)
//   DOWN   x += Wd act (MoE: selected experts in selection order)
// or, with the fused FFN (bf16 weights, hidden % 128 == 0, ffn % 16 == 0):
//   FFN    RMSNorm [-> router] -> each CTA's (slot, ffn) slice: silu(gate) * up, then
//          that slice's rows of the transposed Wd into a partial sum over hidden
//   SUM    x += the CTAs' partials, summed in CTA order
// then LMHEAD: final RMSNorm -> logits + argmax.  Cross-CTA data (x, q,
// partials, act) is read with ld.global.cg so no stale L1 line is used.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "runtime.h"
#include "tc.cuh"

namespace dec {

constexpr int MK_COMPUTE_WARPS = 8;
constexpr int MK_COMPUTE = MK_COMPUTE_WARPS * 32;   // 256 compute threads
constexpr int MK_THREADS = 2 * MK_COMPUTE;          // + one producer warp per compute warp
constexpr int MK_REGS = 128;                         // registers per thread at launch (65536 / MK_THREADS)
constexpr int MK_REGS_PRODUCER = 64, MK_REGS_COMPUTE = 192;   // after the split (multiples of 8)
static_assert(MK_COMPUTE * MK_REGS_PRODUCER + MK_COMPUTE * MK_REGS_COMPUTE == MK_THREADS * MK_REGS,
              "the split hands out exactly the launch's registers");
constexpr int MK_WARP_RING = 16 * 1024;            // weight ring of one compute warp
constexpr int MK_RING_BYTES = MK_COMPUTE_WARPS * MK_WARP_RING;  // 128 KB
constexpr int MK_MAX_STAGES = 8;
constexpr int MK_KS = 64;                           // keys per attention chunk

// Weight-ring stages by weight type.  bf16 weights: tensor-core GEMV, a stage
// is 16 rows x MK_KG columns as MK_BPS TMA boxes of 64 columns side by side
// (128-byte swizzled), so each weight row is fetched in runs of MK_KG * 2
// bytes (DRAM page locality).  f32
// weights: CUDA-core GEMV, a stage is up to 4 KB of whole rows or one piece
// of a longer row.
template <typename W> struct MkRing;
template <> struct MkRing<float> {
  static constexpr int STAGES = 4, BYTES = 4096;
  static constexpr bool MMA = false, Q8 = false;
};
#ifndef MK_BPS
#define MK_BPS 2   // 64-column boxes per stage of the tensor-core GEMV
#endif
constexpr int MK_TM = 16, MK_TK = 64;               // one TMA box: rows x columns (2 KB bf16)
constexpr int MK_KG = MK_TK * MK_BPS;               // columns per stage: each row read in runs of 2^7 * MK_BPS B
template <> struct MkRing<__nv_bfloat16> {
  static constexpr int STAGES = 8 / MK_BPS, BYTES = 2048 * MK_BPS;
  static constexpr bool MMA = true, Q8 = false;
};
// 8-bit projections (weight_quant = 1): a stage is 16 rows x MK_QKG int8 codes as
// two 128-byte swizzled TMA boxes of 128 columns (each row read in 256-byte runs,
// as on the bf16 path) followed by the rows' f32 scales (16 x 8 groups of 32
// columns, 512 bytes); three stages per warp.  Embeddings, the router and a tied
// head stay bf16.
struct WQ8 {};
constexpr int MK_QKG = 256;                         // int8 columns per stage
constexpr int MK_QSC = 4096;                        // offset of a stage's scales
constexpr int MK_QSTAGE = MK_QSC + 16 * (MK_QKG / 32) * 4;   // bytes a stage receives (4608)
template <> struct MkRing<WQ8> {
  // Slots 1024-byte aligned (the swizzled boxes' alignment): 5 KB each.
  static constexpr int STAGES = 3, BYTES = 5120;
  static constexpr bool MMA = true, Q8 = true;
};
// int8 K/V cache (rml "The decoder", KV cache): a ring row is [group scales of
// every kv head, f32][codes, int8]; a group is 32 channels of one head.
struct KVI8 {};
constexpr int MK_I8_RPP = 8;    // keys per attention piece (one TMA box of codes, one of scales; 8 measured faster than 16)
template <typename KV> constexpr bool kMkKvI8 = false;
template <> constexpr bool kMkKvI8<KVI8> = true;

// Element type of the weights that are never quantised (embeddings, router, a tied head).
template <typename W> struct MkElem { using T = W; };
template <> struct MkElem<WQ8> { using T = __nv_bfloat16; };
// Activation planes are zero-padded to whole stages of either path.
constexpr int MK_PADK = 256;
constexpr int MK_CHUNK = 8;                         // row blocks reduced together (partials in smem)
constexpr int MK_MAX_LAYERS = 128;                  // layers of the persistent step (its parameter block)
// Fused FFN: a CTA owns a contiguous range of ffn tasks (slot, ffn index), a
// multiple of MK_FTS of them and at most MK_FT.
constexpr int MK_FTS = 16, MK_FT = 256;
// Tensor maps per layer (bf16 weights): QKV, O, gate/up, down, and the K and V
// rings (3D: head_dim x kv heads x slots, one box = one attention piece); then the head.
enum MkMap { MAP_QKV = 0, MAP_O, MAP_GATEUP, MAP_DOWN, MAP_K, MAP_V,
             MAP_QKV_S, MAP_O_S, MAP_GATEUP_S, MAP_DOWN_S, MAP_DOWN_T, MAP_KS, MAP_VS, MAPS_PER_LAYER };
constexpr int MAP_SCALE_OFF = MAP_QKV_S - MAP_QKV;   // a projection's scale map, 8-bit weights
// After the layers: the head, then (8-bit untied head) its scales.

enum MkPhase { PH_QKV = 0, PH_ATTN, PH_MERGE, PH_OPROJ, PH_GATEUP, PH_DOWN, PH_LMHEAD };

struct MkParams {
  int n_layers, h, nq, nkv, hd, f, V, E, k, max_seq, sliding, nsplit, sps, merge_phase, nb;
  float eps;
  // The layer table in the kernel's parameters: read through the constant cache,
  // so a phase's first use of a layer pointer needs no global load (from a
  // global-memory table, the attention phase's first K/V row address waited on
  // one L2 round trip before its own load could start).
  MkLayer layers[MK_MAX_LAYERS];
  const void* embed;
  const float* out_norm;
  const void* head;
  DeviceState* st;
  const double* inv_freq;
  const double* inv_freq_local;   // per-layer RoPE base: the local layers' frequencies (nullable)
  float* x;
  float* q;
  float* attn;
  float* act;                     // [k][f]
  float* part;
  float* amax_val;
  int32_t* amax_idx;
  int32_t* ids_out;               // [k] selected experts of the last MoE layer (for inspection)
  float* logits;
  int32_t* d_argmax;
  const int32_t* d_token;
  int token, pos;
  int32_t* trace_ids;
  float* trace_logits;
  int trace_cap;
  int u_bytes;                    // bytes of the shared region after the weight ring
  unsigned long long* stamps;     // nullable: %globaltimer after each phase (CTA 0), [0] = start
  int kv_bytes;                   // bytes per KV element
  int cluster;                    // > 0: the grid is ONE thread-block cluster of this many CTAs
  const CUtensorMap* maps;        // bf16 weights: [n_layers * MAPS_PER_LAYER + 1] (global memory)
  int xb_plane;                   // bf16 weights: elements per plane of the (hi, lo) activation copy
  int xs_floats;                  // floats of the f32 activation vector region
  int attn_warp;                  // attention as per-warp tasks fed by the producer rings
  int attn_ns;                    // warp-task attention: target splits per kv head (<= 32)
  int head_q8;                    // 8-bit weights: the LM head is quantised too (untied)
  int ffn_fused;                  // FFN as one phase over ffn slices + a partial-sum phase (below)
  float* fpart;                   // fused FFN: [nb][h] per-CTA partial sums of the down projection
  float* kv_cur;                  // int8 cache: [2][nkv*hd] this position's K and V rows in f32
  int kv_code_off;                // int8 cache: byte offset of a row's codes (after its scales)
  int kv_row_bytes;               // int8 cache: bytes of one ring row
  int qkn;                        // per-head QK-norm: q and the current k are normalised and rotated in ATTN
};

// The weight rows one CTA handles in one phase: up to k contiguous segments
// (one per selected expert).  Producer and consumers both derive it, so they
// agree stage by stage.  On the tensor-core path every CTA's share is a
// multiple of 16 rows (the MMA's M), so no CTA reads rows another one owns.
struct MkSeg {
  const uint8_t* base;   // row 0 of the segment's matrix
  int row0, rows;        // rows [row0, row0 + rows)
  int out0;              // output index of the segment's first row (task space)
  int slot;              // expert slot (MoE), else 0
  int map;               // tensor map of the matrix (bf16 weights)
  int maprow;            // row of the map holding the segment's row row0
};
struct MkRows {
  int nseg;
  MkSeg seg[MAX_EXPERTS_USED];
  int K;                 // row length (elements)
  int rowbytes;
  int rps;               // rows per stage (CUDA-core path)
  bool paired;
};

// Shared-memory bookkeeping after the weight ring and the union region.
struct MkMisc {
  uint64_t full[MK_COMPUTE_WARPS][MK_MAX_STAGES];
  uint64_t empty[MK_COMPUTE_WARPS][MK_MAX_STAGES];
  float part[MK_CHUNK][MK_COMPUTE_WARPS][MK_TM];  // tensor-core GEMV: per-warp row partials
  float2 cs[128];                // (cos, sin) of this position's rotary pairs; [64..]: the local base's
  float red[40];
  float logits[MAX_EXPERTS];
  int ids[MAX_EXPERTS_USED];
  float wts[MAX_EXPERTS_USED];
  float acc[256];                // MoE down: per-row sums over the selected experts
  float wbest[MK_COMPUTE_WARPS];
  int wbidx[MK_COMPUTE_WARPS];
  int token;
  int abort_flag;
  uint64_t moe_bar;              // completes once per MoE layer when its expert ids are in ids[]
  int consumed[MK_COMPUTE_WARPS];  // stages each warp consumed (for the abort drain)
  int is_last;
  float mrow[MAX_GROUP], lrow[MAX_GROUP], alpha[MAX_GROUP];
  float mscale[8 * 32];          // warp-task attention merge: weight of split s for query head h
  int lastg[MK_COMPUTE_WARPS];   // kv heads whose last split this CTA finished in the current round
  float fact[MK_FT];             // fused FFN: this CTA's SwiGLU outputs (router-weighted)
  // Each warp's row plan of its current phase (compute warps, then producers), in
  // shared memory: as a local array it lived in local memory that the 28 KB L1 beside
  // this kernel's shared memory could not keep, so reading a phase's segments cost a
  // round trip to L2.
  MkRows rows[2 * MK_COMPUTE_WARPS];
  __nv_bfloat16 fxb[2][MK_FT];   // fused FFN: the same as bf16 (hi, lo) planes
  uint64_t cbar;                 // cluster mode: phase barrier, one arrival per CTA of the cluster
  unsigned cgen;                 // cluster mode: barrier instances completed
};

// ------------------------------------------------------------------ sync
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(MK_COMPUTE) : "memory"); }

__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of the compute groups of all CTAs (bounded wait), on a
// 64-bit arrival counter that only grows: barrier instance k of a launch is
// passed once the counter reaches base + k * nb, base being the counter's value
// when the launch began (a multiple of nb: every earlier launch added nb per
// barrier, and a CTA reads it before its own first arrival, when fewer than nb
// arrivals of this launch can have happened).  Arrival is one release
// reduction after the CTA's bar.sync (the CTA's writes are released with it),
// the wait an acquire poll; no read-modify-write round trip and no separate
// generation word.
__device__ __forceinline__ unsigned long long* mk_bar_counter(DeviceState* st) {
  static_assert(offsetof(DeviceState, counters) % 8 == 0 && CNT_MK_GEN == CNT_MK_BAR + 1 && CNT_MK_BAR % 2 == 0,
                "the barrier counter is one aligned 64-bit word");
  return reinterpret_cast<unsigned long long*>(&st->counters[CNT_MK_BAR]);
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool mk_grid_sync(DeviceState* st, unsigned long long target, volatile int* abort_flag,
                                             unsigned site, uint64_t limit_ns = WAIT_LIMIT_NS) {
  compute_sync();
  if (threadIdx.x == 0 && !*abort_flag) {
    unsigned long long* cnt = mk_bar_counter(st);
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(cnt) : "memory");
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_u64(cnt) < target) {
      if (globaltimer_ns() - t0 > limit_ns) {
        raise_error(st, ERR_TIMEOUT, site);
        *abort_flag = 1;
        break;
      }
    }
  }
  compute_sync();
  return !*abort_flag;
}

// Cluster mode: the same phase barrier over the CTAs of one cluster.  Each
// CTA's thread 0 arrives (release, cluster scope) on the barrier in every
// CTA's shared memory, then waits (acquire, cluster scope) for the arrivals
// of all CTAs on its own.  A CTA can be at most one instance ahead of any
// other, so the parity of the instance count names the phase to wait for.
__device__ __forceinline__ bool mk_cluster_sync(DeviceState* st, unsigned nb, uint64_t* cbar, unsigned* cgen,
                                                volatile int* abort_flag, unsigned site) {
  compute_sync();
  if (threadIdx.x == 0 && !*abort_flag) {
    const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(cbar));
    for (unsigned r = 0; r < nb; ++r) {
      uint32_t ra;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(r));
      asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
    }
    const uint32_t parity = *cgen & 1u;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(la), "r"(parity)
          : "memory");
      if (ok) break;
      if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        raise_error(st, ERR_TIMEOUT, site);
        *abort_flag = 1;
        break;
      }
    }
    ++*cgen;
  }
  compute_sync();
  return !*abort_flag;
}

// ------------------------------------------------------------------ mbarrier / bulk copy
__device__ __forceinline__ uint32_t mk_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mk_mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mk_smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mk_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mk_smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mk_mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mk_smem_u32(bar)), "r"(bytes)
               : "memory");
}
// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes (or about 20 us pass) instead of spinning.
__device__ __forceinline__ bool mk_mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(mk_smem_u32(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}
// Bounded wait; gives up when another role has given up.
__device__ __forceinline__ bool mk_mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             DeviceState* st, unsigned site) {
  if (mk_mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mk_mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      raise_error(st, ERR_TIMEOUT, site);
      *abort_flag = 1;
      return false;
    }
  }
}
// Asks L2 to fetch `bytes` (multiple of 16) from global memory ahead of use.
__device__ __forceinline__ void mk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The same for any pointer and size: the whole 16-byte units of a 16-byte aligned range, else nothing.
__device__ __forceinline__ void mk_prefetch_l2_any(const void* src, uint32_t bytes) {
  if (src && ((uintptr_t)src & 15u) == 0 && (bytes & ~15u) != 0) mk_prefetch_l2(src, bytes & ~15u);
}

// Contiguous global -> shared copy of `bytes` (multiple of 16, 16-byte aligned).
__device__ __forceinline__ void mk_bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   mk_smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(mk_smem_u32(bar))
               : "memory");
}

}  // namespace dec

namespace dec {

// ------------------------------------------------------------------ schedule

__device__ __forceinline__ bool mk_is_gemv(const MkParams& P, int ph) {
  return ph != PH_ATTN && ph != PH_MERGE && !(ph == PH_DOWN && P.ffn_fused);
}

// ceil(n / nb) rounded up to a multiple of g.
__device__ __forceinline__ int mk_share(int n, int nb, int g) { return ((n + nb - 1) / nb + g - 1) / g * g; }

template <typename W>
__device__ void mk_phase_rows(const MkParams& P, int ph, int l, const int* ids, MkRows& R) {
  const int es = (int)sizeof(typename MkElem<W>::T);
  const int b = blockIdx.x, nb = P.nb;
  const MkLayer& L = P.layers[l < P.n_layers ? l : 0];
  const int qd = P.nq * P.hd, kd = P.nkv * P.hd;
  const int g = MkRing<W>::MMA ? MK_TM : 1;     // row granularity of a CTA's share
  const int mbase = (l < P.n_layers ? l : 0) * MAPS_PER_LAYER;
  R.nseg = 0;
  auto single = [&](const void* mat, int N, int K, int map) {
    const int per = mk_share(N, nb, g);
    const int r0 = min(N, b * per), r1 = min(N, r0 + per);
    R.K = K;
    R.paired = false;
    if (r1 > r0) R.seg[R.nseg++] = MkSeg{(const uint8_t*)mat, r0, r1 - r0, r0, 0, map, r0};
  };
  auto paired = [&](const void* mat, int N, int K, int map) {
    const int P2 = N / 2, per = mk_share(P2, nb, (g + 1) / 2);
    const int p0 = min(P2, b * per), p1 = min(P2, p0 + per);
    R.K = K;
    R.paired = true;
    if (p1 > p0) R.seg[R.nseg++] = MkSeg{(const uint8_t*)mat, 2 * p0, 2 * (p1 - p0), 2 * p0, 0, map, 2 * p0};
  };
  switch (ph) {
    case PH_QKV: paired(L.wqkv, qd + 2 * kd, P.h, mbase + MAP_QKV); break;
    case PH_OPROJ: single(L.wo, P.h, qd, mbase + MAP_O); break;
    case PH_LMHEAD: single(P.head, P.V, P.h, P.n_layers * MAPS_PER_LAYER); break;
    case PH_GATEUP:
      if (P.E == 0 && !P.ffn_fused) {
        paired(L.w_gateup, 2 * P.f, P.h, mbase + MAP_GATEUP);
      } else {
        // Tasks = (slot, gate/up row pair), slot-major, split evenly over CTAs.
        // Fused FFN: shares of MK_FTS tasks, and out0 = the segment's first task
        // within the CTA's own range.
        const int T = P.k * P.f, per = mk_share(T, nb, P.ffn_fused ? MK_FTS : (g + 1) / 2);
        const int t0 = min(T, b * per), t1 = min(T, t0 + per);
        R.K = P.h;
        R.paired = true;
        for (int j = 0; j < P.k; ++j) {
          const int a = max(t0, j * P.f), e = min(t1, (j + 1) * P.f);
          if (e <= a) continue;
          const int eid = P.E > 0 ? ids[j] : 0;
          const uint8_t* base = (const uint8_t*)L.w_gateup + (size_t)eid * 2 * P.f * P.h * es;
          const int r0 = 2 * (a - j * P.f);
          R.seg[R.nseg++] =
              MkSeg{base, r0, 2 * (e - a), P.ffn_fused ? a - t0 : a, j, mbase + MAP_GATEUP, eid * 2 * P.f + r0};
        }
      }
      break;
    case PH_DOWN:
      if (P.E == 0) {
        single(L.w_down, P.h, P.f, mbase + MAP_DOWN);
      } else {
        const int per = mk_share(P.h, nb, g);
        const int r0 = min(P.h, b * per), r1 = min(P.h, r0 + per);
        R.K = P.f;
        R.paired = false;
        if (r1 > r0)
          for (int j = 0; j < P.k; ++j) {
            const uint8_t* base = (const uint8_t*)L.w_down + (size_t)ids[j] * P.h * P.f * es;
            R.seg[R.nseg++] = MkSeg{base, r0, r1 - r0, r0, j, mbase + MAP_DOWN, ids[j] * P.h + r0};
          }
      }
      break;
    default: break;
  }
  R.rowbytes = R.K * es;
  int rps = MkRing<W>::BYTES / R.rowbytes;
  if (R.paired) rps &= ~1;
  R.rps = rps < 1 ? 1 : rps;
}

// The phase sequence of one step: per layer QKV, ATTN, [MERGE], OPROJ, GATEUP,
// DOWN; then LMHEAD.  Index i -> (phase, layer).
__device__ __forceinline__ int mk_phases_per_layer(const MkParams& P) { return P.merge_phase ? 6 : 5; }
__device__ __forceinline__ void mk_phase_at(const MkParams& P, int i, int& ph, int& l) {
  const int ppl = mk_phases_per_layer(P);
  l = i / ppl;
  if (l >= P.n_layers) {
    ph = PH_LMHEAD;
    return;
  }
  int j = i - l * ppl;
  if (!P.merge_phase && j >= PH_MERGE) ++j;
  ph = j;
}

// ------------------------------------------------------------------ dot products
// This warp's share of one row's dot product: chunks c = 32*(warp + 8i) + lane
// of the 16-byte chunks, so the 8 compute warps split every row's K.
template <typename W>
__device__ __forceinline__ float mk_dot_slice(const uint8_t* row, const float* xs, int K) {
  constexpr int V = Chunk<W>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float a = 0.f;
  for (int c = 32 * warp + lane; c < K / V; c += MK_COMPUTE) {
    float w[V];
    Chunk<W>::widen(*reinterpret_cast<const uint4*>(row + (size_t)c * 16), w);
    const float* xv = xs + c * V;
#pragma unroll
    for (int e = 0; e < V; ++e) a = fmaf(w[e], xv[e], a);
  }
  return warp_sum(a);
}

// Dot of one weight row in shared memory with the f32 vector xs (also in
// shared memory), one warp; K * sizeof(W) is a multiple of 16 bytes.
template <typename W>
__device__ __forceinline__ float mk_dot_row(const uint8_t* row, const float* xs, int K) {
  constexpr int V = Chunk<W>::N;
  const int lane = threadIdx.x & 31;
  float a = 0.f;
  for (int c = lane; c < K / V; c += 32) {
    float w[V];
    Chunk<W>::widen(*reinterpret_cast<const uint4*>(row + (size_t)c * 16), w);
    const float* xv = xs + c * V;
#pragma unroll
    for (int e = 0; e < V; ++e) a = fmaf(w[e], xv[e], a);
  }
  return warp_sum(a);
}

}  // namespace dec

namespace dec {

// ------------------------------------------------------------------ compute prologues
// dst[0..K) = src[0..K): global f32 written by other CTAs, fetched with 16-byte
// asynchronous copies through L2, all in flight at once (src, dst 16-byte
// aligned).
__device__ void mk_fetch(const float* src, int K, float* dst) {
  const int nv = K >> 2;
  for (int i = threadIdx.x; i < nv; i += MK_COMPUTE) cp_async16(dst + 4 * i, src + 4 * i);
  cp_async_commit();
  for (int k = 4 * nv + threadIdx.x; k < K; k += MK_COMPUTE) dst[k] = __ldcg(src + k);
  cp_async_wait_all();
  compute_sync();
}

// Element k of the activation as a bf16 (hi, lo) pair: the B operand of the
// tensor-core GEMV (x = hi + lo to ~16 bits).
// With f16 (8-bit weight phases) the pair is two halves instead: hi = f16(v),
// lo = f16(v - hi), about 22 bits for |v| >= 2^-3 and an absolute error below
// 2^-25 below that.
__device__ __forceinline__ void mk_put_xb(__nv_bfloat16* xb, int plane, int k, float v, bool f16 = false) {
  if (f16) {
    __half* xh = reinterpret_cast<__half*>(xb);
    const __half hi = __float2half_rn(v);
    xh[k] = hi;
    xh[plane + k] = __float2half_rn(v - __half2float(hi));
    return;
  }
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  xb[k] = hi;
  xb[plane + k] = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// xs = v / sqrt(mean(v^2) + eps) * wn over the 256 compute threads, with v the
// embedding row (erow) or the residual x (fetched from L2).  With xb, the
// result also goes to the bf16 (hi, lo) planes, zero-padded to kpad columns.
template <typename W>
__device__ void mk_norm_to_xs(const float* x, const W* erow, const float* __restrict__ wn, int K, float eps,
                              float* xs, MkMisc* M, __nv_bfloat16* xb = nullptr, int plane = 0, int kpad = 0,
                              bool f16 = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (erow) {
    for (int k = tid; k < K; k += MK_COMPUTE) xs[k] = to_f32(erow[k]);
    compute_sync();
  } else {
    mk_fetch(x, K, xs);
  }
  float ss = 0.f;
  for (int k = tid; k < K; k += MK_COMPUTE) ss = fmaf(xs[k], xs[k], ss);
  ss = warp_sum(ss);
  if (lane == 0) M->red[warp] = ss;
  compute_sync();
  if (warp == 0) {
    float v = lane < MK_COMPUTE_WARPS ? M->red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) M->red[32] = v;
  }
  compute_sync();
  const float inv = 1.0f / sqrtf(M->red[32] / (float)K + eps);
  const int kend = xb && kpad > K ? kpad : K;
  // Norm weights four at a time, their loads issued before any use.
  for (int k0 = tid; k0 < kend; k0 += 4 * MK_COMPUTE) {
    float wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * MK_COMPUTE;
      wv[u] = k < K ? wn[k] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * MK_COMPUTE;
      if (k >= kend) break;
      const float v = k < K ? xs[k] * inv * wv[u] : 0.f;
      if (k < K) xs[k] = v;
      if (xb) mk_put_xb(xb, plane, k, v, f16);
    }
  }
  compute_sync();
}

__device__ void mk_copy_to_xs(const float* src, int K, float* xs) { mk_fetch(src, K, xs); }

// Merges split partials of `heads` query heads [h0, h0+heads) into dst
// (dst[(h - h0) * HD + d]); scale is [heads][nsplit] scratch.  Weight of split
// s: exp(m_s - M) / sum_s l_s exp(m_s - M) (one-pass softmax state, rml Attend).
__device__ void mk_merge_heads(const float* part, int nsplit, int HD, int h0, int heads, float* scale, float* dst,
                               bool dst_global) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int hh = warp; hh < heads; hh += MK_COMPUTE_WARPS) {
    const float* base = part + (size_t)(h0 + hh) * nsplit * (HD + 2);
    float mloc = -INFINITY;
    for (int s2 = lane; s2 < nsplit; s2 += 32) mloc = fmaxf(mloc, __ldcg(base + s2 * (HD + 2) + HD));
    const float Mx = warp_max(mloc);
    float lsum = 0.f;
    for (int s2 = lane; s2 < nsplit; s2 += 32) {
      const float ms = __ldcg(base + s2 * (HD + 2) + HD);
      const float sc = ms == -INFINITY ? 0.f : __expf(ms - Mx);
      scale[hh * nsplit + s2] = sc;
      lsum = fmaf(__ldcg(base + s2 * (HD + 2) + HD + 1), sc, lsum);
    }
    const float Ls = warp_sum(lsum);
    __syncwarp();
    for (int s2 = lane; s2 < nsplit; s2 += 32) scale[hh * nsplit + s2] /= Ls;
  }
  compute_sync();
  for (int idx = tid; idx < heads * HD; idx += MK_COMPUTE) {
    const int hh = idx / HD, d = idx - hh * HD;
    const float* base = part + (size_t)(h0 + hh) * nsplit * (HD + 2) + d;
    const float* sc = scale + hh * nsplit;
    float o = 0.f;
#pragma unroll 8
    for (int s2 = 0; s2 < nsplit; ++s2) o = fmaf(sc[s2], __ldcg(base + (size_t)s2 * (HD + 2)), o);
    if (dst_global) dst[(size_t)(h0 + hh) * HD + d] = o;
    else dst[idx] = o;
  }
  compute_sync();
}

// Router of one MoE layer, computed identically by every CTA: logits = Wr xs,
// top-k by repeated selection (ties -> lower id), weights renormalised over the
// selection (Pantheon Mixture of Experts; rml Mixture of experts).
template <typename W>
__device__ void mk_router(const MkParams& P, int l, const float* xs, MkMisc* M) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const W* router = (const W*)P.layers[l].router;
  constexpr int V = Chunk<W>::N;
  // One warp per expert row; each lane requests up to 16 of its 16-byte chunks
  // before the first product (same order of products as one chunk at a time).
  constexpr int RJ = 16;
  const int nc = P.h / V;
  for (int e = warp; e < P.E; e += MK_COMPUTE_WARPS) {
    const W* row = router + (size_t)e * P.h;
    float a = 0.f;
    for (int c0 = lane; c0 < nc; c0 += 32 * RJ) {
      uint4 u[RJ];
#pragma unroll
      for (int j = 0; j < RJ; ++j) {
        const int c = c0 + 32 * j;
        u[j] = c < nc ? ld_stream16(row + (size_t)c * V) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < RJ; ++j) {
        const int c = c0 + 32 * j;
        if (c < nc) {
          float wv[V];
          Chunk<W>::widen(u[j], wv);
#pragma unroll
          for (int q = 0; q < V; ++q) a = fmaf(wv[q], xs[c * V + q], a);
        }
      }
    }
    a = warp_sum(a);
    if (lane == 0) M->logits[e] = a;
  }
  compute_sync();
  if (warp == 0) {
    // Top-k by repeated selection, ties to the lower id (rml "The decoder",
    // Mixture of experts): lane l owns experts l, l + 32, ...; each round takes
    // the lanes' best untaken expert and the warp's best of those.  Lane j keeps
    // selection j.
    constexpr int NONE = 0x7fffffff;
    unsigned taken = 0u;
    int my_id = 0;
    float my_logit = 0.f;
    for (int j = 0; j < P.k; ++j) {
      float bv = -INFINITY;
      int bi = NONE;
      for (int i = 0, e = lane; e < P.E; ++i, e += 32) {
        if ((taken >> i) & 1u) continue;
        const float v = M->logits[e];
        if (bi == NONE || v > bv) {
          bv = v;
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (oi != NONE && (bi == NONE || ov > bv || (ov == bv && oi < bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_id = bi;
        my_logit = bv;
      }
    }
    // Softmax over the selected logits (the first selection is their maximum),
    // summed in selection order.
    const float mx = __shfl_sync(0xffffffffu, my_logit, 0);
    const float pj = lane < P.k ? expf(my_logit - mx) : 0.f;
    float tot = 0.f;
    for (int j = 0; j < P.k; ++j) tot += __shfl_sync(0xffffffffu, pj, j);
    const float wj = pj / tot;
    for (int j = 0; j < P.k; ++j) {
      const int idj = __shfl_sync(0xffffffffu, my_id, j);
      const float wtj = __shfl_sync(0xffffffffu, wj, j);
      if (lane == 0) {
        M->ids[j] = idj;
        M->wts[j] = wtj;
      }
    }
    if (blockIdx.x == 0) {
      if (lane < P.k) P.ids_out[lane] = my_id;
      if (P.trace_ids) {
        const size_t row = (size_t)l * P.trace_cap + (P.pos % P.trace_cap);
        if (lane < P.k) P.trace_ids[row * P.k + lane] = my_id;
        for (int e = lane; e < P.E; e += 32) P.trace_logits[row * P.E + e] = M->logits[e];
      }
    }
    // Releases this layer's expert rows to the producers (the arrival orders
    // lane 0's ids / wts writes before their wait returns).
    if (lane == 0) mk_mbar_arrive(&M->moe_bar);
  }
  compute_sync();
}

}  // namespace dec

namespace dec {

// ------------------------------------------------------------------ GEMV phase (consumer side)
constexpr int MK_RB = 4;   // rows reduced together per pass (CUDA-core path)

// V consecutive floats of the activation vector in shared memory (16-byte aligned).
template <int V>
__device__ __forceinline__ void mk_load_xs(const float* p, float* v) {
#pragma unroll
  for (int i = 0; i < V; i += 4) {
    const float4 t = *reinterpret_cast<const float4*>(p + i);
    v[i] = t.x;
    v[i + 1] = t.y;
    v[i + 2] = t.z;
    v[i + 3] = t.w;
  }
}

// Rows [r0, r1) of segment S (relative to S.row0) that warp w reduces on the
// CUDA-core path: a contiguous block of whole units (a unit is a row, or a
// row pair for the paired epilogues).  Rows of up to one stage are streamed
// several per stage, longer rows in stage-sized pieces; producer and consumer
// walk the same plan.
__device__ __forceinline__ void mk_warp_rows(const MkRows& R, const MkSeg& S, int w, int& r0, int& r1) {
  const int nrow = R.paired ? 2 : 1;
  const int units = S.rows / nrow;
  const int upw = (units + MK_COMPUTE_WARPS - 1) / MK_COMPUTE_WARPS;
  const int u0 = min(units, w * upw), u1 = min(units, u0 + upw);
  r0 = u0 * nrow;
  r1 = u1 * nrow;
}

// Tensor-core path: segment S is cut into 16-row blocks, taken MK_CHUNK at a
// time; inside a chunk, tile (b, kb) (local block b, MK_KG-column group kb) is
// number t = b * KB + kb and belongs to warp t % 8.  The first kb of local
// block b that warp w owns:
__device__ __forceinline__ int mk_first_kb(int b, int KB, int w) {
  return ((w - (b * KB) % MK_COMPUTE_WARPS) % MK_COMPUTE_WARPS + MK_COMPUTE_WARPS) % MK_COMPUTE_WARPS;
}

// Epilogue of a row pair (rl = even row relative to S.row0): QKV bias, RoPE and
// the q / K / V stores, or SwiGLU for gate/up.
template <typename KV>
__device__ __forceinline__ void mk_epi_pair(const MkParams& P, int ph, const MkLayer& L, const MkSeg& S,
                                            MkMisc* M, int rl, float a0, float a1) {
  const int qd = P.nq * P.hd, kd = P.nkv * P.hd;
  if (ph == PH_QKV) {
    const int row = S.row0 + rl;
    float v0 = a0, v1 = a1;
    if (L.bqkv) {
      v0 += L.bqkv[row];
      v1 += L.bqkv[row + 1];
    }
    if (row < qd + kd && !P.qkn) {   // (QK-norm: normalised before the rotation, in ATTN)
      const int d = (row < qd ? row : row - qd) % P.hd;
      const float2 cs = M->cs[(L.rope_local ? 64 : 0) + (d >> 1)];
      const float b0 = v0 * cs.x - v1 * cs.y, b1 = v0 * cs.y + v1 * cs.x;
      v0 = b0;
      v1 = b1;
    }
    const int slot = P.sliding > 0 ? P.pos % P.max_seq : P.pos;
    if (row < qd) {
      P.q[row] = v0;
      P.q[row + 1] = v1;
    } else if constexpr (kMkKvI8<KV>) {
      // int8 cache: the row is quantised per 32-channel group by the attention task
      // that holds this position (a group's rows are spread over several CTAs here).
      P.kv_cur[row - qd] = v0;
      P.kv_cur[row - qd + 1] = v1;
      (void)slot;
    } else if (P.qkn && row < qd + kd) {   // raw k, normalised and stored by ATTN
      P.kv_cur[row - qd] = v0;
      P.kv_cur[row - qd + 1] = v1;
    } else {
      const bool is_k = row < qd + kd;
      KV* dst = (KV*)(is_k ? L.kc : L.vc);
      const size_t o = (size_t)slot * kd + (is_k ? row - qd : row - qd - kd);
      dst[o] = from_f32<KV>(v0);
      dst[o + 1] = from_f32<KV>(v1);
    }
  } else if (P.ffn_fused) {   // PH_GATEUP, fused FFN: the CTA's own task slot, times the router weight
    M->fact[S.out0 + (rl >> 1)] = (P.E > 0 ? M->wts[S.slot] : 1.f) * (silu_f(a0) * a1);
  } else {  // PH_GATEUP: act[task] = silu(gate) * up
    const int task = P.E > 0 ? S.out0 + (rl >> 1) : (S.row0 + rl) >> 1;
    P.act[task] = silu_f(a0) * a1;
  }
}

// Epilogue of a single row: logits (+ running argmax), the MoE down row sum
// over the selected experts, or the residual increment of O / down.
__device__ __forceinline__ void mk_epi_row(const MkParams& P, int ph, const MkSeg& S, MkMisc* M, int rl, float a,
                                           float& bst, int& bix) {
  const int row = S.row0 + rl;
  if (ph == PH_LMHEAD) {
    if (P.logits) P.logits[row] = a;
    if (a > bst || (a == bst && row < bix)) {
      bst = a;
      bix = row;
    }
  } else if (ph == PH_DOWN && P.E > 0) {
    float& acc = M->acc[rl];
    acc = S.slot == 0 ? M->wts[0] * a : fmaf(M->wts[S.slot], a, acc);
  } else {  // PH_OPROJ, dense PH_DOWN: added to the residual row after the phase
    M->acc[rl] = a;
  }
}

// Four 8x8 b16 matrices from shared memory (lane l gives row l % 8 of matrix l / 8).
__device__ __forceinline__ void mk_ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// d (16x8 f32) += a (16x16 bf16, row) . b (16x8 bf16, col).
__device__ __forceinline__ void mk_mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four int8 codes (one 32-bit word, bytes = consecutive columns) -> two f16
// pairs, exactly: each code is biased by 128 and becomes the low byte of the
// half 1024 + (c + 128), two halves per byte permute, and one paired
// subtraction of 1152 leaves c exactly.
__device__ __forceinline__ void mk_q8_f16x2(uint32_t u, uint32_t& lo2, uint32_t& hi2) {
  const uint32_t v = u ^ 0x80808080u;
  const uint32_t bias = 0x64806480u;   // (1152, 1152) as halves
  const uint32_t p01 = __byte_perm(v, 0x64646464u, 0x4140), p23 = __byte_perm(v, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo2) : "r"(p01), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi2) : "r"(p23), "r"(bias));
}

// d (16x8 f32) += a (16x16 f16, row) . b (16x8 f16, col).
__device__ __forceinline__ void mk_mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One stage of 8-bit weights: 16 rows x MK_QKG codes (two 128-column boxes,
// 128-byte swizzled) and their scales.  Each 32-column group is reduced with two
// MMAs into its own accumulator, then scaled by the row's group scale: d[0] / d[2]
// collect rows grp / grp + 8 (lanes with t4 == 0 hold the activation's columns).
// Within a 16-column step lane t4 takes 4 consecutive codes as fragment columns
// (2t4, 2t4+1, 2t4+8, 2t4+9), and the activation's same 4 columns as B: the same
// permutation of k on both operands leaves the sum unchanged.
__device__ __forceinline__ void mk_q8_stage(const uint8_t* tile, int kb, int grp, int t4, bool bl,
                                            const __nv_bfloat16* xbl, float* d) {
  const uint32_t sbase = mk_smem_u32(tile);
  const float* sc = reinterpret_cast<const float*>(tile + MK_QSC);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t base = sbase + 2048u * j;
    const uint32_t sw0 = ((base >> 7) + (uint32_t)grp) & 7u, sw8 = ((base >> 7) + (uint32_t)grp + 8u) & 7u;
    const uint32_t r0 = base + (uint32_t)grp * 128u + 4u * (uint32_t)t4, r8 = r0 + 8u * 128u;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float dg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t ks = (uint32_t)(2 * g + hh);
        uint32_t u0, u8;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(u0) : "r"(r0 + ((ks ^ sw0) << 4)));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(u8) : "r"(r8 + ((ks ^ sw8) << 4)));
        uint32_t a0, a1, a2, a3;
        mk_q8_f16x2(u0, a0, a2);
        mk_q8_f16x2(u8, a1, a3);
        const int k0 = kb * MK_QKG + j * 128 + (int)ks * 16 + 4 * t4;
        const uint2 bv = bl ? *reinterpret_cast<const uint2*>(xbl + k0) : make_uint2(0u, 0u);   // f16 planes
        mk_mma_f16(dg, a0, a1, a2, a3, bv.x, bv.y);
      }
      const int gi = j * 4 + g;
      d[0] = fmaf(sc[grp * 8 + gi], dg[0] + dg[1], d[0]);
      d[2] = fmaf(sc[(grp + 8) * 8 + gi], dg[2] + dg[3], d[2]);
    }
  }
}

// Barrier 1 over the compute threads; returns whether any of them passed
// `pred`, so that every compute warp takes the same way out of a phase.
__device__ __forceinline__ bool compute_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(MK_COMPUTE)
      : "memory");
  return r != 0;
}

// The activation vector as bf16 (hi, lo) planes, zero-padded to whole column
// groups.  A global source (the FFN activation, K a multiple of 4) is read
// as float4, four loads in flight per thread.
__device__ void mk_to_xb(const float* src, bool src_global, int K, __nv_bfloat16* xb, int plane, bool f16 = false) {
  const int KP = (K + MK_PADK - 1) / MK_PADK * MK_PADK;
  if (src_global) {
    const int nv = K >> 2, np = KP >> 2;
    for (int i0 = threadIdx.x; i0 < np; i0 += 4 * MK_COMPUTE) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * MK_COMPUTE;
        v[u] = i < nv ? __ldcg(reinterpret_cast<const float4*>(src) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * MK_COMPUTE;
        if (i < np) {
          mk_put_xb(xb, plane, 4 * i, v[u].x, f16);
          mk_put_xb(xb, plane, 4 * i + 1, v[u].y, f16);
          mk_put_xb(xb, plane, 4 * i + 2, v[u].z, f16);
          mk_put_xb(xb, plane, 4 * i + 3, v[u].w, f16);
        }
      }
    }
  } else {
    for (int k = threadIdx.x; k < KP; k += MK_COMPUTE) mk_put_xb(xb, plane, k, k < K ? src[k] : 0.f, f16);
  }
  compute_sync();
}

// One GEMV phase on the compute side.  Every compute warp runs the same loop
// structure whatever happens to its waits (a warp whose wait gave up skips
// work, not loops), so all of them meet at every compute_sync.
template <typename W, typename KV>
__device__ bool mk_gemv_phase(const MkParams& P, int ph, int l, const MkRows& R, uint8_t* ring, MkMisc* M,
                              float* xs, uint32_t& sc, float& best, int& bidx) {
  constexpr int NS = MkRing<W>::STAGES, SB = MkRing<W>::BYTES;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const MkLayer& L = P.layers[l < P.n_layers ? l : 0];
  volatile int* abort_flag = &M->abort_flag;
  uint8_t* wring = ring + (size_t)warp * MK_WARP_RING;
  // Hot-loop state in registers (the by-reference arguments are written back
  // at the end).
  uint32_t scl = sc;
  float bst = best;
  int bix = bidx;
  DeviceState* const stp = P.st;
  bool ok = true;
  auto next_stage = [&]() -> const uint8_t* {
    const int st = scl % NS;
    const uint32_t par = (scl / NS) & 1u;
    if (!mk_mbar_wait(&M->full[warp][st], par, abort_flag, stp, 201)) return nullptr;
    return wring + (size_t)st * SB;
  };
  auto release_stage = [&]() {
    __syncwarp();
    const int st = scl % NS;
    if (lane == 0) mk_mbar_arrive(&M->empty[warp][st]);
    ++scl;
    if (lane == 0) M->consumed[warp] = (int)scl;
  };
  if constexpr (!MkRing<W>::MMA) {
    // ---------------- CUDA-core path (f32 weights)
    constexpr int V = Chunk<W>::N;
    const int cpr = R.rowbytes / 16;   // 16-byte chunks per row
    for (int si = 0; si < R.nseg; ++si) {
      const MkSeg S = R.seg[si];   // by value: its fields stay in registers
      if (ph == PH_DOWN && P.E > 0) {
        // Expert slot S.slot multiplies its own activation vector.
        compute_sync();
        mk_copy_to_xs(P.act + (size_t)S.slot * P.f, P.f, xs);
      }
      int r0, r1;
      mk_warp_rows(R, S, warp, r0, r1);
      float pend = 0.f;   // sum of the even row of a pair in progress
      auto finish = [&](int rl, float sum) {
        if (R.paired) {
          if ((rl & 1) == 0) {
            pend = sum;
            return;
          }
          if (lane == 0) mk_epi_pair<KV>(P, ph, L, S, M, rl - 1, pend, sum);
        } else if (lane == 0) {
          mk_epi_row(P, ph, S, M, rl, sum, bst, bix);
        }
      };
      if (R.rowbytes <= SB) {
        // Up to MK_RB rows of a stage per pass: each xs chunk is read once for
        // all of them, and their FMA chains and shuffle reductions interleave.
        const int rps = SB / R.rowbytes;
        for (int r = r0; r < r1 && ok; r += rps) {
          const int n = min(rps, r1 - r);
          const uint8_t* piece = next_stage();
          if (!piece) {
            ok = false;
            break;
          }
          for (int j0 = 0; j0 < n; j0 += MK_RB) {
            const int nj = min(MK_RB, n - j0);
            const uint8_t* rows = piece + (size_t)j0 * R.rowbytes;
            float acc[MK_RB];
#pragma unroll
            for (int j = 0; j < MK_RB; ++j) acc[j] = 0.f;
            for (int c = lane; c < cpr; c += 32) {
              float xv[V];
              mk_load_xs<V>(xs + c * V, xv);
#pragma unroll
              for (int j = 0; j < MK_RB; ++j) {
                if (j < nj) {
                  float wv[V];
                  Chunk<W>::widen(*reinterpret_cast<const uint4*>(rows + (size_t)j * R.rowbytes + (size_t)c * 16), wv);
#pragma unroll
                  for (int e = 0; e < V; ++e) acc[j] = fmaf(wv[e], xv[e], acc[j]);
                }
              }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
              for (int j = 0; j < MK_RB; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
            for (int j = 0; j < nj; ++j) finish(r + j0 + j, acc[j]);
          }
          release_stage();
        }
      } else {
        for (int r = r0; r < r1 && ok; ++r) {
          float acc0 = 0.f, acc1 = 0.f;
          for (int off = 0; off < R.rowbytes; off += SB) {
            const int len = min(SB, R.rowbytes - off);
            const uint8_t* piece = next_stage();
            if (!piece) {
              ok = false;
              break;
            }
            const int c0 = off / 16, nc = len / 16;
            int c = lane;
            for (; c + 32 < nc; c += 64) {
              float w0[V], w1[V], x0[V], x1[V];
              Chunk<W>::widen(*reinterpret_cast<const uint4*>(piece + (size_t)c * 16), w0);
              Chunk<W>::widen(*reinterpret_cast<const uint4*>(piece + (size_t)(c + 32) * 16), w1);
              mk_load_xs<V>(xs + (c0 + c) * V, x0);
              mk_load_xs<V>(xs + (c0 + c + 32) * V, x1);
#pragma unroll
              for (int e = 0; e < V; ++e) {
                acc0 = fmaf(w0[e], x0[e], acc0);
                acc1 = fmaf(w1[e], x1[e], acc1);
              }
            }
            if (c < nc) {
              float w0[V], x0[V];
              Chunk<W>::widen(*reinterpret_cast<const uint4*>(piece + (size_t)c * 16), w0);
              mk_load_xs<V>(xs + (c0 + c) * V, x0);
#pragma unroll
              for (int e = 0; e < V; ++e) acc0 = fmaf(w0[e], x0[e], acc0);
            }
            release_stage();
          }
          if (ok) finish(r, warp_sum(acc0 + acc1));
        }
      }
    }
  } else {
    // ---------------- tensor-core path (bf16 weights)
    // A = a 16 x 64 weight tile from the ring (128-byte swizzled by TMA), via
    // ldmatrix; B = the activation's (hi, lo) bf16 planes as columns 0 and 1
    // of the 16 x 8 operand (lanes of groups 0 and 1 carry them, the others
    // zeros); row r's dot product is D[r][0] + D[r][1], f32-accumulated.
    // 8-bit weights: every projection, and the head when it is quantised too.
    const bool q8 = MkRing<W>::Q8 && (ph != PH_LMHEAD || P.head_q8);
    const int kgs = q8 ? MK_QKG : MK_KG;
    const int KB = (R.K + kgs - 1) / kgs;   // column groups (stages) per row block
    const int grp = lane >> 2, t4 = lane & 3;
    __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(xs + P.xs_floats);
    const __nv_bfloat16* xbl = xb + (grp & 1) * P.xb_plane;   // plane of lane groups 0 / 1
    const bool bl = grp < 2;
    // ldmatrix.x4 lane roles: matrix q = lane / 8 covers rows (q & 1) * 8 + lane % 8
    // and 16-byte column chunk (q >> 1) of each 16-column step.
    const int lrow = ((lane >> 3) & 1) * 8 + (lane & 7), lch = lane >> 4;
    for (int si = 0; si < R.nseg; ++si) {
      const MkSeg S = R.seg[si];   // by value: its fields stay in registers
      if (ph == PH_DOWN) {
        // The activation this segment multiplies (MoE: its expert slot's).
        compute_sync();
        mk_to_xb(P.act + (size_t)(P.E > 0 ? S.slot : 0) * P.f, true, P.f, xb, P.xb_plane, q8);
      }
      const int nblk = (S.rows + MK_TM - 1) / MK_TM;
      for (int c0 = 0; c0 < nblk; c0 += MK_CHUNK) {
        const int nbc = min(MK_CHUNK, nblk - c0);
        for (int b = 0; b < nbc; ++b) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          for (int kb = mk_first_kb(b, KB, warp); kb < KB && ok; kb += MK_COMPUTE_WARPS) {
            const uint8_t* tile = next_stage();
            if (!tile) {
              ok = false;
              break;
            }
            if constexpr (MkRing<W>::Q8) {
              if (q8) {
                mk_q8_stage(tile, kb, grp, t4, bl, xbl, d);
                release_stage();
                continue;
              }
            }
#pragma unroll
            for (int j = 0; j < MK_BPS; ++j) {
              const uint32_t base = mk_smem_u32(tile) + 2048u * j;
              const uint32_t rsw = ((base >> 7) + (uint32_t)lrow) & 7u;   // swizzle phase of this lane's row
#pragma unroll
              for (int ks = 0; ks < MK_TK / 16; ++ks) {
                uint32_t a0, a1, a2, a3;
                mk_ldsm4(base + (uint32_t)lrow * 128u + (((uint32_t)(2 * ks + lch) ^ rsw) << 4), a0, a1, a2, a3);
                const int k0 = (kb * MK_BPS + j) * MK_TK + ks * 16 + 2 * t4;
                const uint32_t b0 = bl ? *reinterpret_cast<const uint32_t*>(xbl + k0) : 0u;
                const uint32_t b1 = bl ? *reinterpret_cast<const uint32_t*>(xbl + k0 + 8) : 0u;
                mk_mma_bf16(d, a0, a1, a2, a3, b0, b1);
              }
            }
            release_stage();
          }
          if (t4 == 0) {
            M->part[b][warp][grp] = d[0] + d[1];
            M->part[b][warp][grp + 8] = d[2] + d[3];
          }
        }
        compute_sync();
        // Rows of the chunk: the 8 warps' partials summed in warp order.
        if (R.paired) {
          for (int i = threadIdx.x; i < nbc * (MK_TM / 2); i += MK_COMPUTE) {
            const int b = i / (MK_TM / 2), pr = 2 * (i % (MK_TM / 2));
            const int rl = (c0 + b) * MK_TM + pr;
            if (rl >= S.rows) continue;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < MK_COMPUTE_WARPS; ++w) {
              a0 += M->part[b][w][pr];
              a1 += M->part[b][w][pr + 1];
            }
            mk_epi_pair<KV>(P, ph, L, S, M, rl, a0, a1);
          }
        } else {
          for (int i = threadIdx.x; i < nbc * MK_TM; i += MK_COMPUTE) {
            const int b = i / MK_TM, r = i % MK_TM;
            const int rl = (c0 + b) * MK_TM + r;
            if (rl >= S.rows) continue;
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < MK_COMPUTE_WARPS; ++w) a += M->part[b][w][r];
            mk_epi_row(P, ph, S, M, rl, a, bst, bix);
          }
        }
        compute_sync();
      }
    }
  }
  sc = scl;
  best = bst;
  bidx = bix;
  if (ph == PH_OPROJ || ph == PH_DOWN) {
    // The residual rows this CTA owns (at most 256), one coalesced pass.
    compute_sync();
    if (R.nseg > 0)
      for (int i = threadIdx.x; i < R.seg[0].rows; i += MK_COMPUTE) {
        const int row = R.seg[0].row0 + i;
        P.x[row] = __ldcg(P.x + row) + M->acc[i];
      }
  }
  return ok;
}

// ldmatrix.x4.trans: the four 8x8 b16 matrices whose rows lane l % 8 of lane
// group l / 8 points to, each delivered transposed.
__device__ __forceinline__ void mk_ldsm4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Fused FFN, second half of its phase (Pantheon "Llama Forward Pass", feed
// forward: down(silu(gate) * up), summed over the selected experts with their
// router weights).  The CTA's tasks tau (its ffn slice, per expert slot) give
// a[tau] = w_slot * silu(gate) * up (in M->fact); its share of the down
// projection is then out[n] = sum_tau Wt[tau][n] a[tau] over the transposed copy
// Wt of W_down (rows = ffn index, columns = hidden), written to fpart[CTA][n].
// Warp w owns the MK_KG-column blocks w, w + 8, ...; a stage holds Wt[16 tasks]
// [MK_KG columns] as MK_BPS 64-column boxes (128-byte swizzled).  A = (columns x
// tasks) by ldmatrix.trans of that tile, B = a's (hi, lo) bf16 planes as columns
// 0 and 1; column n's sum is D[n][0] + D[n][1], f32-accumulated over the tasks
// in their order.
template <typename W>
__device__ bool mk_ffn_down_part(const MkParams& P, const MkRows& R, uint8_t* ring, MkMisc* M, uint32_t& sc) {
  constexpr int NS = MkRing<W>::STAGES, SB = MkRing<W>::BYTES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  volatile int* abort_flag = &M->abort_flag;
  uint8_t* wring = ring + (size_t)warp * MK_WARP_RING;
  DeviceState* const stp = P.st;
  int ntask = 0;
  for (int si = 0; si < R.nseg; ++si) ntask += R.seg[si].rows / 2;
  // The activations as (hi, lo) planes (every task written by the gate/up epilogue).
  compute_sync();
  for (int i = tid; i < ntask; i += MK_COMPUTE) {
    const float v = M->fact[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    M->fxb[0][i] = hi;
    M->fxb[1][i] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
  compute_sync();
  if (ntask == 0) return true;   // a CTA past the last task (its partial row is never read)
  uint32_t scl = sc;
  bool ok = true;
  const int grp = lane >> 2, t4 = lane & 3;
  const bool bl = grp < 2;
  const __nv_bfloat16* fxbl = M->fxb[grp & 1];
  // ldmatrix.x4.trans lane roles: matrix q = lane / 8 takes task rows (q >> 1) * 8 + lane % 8
  // and the 8-column chunk (q & 1) of each 16-column step.
  const int trow = ((lane >> 4) << 3) + (lane & 7), tch = (lane >> 3) & 1;
  for (int nbk = warp; nbk < P.h / MK_KG; nbk += MK_COMPUTE_WARPS) {
    float d[MK_BPS * 4][4];
#pragma unroll
    for (int i = 0; i < MK_BPS * 4; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
    int toff = 0;
    for (int si = 0; si < R.nseg && ok; ++si) {
      const int ntb = R.seg[si].rows / (2 * MK_FTS);
      for (int tb = 0; tb < ntb; ++tb) {
        const int st = scl % NS;
        if (!mk_mbar_wait(&M->full[warp][st], (scl / NS) & 1u, abort_flag, stp, 205)) {
          ok = false;
          break;
        }
        const uint32_t tile = mk_smem_u32(wring + (size_t)st * SB);
        const int k0 = toff + tb * MK_FTS + 2 * t4;
        const uint32_t b0 = bl ? *reinterpret_cast<const uint32_t*>(fxbl + k0) : 0u;
        const uint32_t b1 = bl ? *reinterpret_cast<const uint32_t*>(fxbl + k0 + 8) : 0u;
#pragma unroll
        for (int j = 0; j < MK_BPS; ++j) {
          const uint32_t base = tile + 2048u * j;
          const uint32_t rsw = ((base >> 7) + (uint32_t)trow) & 7u;   // swizzle phase of this lane's row
#pragma unroll
          for (int mt = 0; mt < MK_TK / 16; ++mt) {
            uint32_t a0, a1, a2, a3;
            mk_ldsm4_t(base + (uint32_t)trow * 128u + (((uint32_t)(2 * mt + tch) ^ rsw) << 4), a0, a1, a2, a3);
            mk_mma_bf16(d[j * 4 + mt], a0, a1, a2, a3, b0, b1);
          }
        }
        __syncwarp();
        if (lane == 0) mk_mbar_arrive(&M->empty[warp][st]);
        ++scl;
        if (lane == 0) M->consumed[warp] = (int)scl;
      }
      toff += R.seg[si].rows / 2;
    }
    if (ok && t4 == 0) {
      float* out = P.fpart + (size_t)blockIdx.x * P.h + (size_t)nbk * MK_KG + grp;
#pragma unroll
      for (int i = 0; i < MK_BPS * 4; ++i) {
        out[16 * i] = d[i][0] + d[i][1];
        out[16 * i + 8] = d[i][2] + d[i][3];
      }
    }
  }
  sc = scl;
  return ok;
}

// Fused FFN, partial-sum phase: the hidden rows this CTA owns get the down
// projection's partials of all CTAs that had tasks, summed in CTA order (8
// interleaved running sums, then those in order), added to the residual.  Each
// thread requests up to MK_RED_J partials (and its residual row) before adding.
constexpr int MK_RED_J = 20;
__device__ void mk_ffn_reduce(const MkParams& P, float* red) {
  const int tid = threadIdx.x, g8 = tid >> 5, i = tid & 31;
  const int T = P.k * P.f, per_t = mk_share(T, P.nb, MK_FTS);
  const int nbusy = (T + per_t - 1) / per_t;
  const int per = (P.h + P.nb - 1) / P.nb;
  const int r0 = min(P.h, (int)blockIdx.x * per), r1 = min(P.h, r0 + per);
  for (int n0 = r0; n0 < r1; n0 += 32) {
    const int n = n0 + i;
    const bool live = n < r1;
    const float xo = (g8 == 0 && live) ? __ldcg(P.x + n) : 0.f;
    float s = 0.f;
    for (int c0 = g8; c0 < nbusy; c0 += MK_RED_J * MK_COMPUTE_WARPS) {
      float v[MK_RED_J];
#pragma unroll
      for (int j = 0; j < MK_RED_J; ++j) {
        const int c = c0 + MK_COMPUTE_WARPS * j;
        v[j] = (live && c < nbusy) ? __ldcg(P.fpart + (size_t)c * P.h + n) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < MK_RED_J; ++j) s += v[j];
    }
    red[g8 * 32 + i] = s;
    compute_sync();
    if (tid < 32 && live) {
      float t = 0.f;
#pragma unroll
      for (int g = 0; g < MK_COMPUTE_WARPS; ++g) t += red[g * 32 + tid];
      P.x[n] = xo + t;
    }
    compute_sync();
  }
}

// ------------------------------------------------------------------ attention phase, warp tasks
// Task t = (kv head g, split) belongs to warp (t / nb) % 8 of CTA t % nb.  That
// warp's producer streams the task's K and V rows (one head's row = HD
// elements) through the warp's weight ring, RPP keys per stage: K piece, then
// V piece.  The row of the current position is rewritten by this step's QKV
// phase, possibly after its producer copied it: the consumer reads that row
// from global memory (through L2).  Used for head_dim 64/128 and at most 8
// query heads per kv head; partials have the same layout as the CTA tasks'.
template <typename W, typename KV, int HD>
struct MkAttnGeom {
  static constexpr bool I8 = kMkKvI8<KV>;
  static constexpr int SB = MkRing<W>::BYTES < 4096 ? MkRing<W>::BYTES : 4096;   // bytes of one piece
  static constexpr int RB = I8 ? HD : HD * (int)sizeof(KV);   // bytes of one head's K or V row (codes)
  // int8: MK_I8_RPP keys per piece, codes then the keys' group scales (HD / 32 floats each).
  static constexpr int RPP = I8 ? MK_I8_RPP : SB / RB;   // keys per piece (stage)
  static constexpr int SCB = I8 ? HD / 32 * 4 : 0;   // scale bytes of one head's row
  static constexpr int SC_OFF = RPP * RB;            // offset of the scales in a stage
  static constexpr int BYTES = RPP * RB + RPP * SCB; // bytes a piece receives
  static_assert(BYTES <= SB, "a piece fits a stage");
};

// The warp-task attention plan of one step: the m readable slots of each kv head
// are cut into ns splits of sps keys (a multiple of 8), ns close to
// P.attn_ns (about one task per CTA) and at most P.nsplit (the partials' stride).
// It depends on the position only, so producer and consumer agree.
struct MkAttnPlan {
  int ns, sps, tasks;
};
__device__ __forceinline__ MkAttnPlan mk_attn_plan(const MkParams& P, int m) {
  MkAttnPlan a;
  const int target = max(1, min(P.attn_ns, P.nsplit));
  a.sps = ((m + target - 1) / target + 7) & ~7;
  a.ns = (m + a.sps - 1) / a.sps;
  a.tasks = P.nkv * a.ns;
  return a;
}

__device__ __forceinline__ void mk_attn_task(const MkAttnPlan& A, int t, int m, int& g, int& split, int& s0,
                                             int& j1) {
  g = t / A.ns;
  split = t - g * A.ns;
  s0 = split * A.sps;
  j1 = min(s0 + A.sps, m);
}

// A CTA's attention tasks t = blockIdx.x + i * nb (i < per = ceil(tasks / nb),
// the same for every CTA) are each cut into S slices of their key range, S the
// largest power of two <= 8 with per * S <= 8 (at least 1): sub-task j = i * S + k
// runs on warp j % 8 in round j / 8 and takes slice k.  The S softmax states of a
// task are combined in shared memory at the end of its round.
__device__ __forceinline__ int mk_attn_ways(const MkParams& P, const MkAttnPlan& A) {
  const int per = (A.tasks + P.nb - 1) / P.nb;
  int S = 1;
  while (S < 8 && 2 * S * per <= MK_COMPUTE_WARPS) S *= 2;
  return S;
}
__device__ __forceinline__ int mk_attn_subtasks(const MkParams& P, const MkAttnPlan& A, int S) {
  return (A.tasks + P.nb - 1) / P.nb * S;
}
__device__ __forceinline__ bool mk_attn_sub(const MkParams& P, const MkAttnPlan& A, int j, int S, int m, int& t,
                                            int& g, int& split, int& a, int& b) {
  t = blockIdx.x + (j / S) * P.nb;
  if (t >= A.tasks) return false;
  int s0, j1;
  mk_attn_task(A, t, m, g, split, s0, j1);
  const int len = max(0, j1 - s0), k = j % S;
  a = s0 + (len * k) / S;
  b = s0 + (len * (k + 1)) / S;
  return true;
}

// Merge of kv head g's split partials into the normalised outputs of its G query
// heads (by the CTA that finished the head's last split; all compute threads).
// Weight of split s: exp(m_s - M) / sum_s l_s exp(m_s - M) (rml Attend, one-pass
// softmax state).  Every load of one output is issued before the first use.
template <int HD>
__device__ void mk_merge_kv_head(const MkParams& P, int g, int ns, MkMisc* M) {
  const int G = P.nq / P.nkv, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (warp < G) {
    const float* base = P.part + (size_t)(g * G + warp) * P.nsplit * (HD + 2);
    const float ms = lane < ns ? __ldcg(base + (size_t)lane * (HD + 2) + HD) : -INFINITY;
    const float ls = lane < ns ? __ldcg(base + (size_t)lane * (HD + 2) + HD + 1) : 0.f;
    const float Mx = warp_max(ms);
    const float w = ms == -INFINITY ? 0.f : __expf(ms - Mx);
    const float L = warp_sum(ls * w);
    M->mscale[warp * 32 + lane] = L > 0.f ? w / L : 0.f;
  }
  compute_sync();
  for (int idx = tid; idx < G * HD; idx += MK_COMPUTE) {
    const int h = idx / HD, d = idx - h * HD;
    const float* base = P.part + (size_t)(g * G + h) * P.nsplit * (HD + 2) + d;
    float v[32];
#pragma unroll
    for (int s2 = 0; s2 < 32; ++s2) v[s2] = s2 < ns ? __ldcg(base + (size_t)s2 * (HD + 2)) : 0.f;
    float o = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < 32; ++s2) o = fmaf(M->mscale[h * 32 + s2], v[s2], o);
    P.attn[(size_t)(g * G + h) * HD + d] = o;
  }
  compute_sync();
}

// 2^x on the special-function unit (subnormal results flushed to zero).
__device__ __forceinline__ float ex2f_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 partial sums per lane -> lane i holds the warp-wide sum of slot i (31 shuffles).
__device__ __forceinline__ void mk_reduce_scatter32(float* v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int n = 16; n >= 1; n >>= 1) {
    const bool upper = (lane & n) != 0;
#pragma unroll
    for (int j = 0; j < n; ++j) {
      const float send = upper ? v[j] : v[j + n];
      const float keep = upper ? v[j + n] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, n);
    }
  }
}

// DPL consecutive elements of a K/V row (this lane's dims), as f32.
template <typename KV, int DPL>
__device__ __forceinline__ void mk_load_dims(const KV* p, float* v, bool global) {
  if constexpr (sizeof(KV) == 4) {
    if constexpr (DPL == 4) {
      const float4 t = global ? __ldcg(reinterpret_cast<const float4*>(p)) : *reinterpret_cast<const float4*>(p);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = global ? __ldcg(reinterpret_cast<const float2*>(p)) : *reinterpret_cast<const float2*>(p);
      v[0] = t.x; v[1] = t.y;
    }
  } else {
#pragma unroll
    for (int d = 0; d < DPL; d += 2) {
      const uint32_t u = global ? __ldcg(reinterpret_cast<const unsigned int*>(p + d))
                                : *reinterpret_cast<const uint32_t*>(p + d);
      v[d] = bf16_lo(u);
      v[d + 1] = bf16_hi(u);
    }
  }
}

// DPL consecutive K/V elements at a shared-memory address, as f32 (explicit
// ld.shared, so a piece's loads issue back to back without a generic-address check).
template <typename KV, int DPL>
__device__ __forceinline__ void mk_lds_dims(uint32_t a, float* v) {
  if constexpr (sizeof(KV) == 4 && DPL == 4) {
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(a));
  } else if constexpr (sizeof(KV) == 4 && DPL == 2) {
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v[0]), "=f"(v[1]) : "r"(a));
  } else if constexpr (sizeof(KV) == 2 && DPL == 4) {
    uint32_t u0, u1;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(u0), "=r"(u1) : "r"(a));
    v[0] = bf16_lo(u0); v[1] = bf16_hi(u0); v[2] = bf16_lo(u1); v[3] = bf16_hi(u1);
  } else {
    static_assert(sizeof(KV) == 2 && DPL == 2, "K/V row slices of 2 or 4 elements");
    uint32_t u0;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(u0) : "r"(a));
    v[0] = bf16_lo(u0); v[1] = bf16_hi(u0);
  }
}

// Four int8 codes at a shared-memory address and their group scale -> f32
// (code * scale, one correctly rounded product each, as the cache's reader).
__device__ __forceinline__ void mk_lds_i8(uint32_t a, uint32_t sa, float* v) {
  uint32_t u;
  float sc;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(u) : "r"(a));
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sc) : "r"(sa));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __fmul_rn((float)(int)(signed char)((u >> (8 * i)) & 0xffu), sc);
}

// int8 cache: this lane's 4 channels of the current position's row (f32) ->
// the values the cache will hold (per 32-channel group, eight lanes: s = max|x| /
// 127, codes round(x / s) clamped to +-127, as the cache's quantiser); the lanes of
// the task that holds the position also write the row's codes and scales for head g.
__device__ __forceinline__ void mk_quant_i8_row(float* x, bool write, char* row, int code_off, int g, int HD) {
  const int lane = threadIdx.x & 31;
  float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float sc = __fdiv_rn(m, 127.0f);
  uint32_t packed = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int code = 0;
    if (sc > 0.f) code = (int)fminf(fmaxf(roundf(__fdiv_rn(x[i], sc)), -127.0f), 127.0f);
    x[i] = __fmul_rn((float)code, sc);
    packed |= ((uint32_t)code & 0xffu) << (8 * i);
  }
  if (write) {
    *reinterpret_cast<uint32_t*>(row + code_off + g * HD + lane * 4) = packed;
    if ((lane & 7) == 0) reinterpret_cast<float*>(row)[g * (HD / 32) + (lane >> 3)] = sc;
  }
}

template <typename W, typename KV, int HD, int GP>
__device__ bool mk_attention_warp(const MkParams& P, int l, uint8_t* ring, uint8_t* ureg, MkMisc* M, uint32_t& sc) {
  using AG = MkAttnGeom<W, KV, HD>;
  constexpr int NS = MkRing<W>::STAGES, SB = MkRing<W>::BYTES, RB = AG::RB, RPP = AG::RPP;   // SB: slot stride
  constexpr int DPL = HD / 32;                                  // dims per lane
  constexpr int KG = (32 / GP) < RPP ? (32 / GP) : RPP;         // keys per reduce group
  constexpr int NG = RPP / KG;                                  // groups per piece
  constexpr float LOG2E = 1.4426950408889634f;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const MkLayer& L = P.layers[l];
  const KV* kc = (const KV*)L.kc;
  const KV* vc = (const KV*)L.vc;
  const int G = P.nq / P.nkv, kd = P.nkv * HD, tasks = P.nkv * P.nsplit;
  const int m = P.sliding > 0 ? min(P.pos + 1, P.max_seq) : P.pos + 1;
  const int slot_pos = P.sliding > 0 ? P.pos % P.max_seq : P.pos;
  const float qscale = LOG2E / sqrtf((float)HD);               // scores in log2 units
  volatile int* abort_flag = &M->abort_flag;
  uint8_t* wring = ring + (size_t)warp * MK_WARP_RING;
  DeviceState* const stp = P.st;
  uint32_t scl = sc;
  bool ok = true;
  const int own = lane % GP;                                    // this lane's head in the score slots
  const MkAttnPlan A = mk_attn_plan(P, m);
  const int S = mk_attn_ways(P, A), nsub = mk_attn_subtasks(P, A, S);
  float* sst = reinterpret_cast<float*>(ureg);                  // [8 slots][G][HD + 2] softmax states
  (void)tasks;
  for (int j0 = 0; j0 < nsub; j0 += MK_COMPUTE_WARPS) {
   const int j = j0 + warp;
   int t, g = 0, split, s0 = 0, j1 = 0;
   const bool task = j < nsub && mk_attn_sub(P, A, j, S, m, t, g, split, s0, j1);
   // The query rows and the current position's K/V row (written by this step's
   // QKV phase, possibly after the producer copied the slot, so read from global
   // memory once) are all requested before any of them is used.
   float qv[GP][DPL], kcur[DPL], vcur[DPL];
   const bool has_cur = task && slot_pos >= s0 && slot_pos < j1;
   if (task) {
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
      for (int d = 0; d < DPL; ++d) qv[h][d] = h < G ? __ldcg(P.q + (size_t)(g * G + h) * HD + lane * DPL + d) : 0.f;
    if constexpr (AG::I8) {
      // int8 cache: this position's rows come in f32 from the QKV phase.
      const float4 a = __ldcg(reinterpret_cast<const float4*>(P.kv_cur + (size_t)g * HD + lane * DPL));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(P.kv_cur + kd + (size_t)g * HD + lane * DPL));
      kcur[0] = a.x; kcur[1] = a.y; kcur[2] = a.z; kcur[3] = a.w;
      vcur[0] = b.x; vcur[1] = b.y; vcur[2] = b.z; vcur[3] = b.w;
    } else {
      const size_t co = (size_t)(has_cur ? slot_pos : 0) * kd + (size_t)g * HD + lane * DPL;
      if (P.qkn) {   // the raw k of this position (f32, from the QKV phase)
#pragma unroll
        for (int d = 0; d < DPL; ++d) kcur[d] = __ldcg(P.kv_cur + (size_t)g * HD + lane * DPL + d);
      } else {
        mk_load_dims<KV, DPL>(kc + co, kcur, true);
      }
      mk_load_dims<KV, DPL>(vc + co, vcur, true);
    }
   }
   if (task) {
    if constexpr (!AG::I8) {
      if (P.qkn) {
        // Per-head QK-norm, then the rotation (rml "The decoder", One forward pass):
        // each of the task's query heads and the current key is RMS-normalised over
        // head_dim with its shared weight, then turned by this position's adjacent-pair
        // table; the task that holds the position stores the key.
        const float* wq = L.q_norm;
        const float* wk = L.k_norm;
        float w_q[DPL], w_k[DPL];
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
          w_q[d] = wq[lane * DPL + d];
          w_k[d] = wk[lane * DPL + d];
        }
        auto norm_rope = [&](float* x, const float* w) {
          float ss = 0.f;
#pragma unroll
          for (int d = 0; d < DPL; ++d) ss = fmaf(x[d], x[d], ss);
          const float inv = 1.0f / sqrtf(warp_sum(ss) / (float)HD + P.eps);
#pragma unroll
          for (int d = 0; d < DPL; d += 2) {
            const float a = x[d] * inv * w[d], b = x[d + 1] * inv * w[d + 1];
            const float2 c = M->cs[(L.rope_local ? 64 : 0) + ((lane * DPL + d) >> 1)];
            x[d] = a * c.x - b * c.y;
            x[d + 1] = a * c.y + b * c.x;
          }
        };
#pragma unroll
        for (int h = 0; h < GP; ++h)
          if (h < G) norm_rope(qv[h], w_q);
        norm_rope(kcur, w_k);
        if (has_cur) {
          KV* dst = (KV*)L.kc + (size_t)slot_pos * kd + (size_t)g * HD + lane * DPL;
#pragma unroll
          for (int d = 0; d < DPL; ++d) dst[d] = from_f32<KV>(kcur[d]);
        }
      }
    }
    // (the scaling below is the first use of the loads above, QK-norm aside)
    float acc[GP][DPL];
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
      for (int d = 0; d < DPL; ++d) {
        qv[h][d] *= qscale;
        acc[h][d] = 0.f;
      }
    if constexpr (AG::I8) {
      static_assert(!AG::I8 || DPL == 4, "int8 cache rows: four channels per lane");
      if (has_cur) {   // (uniform over the warp)
        const size_t ro = (size_t)slot_pos * P.kv_row_bytes;
        mk_quant_i8_row(kcur, true, (char*)L.kc + ro, P.kv_code_off, g, HD);
        mk_quant_i8_row(vcur, true, (char*)L.vc + ro, P.kv_code_off, g, HD);
      }
    }
#pragma unroll
    for (int d = 0; d < DPL; ++d) {
      kcur[d] = has_cur ? kcur[d] : 0.f;
      vcur[d] = has_cur ? vcur[d] : 0.f;
    }
    float mown = -INFINITY, lown = 0.f;   // running max / sum of head `own`
    const uint32_t lane_off = (uint32_t)(lane * DPL * (int)sizeof(KV));
    for (int c0 = s0; c0 < j1; c0 += RPP) {
      const int nk = min(RPP, j1 - c0);
      // ---- K piece: scores of (key, head) slots, one per lane after the reduction
      float scr[NG];
      const uint8_t* tile = nullptr;
      if (ok) {
        const int st = scl % NS;
        if (mk_mbar_wait(&M->full[warp][st], (scl / NS) & 1u, abort_flag, stp, 203)) tile = wring + (size_t)st * SB;
        else ok = false;
      }
      // Rows past the piece's keys are read too (stale stage bytes) and masked below.
      const uint32_t ktile = mk_smem_u32(tile ? tile : wring) + lane_off;
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KG; ++kk) {
          const int r = q * KG + kk;
          float kv[DPL];
          if constexpr (AG::I8)
            mk_lds_i8(ktile + (uint32_t)(r * RB), ktile - lane_off + AG::SC_OFF + r * AG::SCB + (lane >> 3) * 4, kv);
          else mk_lds_dims<KV, DPL>(ktile + (uint32_t)(r * RB), kv);
          const bool cur = c0 + r == slot_pos;
#pragma unroll
          for (int d = 0; d < DPL; ++d) kv[d] = cur ? kcur[d] : kv[d];
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            float s = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) s = fmaf(qv[h][d], kv[d], s);
            v[kk * GP + h] = s;
          }
        }
        mk_reduce_scatter32(v);
        const int r = q * KG + lane / GP;
        scr[q] = (lane < KG * GP && r < nk && own < G) ? v[0] : -INFINITY;
      }
      if (tile) {
        __syncwarp();
        if (lane == 0) mk_mbar_arrive(&M->empty[warp][scl % NS]);
        ++scl;
        if (lane == 0) M->consumed[warp] = (int)scl;
      }
      // ---- online softmax over the piece (lanes of one head share its state)
      float cm = -INFINITY;
#pragma unroll
      for (int q = 0; q < NG; ++q) cm = fmaxf(cm, scr[q]);
#pragma unroll
      for (int o = GP; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float mn = fmaxf(mown, cm);
      const float al = mown == -INFINITY ? 0.f : ex2f_approx(mown - mn);
      float pr[NG], ps = 0.f;
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        pr[q] = scr[q] == -INFINITY ? 0.f : ex2f_approx(scr[q] - mn);
        ps += pr[q];
      }
#pragma unroll
      for (int o = GP; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      lown = lown * al + ps;
      mown = mn;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float a = __shfl_sync(0xffffffffu, al, h);
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[h][d] *= a;
      }
      // ---- V piece: acc[h] += p[key, h] * V[key]
      tile = nullptr;
      if (ok) {
        const int st = scl % NS;
        if (mk_mbar_wait(&M->full[warp][st], (scl / NS) & 1u, abort_flag, stp, 204)) tile = wring + (size_t)st * SB;
        else ok = false;
      }
      const uint32_t vtile = mk_smem_u32(tile ? tile : wring) + lane_off;
#pragma unroll
      for (int r = 0; r < RPP; ++r) {
        float vv[DPL];
        if constexpr (AG::I8)
          mk_lds_i8(vtile + (uint32_t)(r * RB), vtile - lane_off + AG::SC_OFF + r * AG::SCB + (lane >> 3) * 4, vv);
        else mk_lds_dims<KV, DPL>(vtile + (uint32_t)(r * RB), vv);
        const bool cur = c0 + r == slot_pos, live = ok && r < nk;
        // Rows past the piece's keys may hold any bits: zero them (their weights are 0).
#pragma unroll
        for (int d = 0; d < DPL; ++d) vv[d] = live ? (cur ? vcur[d] : vv[d]) : 0.f;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          const float pw = __shfl_sync(0xffffffffu, pr[r / KG], (r % KG) * GP + h);
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc[h][d] = fmaf(pw, vv[d], acc[h][d]);
        }
      }
      if (tile) {
        __syncwarp();
        if (lane == 0) mk_mbar_arrive(&M->empty[warp][scl % NS]);
        ++scl;
        if (lane == 0) M->consumed[warp] = (int)scl;
      }
    }
    // ---- this slice's state (max in log2 units) into its shared-memory slot
    float* so = sst + (size_t)(j - j0) * G * (HD + 2);
#pragma unroll
    for (int h = 0; h < GP; ++h)
      if (h < G) {
#pragma unroll
        for (int d = 0; d < DPL; ++d) so[h * (HD + 2) + lane * DPL + d] = acc[h][d];
      }
    if (lane < G) {
      so[lane * (HD + 2) + HD] = mown;
      so[lane * (HD + 2) + HD + 1] = lown;
    }
   }
    // ---- combine the S slices of each task of this round: a split partial
    // (max in natural-log units, as the merge expects), or with one split the
    // normalised output.
    compute_sync();
    const int tpr = MK_COMPUTE_WARPS / S;
    for (int e = threadIdx.x; e < tpr * G * HD; e += MK_COMPUTE) {
      const int ti = e / (G * HD), h = (e / HD) % G, d = e % HD;
      const int jt = j0 + ti * S;
      int tt, gg, sp, a, b;
      if (jt >= nsub || !mk_attn_sub(P, A, jt, S, m, tt, gg, sp, a, b)) continue;
      const float* st0 = sst + (size_t)(ti * S) * G * (HD + 2) + h * (HD + 2);
      float mx = -INFINITY;
      for (int k = 0; k < S; ++k) mx = fmaxf(mx, st0[(size_t)k * G * (HD + 2) + HD]);
      float lsum = 0.f, o = 0.f;
      if (mx != -INFINITY)
        for (int k = 0; k < S; ++k) {
          const float* sk = st0 + (size_t)k * G * (HD + 2);
          const float wk = sk[HD] == -INFINITY ? 0.f : ex2f_approx(sk[HD] - mx);
          lsum = fmaf(sk[HD + 1], wk, lsum);
          o = fmaf(sk[d], wk, o);
        }
      if (A.ns == 1) {
        P.attn[(size_t)(gg * G + h) * HD + d] = lsum > 0.f ? o / lsum : 0.f;
      } else {
        float* pp = P.part + ((size_t)(gg * G + h) * P.nsplit + sp) * (HD + 2);
        pp[d] = o;
        if (d == 0) {
          pp[HD] = mx == -INFINITY ? -INFINITY : mx / LOG2E;
          pp[HD + 1] = lsum;
        }
      }
    }
    if (A.ns > 1) {
      // This round's partials are out: count them per kv head; the CTA that
      // writes a head's last split merges the head (no separate merge phase).
      __threadfence();
      compute_sync();
      if (threadIdx.x < tpr) {
        int last = -1, tt, gg, sp, a, b;
        const int jt = j0 + threadIdx.x * S;
        if (jt < nsub && mk_attn_sub(P, A, jt, S, m, tt, gg, sp, a, b)) {
          unsigned* cnt = &stp->counters[CNT_ATTN + gg];
          if (atomicAdd(cnt, 1u) == (unsigned)A.ns - 1) {
            *cnt = 0u;   // every split of this head has arrived: ready for the next layer
            __threadfence();
            last = gg;
          }
        }
        M->lastg[threadIdx.x] = last;
      }
      compute_sync();
      for (int i = 0; i < tpr; ++i) {
        const int lg = M->lastg[i];
        if (lg >= 0) mk_merge_kv_head<HD>(P, lg, A.ns, M);
      }
    }
    compute_sync();
  }
  sc = scl;
  return ok;
}

template <typename W, typename KV, int HD>
__device__ bool mk_attention_warp_any(const MkParams& P, int l, uint8_t* ring, uint8_t* ureg, MkMisc* M,
                                      uint32_t& sc) {
  if constexpr (HD == 64 || HD == 128) {
    // Groups of 1-3 query heads per kv head run in the 4-head layout (unused
    // slots stay empty).  The 8-head layout only at head_dim 64: at 128 its
    // 64 query and accumulator registers per lane would spill, and merely
    // compiling it into the kernel worsens the register allocation of every
    // other phase (measured 2-4% slower decode steps on Mixtral and Mistral).
    if (P.nq / P.nkv <= 4) return mk_attention_warp<W, KV, HD, 4>(P, l, ring, ureg, M, sc);
    if constexpr (HD == 64) return mk_attention_warp<W, KV, HD, 8>(P, l, ring, ureg, M, sc);
    return false;
  } else {
    return false;
  }
}

// ------------------------------------------------------------------ attention phase
// Task (g, split): the G query heads of kv head g over slots
// [split*sps, split*sps + sps) intersected with the readable slots
// (min(pos+1, max_seq) under a window, else pos+1; Pantheon Sliding Window),
// one-pass online softmax in chunks of MK_KS keys (rml Attend).
template <typename KV, int HD>
__device__ void mk_attention(const MkParams& P, int l, uint8_t* ureg, MkMisc* M) {
  constexpr int CE = 16 / sizeof(KV), KROW = HD + CE, CPR = HD / CE;
  constexpr int OUTS = (MAX_GROUP * HD + MK_COMPUTE - 1) / MK_COMPUTE;
  const MkLayer& L = P.layers[l];
  const KV* kc = (const KV*)L.kc;
  const KV* vc = (const KV*)L.vc;
  const int G = P.nq / P.nkv, kd = P.nkv * HD;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  KV* ks = reinterpret_cast<KV*>(ureg);
  KV* vs = ks + MK_KS * KROW;
  float* qs = reinterpret_cast<float*>(vs + MK_KS * HD);
  float* ps = qs + G * HD;
  const int m = P.sliding > 0 ? min(P.pos + 1, P.max_seq) : P.pos + 1;
  const float scale = 1.0f / sqrtf((float)HD);
  const int tasks = P.nkv * P.nsplit;
  for (int t = blockIdx.x; t < tasks; t += P.nb) {
    const int g = t / P.nsplit, split = t - g * P.nsplit;
    const int s0 = split * P.sps, j1 = min(min(s0 + P.sps, P.max_seq), m);
    for (int i = tid; i < G * HD; i += MK_COMPUTE) qs[i] = __ldcg(P.q + (size_t)g * G * HD + i) * scale;
    if (tid < MAX_GROUP) {
      M->mrow[tid] = -INFINITY;
      M->lrow[tid] = 0.f;
    }
    float acc[OUTS];
#pragma unroll
    for (int r = 0; r < OUTS; ++r) acc[r] = 0.f;
    for (int c0 = s0; c0 < j1; c0 += MK_KS) {
      const int nt = min(MK_KS, j1 - c0);
      compute_sync();   // previous chunk's readers are done
      for (int i = tid; i < nt * CPR; i += MK_COMPUTE) {
        const int r = i / CPR, c = i - r * CPR;
        const size_t go = (size_t)(c0 + r) * kd + (size_t)g * HD + c * CE;
        cp_async16(ks + r * KROW + c * CE, kc + go);
        cp_async16(vs + r * HD + c * CE, vc + go);
      }
      cp_async_commit();
      cp_async_wait_all();
      compute_sync();
      for (int idx = tid; idx < G * nt; idx += MK_COMPUTE) {
        const int hh = idx / nt, j = idx - hh * nt;
        const float* qv = qs + hh * HD;
        const KV* kr = ks + j * KROW;
        float sdot = 0.f;
#pragma unroll 8
        for (int d = 0; d < HD; ++d) sdot = fmaf(qv[d], to_f32(kr[d]), sdot);
        ps[hh * MK_KS + j] = sdot;
      }
      compute_sync();
      for (int hh = warp; hh < G; hh += MK_COMPUTE_WARPS) {
        float* pr = ps + hh * MK_KS;
        const float sa = lane < nt ? pr[lane] : -INFINITY;
        const float sb = lane + 32 < nt ? pr[lane + 32] : -INFINITY;
        const float mnew = fmaxf(M->mrow[hh], warp_max(fmaxf(sa, sb)));
        const float pa = lane < nt ? __expf(sa - mnew) : 0.f;
        const float pb = lane + 32 < nt ? __expf(sb - mnew) : 0.f;
        const float psum = warp_sum(pa + pb);
        if (lane < nt) pr[lane] = pa;
        if (lane + 32 < nt) pr[lane + 32] = pb;
        __syncwarp();
        if (lane == 0) {
          const float a = __expf(M->mrow[hh] - mnew);
          M->alpha[hh] = a;
          M->lrow[hh] = M->lrow[hh] * a + psum;
          M->mrow[hh] = mnew;
        }
      }
      compute_sync();
#pragma unroll
      for (int r = 0; r < OUTS; ++r) {
        const int idx = tid + r * MK_COMPUTE;
        if (idx < G * HD) {
          const int hh = idx / HD, d = idx - hh * HD;
          const float* pr = ps + hh * MK_KS;
          float o = acc[r] * M->alpha[hh];
          for (int j = 0; j < nt; ++j) o = fmaf(pr[j], to_f32(vs[j * HD + d]), o);
          acc[r] = o;
        }
      }
    }
    compute_sync();
    if (P.nsplit == 1) {
#pragma unroll
      for (int r = 0; r < OUTS; ++r) {
        const int idx = tid + r * MK_COMPUTE;
        if (idx < G * HD) P.attn[(size_t)g * G * HD + idx] = acc[r] / M->lrow[idx / HD];
      }
    } else {
#pragma unroll
      for (int r = 0; r < OUTS; ++r) {
        const int idx = tid + r * MK_COMPUTE;
        if (idx < G * HD) {
          const int hh = idx / HD, d = idx - hh * HD;
          P.part[((size_t)(g * G + hh) * P.nsplit + split) * (HD + 2) + d] = acc[r];
        }
      }
      if (tid < G) {
        float* pp = P.part + ((size_t)(g * G + tid) * P.nsplit + split) * (HD + 2);
        pp[HD] = M->mrow[tid];
        pp[HD + 1] = M->lrow[tid];
      }
    }
    compute_sync();   // the task's smem is reused by the next task
  }
}

}  // namespace dec

namespace dec {

// L2 prefetch of the K/V rows this CTA's attention tasks of layer l will read,
// shared among the `nparts` producer lanes (part `part`).  The producers reach
// the attention phase while the QKV weights are still streaming, so the
// prefetch runs ahead of the attention phase off the compute path (the current
// position's row, rewritten by the QKV phase, is updated in L2 by that write).
__device__ void mk_prefetch_attention_kv(const MkParams& P, int l, int HD, int part, int nparts) {
  const MkLayer& L = P.layers[l];
  const int kvb = P.kv_bytes;
  const int kd = P.nkv * HD;
  const int m = P.sliding > 0 ? min(P.pos + 1, P.max_seq) : P.pos + 1;
  int ns = P.nsplit, sps = P.sps;
  if (P.attn_warp) {
    const MkAttnPlan A = mk_attn_plan(P, m);
    ns = A.ns;
    sps = A.sps;
  }
  const int tasks = P.nkv * ns;
  int idx = part;
  // With tensor maps (bf16 weights): one prefetch per piece (one ring stage of keys)
  // and map: K and V, and with an int8 cache (MK_I8_RPP keys per piece) their scales too.
  const bool i8 = P.kv_code_off > 0;
  const int rpp = P.maps ? (i8 ? MK_I8_RPP : MkRing<__nv_bfloat16>::BYTES / (HD * kvb)) : 0;
  const int kinds = i8 ? 4 : 2;
  for (int t = blockIdx.x; t < tasks; t += P.nb) {
    const int g = t / ns, split = t - g * ns;
    const int s0 = split * sps, j1 = min(min(s0 + sps, P.max_seq), m);
    const int n = j1 > s0 ? j1 - s0 : 0;
    if (rpp) {
      const int pieces = (n + rpp - 1) / rpp;
      for (; idx < kinds * pieces; idx += nparts) {
        const int kind = idx % kinds;
        const int map = kind == 0 ? MAP_K : kind == 1 ? MAP_V : kind == 2 ? MAP_KS : MAP_VS;
        tma_prefetch_3d(P.maps + l * MAPS_PER_LAYER + map, 0, g, s0 + (idx / kinds) * rpp);
      }
      idx -= kinds * pieces;
      continue;
    }
    for (; idx < 2 * n; idx += nparts) {
      const int r = idx >> 1;
      const uint8_t* base = (const uint8_t*)((idx & 1) ? L.vc : L.kc);
      mk_prefetch_l2(base + ((size_t)(s0 + r) * kd + (size_t)g * HD) * kvb, (uint32_t)(HD * kvb));
    }
    idx -= 2 * n;
  }
}

// ------------------------------------------------------------------ the kernel
template <typename W, typename KV, int HD>
__device__ void mk_produce(const MkParams& P, uint8_t* ring, MkMisc* M);
template <typename W, typename KV, int HD>
__device__ void mk_compute(const MkParams& P, uint8_t* ring, uint8_t* ureg, MkMisc* M);

template <typename W, typename KV, int HD>
__global__ void __launch_bounds__(MK_THREADS, 1) k_decode_step(const __grid_constant__ MkParams P) {
  extern __shared__ __align__(1024) uint8_t mk_smem[];
  uint8_t* ring = mk_smem;
  uint8_t* ureg = mk_smem + MK_RING_BYTES;
  MkMisc* M = reinterpret_cast<MkMisc*>(ureg + P.u_bytes);
  const int tid = threadIdx.x;
  // Swizzled TMA tiles and their ldmatrix addressing assume a 1024-byte
  // aligned window; every CTA of the launch has the same window, so this exit
  // is uniform (also across a cluster).
  if (mk_smem_u32(mk_smem) & 1023u) {
    if (tid == 0) raise_error(P.st, ERR_LAYOUT, 130);
    return;
  }

  if (tid == 0) {
    for (int w = 0; w < MK_COMPUTE_WARPS; ++w)
      for (int s = 0; s < MkRing<W>::STAGES; ++s) {
        mk_mbar_init(&M->full[w][s], 1);
        mk_mbar_init(&M->empty[w][s], 1);
      }
    M->abort_flag = 0;
    mk_mbar_init(&M->moe_bar, 1);
    for (int w = 0; w < MK_COMPUTE_WARPS; ++w) M->consumed[w] = 0;
    if (P.cluster) mk_mbar_init(&M->cbar, (uint32_t)P.cluster);
    M->cgen = 0;
    int t = P.d_token ? *P.d_token : P.token;
    if (t < 0 || t >= P.V) {
      raise_error(P.st, ERR_TOKEN, 0);
      t = 0;
    }
    M->token = t;
    if (blockIdx.x == 0) {
      P.st->token = t;
      P.st->pos = P.pos;
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  for (int i = tid; i < P.hd / 2; i += MK_THREADS) {
    double sn, cn;
    sincos((double)P.pos * P.inv_freq[i], &sn, &cn);
    M->cs[i] = make_float2((float)cn, (float)sn);
    if (P.inv_freq_local) {   // per-layer RoPE base: the local layers' table
      sincos((double)P.pos * P.inv_freq_local[i], &sn, &cn);
      M->cs[64 + i] = make_float2((float)cn, (float)sn);
    }
  }
  __syncthreads();
  // Cluster mode: every CTA's barrier is initialised before any remote
  // arrival, and (at the end) no CTA exits while another may still arrive on
  // its barrier.  barrier.cluster counts every thread of the cluster.
  if (P.cluster) asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  // Register split: the producer warpgroups (one active lane per warp) give
  // registers to the compute warpgroups.  The launch holds MK_THREADS x
  // MK_REGS registers (the host refuses a build with another count), and the
  // two shares add up to exactly that, so the increase always completes once
  // the producers' decrease has run (which waits on nothing).
  if ((tid >> 5) >= MK_COMPUTE_WARPS) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(MK_REGS_PRODUCER) : "memory");
    mk_produce<W, KV, HD>(P, ring, M);
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(MK_REGS_COMPUTE) : "memory");
    mk_compute<W, KV, HD>(P, ring, ureg, M);
  }
  if (P.cluster) asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

template <typename W, typename KV, int HD>
__device__ void mk_produce(const MkParams& P, uint8_t* ring, MkMisc* M) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nphase = P.n_layers * mk_phases_per_layer(P) + 1;
  volatile int* abort_flag = &M->abort_flag;
  {
    // ---------------- producer: warp 8+w streams compute warp w's rows of every phase, in order
    constexpr int NS = MkRing<W>::STAGES, SB = MkRing<W>::BYTES;
    const int w = warp - MK_COMPUTE_WARPS;
    if ((tid & 31) == 0) {
      uint8_t* wring = ring + (size_t)w * MK_WARP_RING;
      uint32_t sc = 0;
      bool ok = true;
      auto claim = [&](uint32_t len) -> int {   // next stage, armed for len bytes; -1 if gave up
        const int st = sc % NS;
        const uint32_t par = (sc / NS) & 1u;
        if (!mk_mbar_wait(&M->empty[w][st], par ^ 1u, abort_flag, P.st, 302)) return -1;
        mk_mbar_expect_tx(&M->full[w][st], len);
        ++sc;
        return st;
      };
      for (int i = 0; i < nphase && ok && !*abort_flag; ++i) {
        int ph, l;
        mk_phase_at(P, i, ph, l);
        // The layer's K/V history is final before its QKV phase (only the current
        // position's row is written there, and the consumer reads that row from
        // global memory): prefetch it into L2 while the QKV weights stream, so the
        // attention phase reads it from L2.
        if (ph == PH_QKV) mk_prefetch_attention_kv(P, l, P.hd, w, MK_COMPUTE_WARPS);
        // The next phases' small operands (norm weights, router rows), read by every
        // CTA right after a barrier: one CTA asks L2 for them a phase ahead.
        if (blockIdx.x == 0 && w == 0 && l < P.n_layers) {
          const MkLayer& Lp = P.layers[l];
          if (ph == PH_OPROJ) {
            mk_prefetch_l2_any(Lp.ffn_norm, (uint32_t)(P.h * 4));
            if (P.E > 0) mk_prefetch_l2_any(Lp.router, (uint32_t)(P.E * P.h * (int)sizeof(typename MkElem<W>::T)));
          } else if (ph == PH_GATEUP) {
            mk_prefetch_l2_any(l + 1 < P.n_layers ? P.layers[l + 1].attn_norm : P.out_norm, (uint32_t)(P.h * 4));
          }
        }
        if constexpr (HD == 64 || HD == 128) {
          if (ph == PH_ATTN && P.attn_warp) {
            // This warp's attention tasks: per RPP keys a K piece, then a V piece,
            // one bulk copy per key row of the task's kv head.
            using AG = MkAttnGeom<W, KV, HD>;
            const MkLayer& L = P.layers[l];
            const int m = P.sliding > 0 ? min(P.pos + 1, P.max_seq) : P.pos + 1;
            const int kd = P.nkv * HD;
            const MkAttnPlan A = mk_attn_plan(P, m);
            const int S = mk_attn_ways(P, A), nsub = mk_attn_subtasks(P, A, S);
            for (int j = w; j < nsub && ok; j += MK_COMPUTE_WARPS) {
              int t, g, split, s0, j1;   // [s0, j1): this sub-task's keys
              if (!mk_attn_sub(P, A, j, S, m, t, g, split, s0, j1)) continue;
              for (int c0 = s0; c0 < j1 && ok; c0 += AG::RPP) {
                const int nk = min(AG::RPP, j1 - c0);
                for (int kv = 0; kv < 2 && ok; ++kv) {
                  // A tensor map moves the piece (RPP keys of head g) in one copy; the
                  // box is always whole (slots past the ring read as zeros, unused).
                  const int st = claim((uint32_t)(P.maps ? AG::BYTES : nk * AG::RB));
                  if (st < 0) {
                    ok = false;
                    break;
                  }
                  if (P.maps) {
                    const CUtensorMap* lm = P.maps + l * MAPS_PER_LAYER;
                    tma_load_3d(wring + (size_t)st * SB, lm + (kv ? MAP_V : MAP_K), &M->full[w][st], 0, g, c0);
                    if constexpr (AG::I8)   // the piece's group scales after its codes
                      tma_load_3d(wring + (size_t)st * SB + AG::SC_OFF, lm + (kv ? MAP_VS : MAP_KS), &M->full[w][st], 0,
                                  g, c0);
                  } else {
                    const KV* base = (const KV*)(kv ? L.vc : L.kc);
                    for (int r = 0; r < nk; ++r)
                      mk_bulk_load(wring + (size_t)st * SB + (size_t)r * AG::RB,
                                   base + (size_t)(c0 + r) * kd + (size_t)g * HD, (uint32_t)AG::RB, &M->full[w][st]);
                  }
                }
              }
            }
            continue;
          }
        }
        if (!mk_is_gemv(P, ph)) continue;
        if (P.E > 0 && (ph == PH_GATEUP || ph == PH_DOWN)) {
          // Expert rows are known once this layer's router has run: its barrier
          // completes once per layer, and this producer is never a whole layer
          // ahead of the router (it needs this layer's rows consumed first), so
          // completion l is the one with parity l & 1.
          if (!mk_mbar_wait(&M->moe_bar, (uint32_t)(l & 1), abort_flag, P.st, 301)) break;
        }
        MkRows& R = M->rows[MK_COMPUTE_WARPS + w];   // written and read by this lane only
        mk_phase_rows<W>(P, ph, l, M->ids, R);
        for (int si = 0; si < R.nseg && ok; ++si) {
          const MkSeg S = R.seg[si];   // by value: its fields stay in registers
          if constexpr (MkRing<W>::MMA) {
            // 16 x 64 tiles in the consumer's order: block by block, this
            // warp's column blocks of each (see mk_first_kb).  8-bit weights:
            // two 128-column code boxes and the rows' scales per stage.
            const CUtensorMap* map = P.maps + S.map;
            const bool q8 = MkRing<W>::Q8 && (ph != PH_LMHEAD || P.head_q8);
            const CUtensorMap* smap =
                P.maps + (S.map < P.n_layers * MAPS_PER_LAYER ? S.map + MAP_SCALE_OFF : S.map + 1);
            const int kgs = q8 ? MK_QKG : MK_KG;
            const int KB = (R.K + kgs - 1) / kgs;
            const int nblk = (S.rows + MK_TM - 1) / MK_TM;
            for (int blk = 0; blk < nblk && ok; ++blk)
              for (int kb = mk_first_kb(blk % MK_CHUNK, KB, w); kb < KB && ok; kb += MK_COMPUTE_WARPS) {
                const int st = claim(q8 ? (uint32_t)MK_QSTAGE : (uint32_t)(2048 * MK_BPS));
                if (st < 0) {
                  ok = false;
                  break;
                }
                if (q8) {
                  for (int j = 0; j < 2; ++j)
                    tma_load_2d(wring + (size_t)st * SB + 2048 * j, map, &M->full[w][st], kb * MK_QKG + j * 128,
                                S.maprow + blk * MK_TM);
                  tma_load_2d(wring + (size_t)st * SB + MK_QSC, smap, &M->full[w][st], kb * (MK_QKG / 32),
                              S.maprow + blk * MK_TM);
                } else {
                  for (int j = 0; j < MK_BPS; ++j)
                    tma_load_2d(wring + (size_t)st * SB + 2048 * j, map, &M->full[w][st], (kb * MK_BPS + j) * MK_TK,
                                S.maprow + blk * MK_TM);
                }
              }
          } else {
            int r0, r1;
            mk_warp_rows(R, S, w, r0, r1);
            const uint8_t* base = S.base + (size_t)S.row0 * R.rowbytes;
            auto issue = [&](const uint8_t* src, int len) -> bool {
              const int st = claim((uint32_t)len);
              if (st < 0) return false;
              mk_bulk_load(wring + (size_t)st * SB, src, (uint32_t)len, &M->full[w][st]);
              return true;
            };
            if (R.rowbytes <= SB) {
              const int rps = SB / R.rowbytes;
              for (int r = r0; r < r1 && ok; r += rps)
                ok = issue(base + (size_t)r * R.rowbytes, min(rps, r1 - r) * R.rowbytes);
            } else {
              for (int r = r0; r < r1 && ok; ++r)
                for (int off = 0; off < R.rowbytes && ok; off += SB)
                  ok = issue(base + (size_t)r * R.rowbytes + off, min(SB, R.rowbytes - off));
            }
          }
        }
        if constexpr (MkRing<W>::MMA && !MkRing<W>::Q8) {
          // Fused FFN: then this warp's stages of the down half (mk_ffn_down_part's
          // order): per owned column block, each segment's tasks 16 rows at a time
          // from the transposed copy (its row = the gate/up map row / 2).
          if (ph == PH_GATEUP && P.ffn_fused) {
            const CUtensorMap* tmap = P.maps + (l * MAPS_PER_LAYER + MAP_DOWN_T);
            for (int nbk = w; nbk < P.h / MK_KG && ok; nbk += MK_COMPUTE_WARPS)
              for (int si = 0; si < R.nseg && ok; ++si) {
                const int y0 = R.seg[si].maprow / 2, ntb = R.seg[si].rows / (2 * MK_FTS);
                for (int tb = 0; tb < ntb && ok; ++tb) {
                  const int st = claim((uint32_t)(2048 * MK_BPS));
                  if (st < 0) {
                    ok = false;
                    break;
                  }
                  for (int j = 0; j < MK_BPS; ++j)
                    tma_load_2d(wring + (size_t)st * SB + 2048 * j, tmap, &M->full[w][st], nbk * MK_KG + j * MK_TK,
                                y0 + tb * MK_FTS);
                }
              }
          }
        }
      }
      if (*abort_flag) {
        // Copies issued but never consumed must land before the CTA exits.
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t k = (uint32_t)*(volatile int*)&M->consumed[w]; k < sc; ++k)
          while (!mk_mbar_try(&M->full[w][k % NS], (k / NS) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
          }
      }
    }
  }
}

template <typename W, typename KV, int HD>
__device__ void mk_compute(const MkParams& P, uint8_t* ring, uint8_t* ureg, MkMisc* M) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nphase = P.n_layers * mk_phases_per_layer(P) + 1;
  volatile int* abort_flag = &M->abort_flag;
  float* xs = reinterpret_cast<float*>(ureg);
  // Tensor-core GEMV operand: the activation as bf16 (hi, lo) planes after xs.
  constexpr bool MMA = MkRing<W>::MMA;
  constexpr bool Q8 = MkRing<W>::Q8;   // 8-bit phases take the activation as f16 (hi, lo) planes
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(xs + P.xs_floats);
  const int kpad_h = (P.h + MK_PADK - 1) / MK_PADK * MK_PADK;
  // ---------------- compute warps
  if (P.stamps && blockIdx.x == 0 && tid == 0) P.stamps[0] = globaltimer_ns();
  const int token = M->token;
  const int qd = P.nq * P.hd;
  // The residual starts as the token's embedding row (every CTA writes a share).
  for (int i = blockIdx.x * MK_COMPUTE + tid; i < P.h; i += P.nb * MK_COMPUTE)
    P.x[i] = to_f32(((const typename MkElem<W>::T*)P.embed)[(size_t)token * P.h + i]);
  uint32_t sc = 0;
  float best = -INFINITY;
  int bidx = 0x7fffffff;
  // Grid barriers: this launch's base count (thread 0 is the only one that uses it).
  unsigned long long bar_target = 0;
  if (tid == 0 && !P.cluster) {
    const unsigned long long c0 = ld_relaxed_u64(mk_bar_counter(P.st));
    bar_target = c0 / (unsigned long long)P.nb * (unsigned long long)P.nb;
  }
  for (int i = 0; i < nphase; ++i) {
    int ph, l;
    mk_phase_at(P, i, ph, l);
    const MkLayer& L = P.layers[l < P.n_layers ? l : 0];
    bool ok = true;
    switch (ph) {
      case PH_QKV:
        mk_norm_to_xs<typename MkElem<W>::T>(P.x, l == 0 ? (const typename MkElem<W>::T*)P.embed + (size_t)token * P.h : nullptr, L.attn_norm, P.h, P.eps,
                         xs, M, MMA ? xb : nullptr, P.xb_plane, kpad_h, Q8);
        break;
      // Head dims 64 / 128 always take the warp-task attention (the host declines
      // the persistent step for their other shapes): the CTA-task attention and its
      // merges are compiled only into the other instantiations, which keeps their
      // code out of the hot kernels.
      case PH_ATTN:
        if constexpr (HD == 64 || HD == 128) ok = mk_attention_warp_any<W, KV, HD>(P, l, ring, ureg, M, sc);
        else mk_attention<KV, HD>(P, l, ureg, M);
        break;
      case PH_MERGE:
        if constexpr (HD != 64 && HD != 128)
          for (int h0 = blockIdx.x; h0 < P.nq; h0 += P.nb)
            mk_merge_heads(P.part, P.nsplit, HD, h0, 1, xs, P.attn, true);
        break;
      case PH_OPROJ:
        if (HD != 64 && HD != 128 && P.nsplit > 1 && !P.merge_phase) {
          mk_merge_heads(P.part, P.nsplit, HD, 0, P.nq, xs + qd, xs, false);
          if (MMA) mk_to_xb(xs, false, qd, xb, P.xb_plane, Q8);
        } else if (MMA) {
          mk_to_xb(P.attn, true, qd, xb, P.xb_plane, Q8);   // the tensor-core GEMV reads only the planes
        } else {
          mk_copy_to_xs(P.attn, qd, xs);
        }
        break;
      case PH_GATEUP:
        mk_norm_to_xs<typename MkElem<W>::T>(P.x, nullptr, L.ffn_norm, P.h, P.eps, xs, M, MMA ? xb : nullptr, P.xb_plane, kpad_h,
                                             Q8);
        if (P.E > 0) mk_router<typename MkElem<W>::T>(P, l, xs, M);
        break;
      case PH_DOWN:
        // (tensor-core path: the activation is converted per segment)
        if (!MMA && P.E == 0) mk_copy_to_xs(P.act, P.f, xs);
        break;
      case PH_LMHEAD:
        mk_norm_to_xs<typename MkElem<W>::T>(P.x, nullptr, P.out_norm, P.h, P.eps, xs, M, MMA ? xb : nullptr, P.xb_plane, kpad_h,
                                             Q8 && P.head_q8);
        break;
    }
    if (mk_is_gemv(P, ph)) {
      MkRows& R = M->rows[warp];
      if ((tid & 31) == 0) mk_phase_rows<W>(P, ph, l, M->ids, R);
      __syncwarp();
      ok = mk_gemv_phase<W, KV>(P, ph, l, R, ring, M, xs, sc, best, bidx);
      if constexpr (MMA && !Q8) {
        if (ph == PH_GATEUP && P.ffn_fused && !compute_sync_or(!ok)) ok = mk_ffn_down_part<W>(P, R, ring, M, sc);
      }
    } else if (ph == PH_DOWN && P.ffn_fused) {
      mk_ffn_reduce(P, xs);
    }
    // Every exit below is agreed by all compute threads (a thread that left
    // alone would leave the others at the next compute barrier).
    if (compute_sync_or(!ok || *abort_flag)) break;
    if (ph != PH_LMHEAD) {
      bar_target += (unsigned long long)P.nb;
      const bool synced = P.cluster ? mk_cluster_sync(P.st, (unsigned)P.nb, &M->cbar, &M->cgen, abort_flag, 400 + ph)
                                    : mk_grid_sync(P.st, bar_target, abort_flag, 400 + ph);
      if (compute_sync_or(!synced)) break;
    }
    if (P.stamps && blockIdx.x == 0 && tid == 0) P.stamps[i + 1] = globaltimer_ns();
  }
  if (compute_sync_or(*abort_flag) || !P.d_argmax) return;

  // ---------------- argmax: CTA best -> per-CTA partial -> last CTA merges
  const int lane = tid & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ov > best || (ov == best && oi < bidx)) {
      best = ov;
      bidx = oi;
    }
  }
  if (lane == 0) {
    M->wbest[warp] = best;
    M->wbidx[warp] = bidx;
  }
  compute_sync();
  if (tid == 0) {
    float b = M->wbest[0];
    int bi = M->wbidx[0];
    for (int w = 1; w < MK_COMPUTE_WARPS; ++w)
      if (M->wbest[w] > b || (M->wbest[w] == b && M->wbidx[w] < bi)) {
        b = M->wbest[w];
        bi = M->wbidx[w];
      }
    P.amax_val[blockIdx.x] = b;
    P.amax_idx[blockIdx.x] = bi;
    __threadfence();
    M->is_last = atomicAdd(&P.st->counters[CNT_ARGMAX], 1u) == (unsigned)P.nb - 1;
  }
  compute_sync();
  if (!M->is_last) return;
  __threadfence();
  float b = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = tid; i < P.nb; i += MK_COMPUTE) {
    const float v = __ldcg(P.amax_val + i);
    const int vi = __ldcg(P.amax_idx + i);
    if (v > b || (v == b && vi < bi)) {
      b = v;
      bi = vi;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, b, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > b || (ov == b && oi < bi)) {
      b = ov;
      bi = oi;
    }
  }
  compute_sync();
  if (lane == 0) {
    M->wbest[warp] = b;
    M->wbidx[warp] = bi;
  }
  compute_sync();
  if (tid == 0) {
    for (int w = 1; w < MK_COMPUTE_WARPS; ++w)
      if (M->wbest[w] > M->wbest[0] || (M->wbest[w] == M->wbest[0] && M->wbidx[w] < M->wbidx[0])) {
        M->wbest[0] = M->wbest[w];
        M->wbidx[0] = M->wbidx[w];
      }
    *P.d_argmax = M->wbidx[0];
    P.st->counters[CNT_ARGMAX] = 0u;
  }
}

}  // namespace dec

namespace dec {

// ------------------------------------------------------------------ bounded-wait self-test
// One CTA enters the persistent step's grid barrier expecting two arrivals.  The
// second never comes, so the wait runs out after limit_ns, records ERR_TIMEOUT with
// the site and returns: the path a real step takes when a peer CTA never arrives.
__global__ void __launch_bounds__(MK_COMPUTE, 1) k_wait_selftest(DeviceState* st, uint64_t limit_ns, unsigned site) {
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  // Target: two arrivals beyond the count before this one's; only one comes.
  const unsigned long long target = ld_relaxed_u64(mk_bar_counter(st)) + 2ull;
  mk_grid_sync(st, target, &abort_flag, site, limit_ns);
}

cudaError_t launch_wait_selftest(const Model& m, cudaStream_t s, uint64_t limit_ns, unsigned site) {
  k_wait_selftest<<<1, MK_COMPUTE, 0, s>>>(m.s.st, limit_ns, site);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host side
// Floats of the f32 activation region xs: the phase inputs (on the tensor-core
// path only those of length hidden or n_heads*head_dim; the FFN activation goes
// straight to the bf16 planes) plus the split-merge scratch of the output
// projection.
static int mk_xs_floats(const dec_config& c, int nsplit) {
  size_t xs = (size_t)c.hidden;
  if ((size_t)c.n_heads * c.head_dim > xs) xs = (size_t)c.n_heads * c.head_dim;
  if (c.weight_dtype != DEC_BF16 && (size_t)c.ffn > xs) xs = c.ffn;
  xs += (size_t)c.n_heads * nsplit;
  return (int)((xs + 3) / 4 * 4);
}

// Elements of one bf16 activation plane (tensor-core path): the longest row,
// in whole 64-column blocks.
static int mk_xb_plane(const dec_config& c) {
  size_t k = (size_t)c.hidden;
  if ((size_t)c.n_heads * c.head_dim > k) k = (size_t)c.n_heads * c.head_dim;
  if ((size_t)c.ffn > k) k = c.ffn;
  return (int)((k + MK_PADK - 1) / MK_PADK * MK_PADK);
}

static size_t mk_u_bytes(const dec_config& c, int nsplit) {
  const size_t kvs = c.kv_dtype == DEC_BF16 ? 2 : 4;
  const size_t ce = 16 / kvs, hd = c.head_dim, G = c.n_heads / c.n_kv_heads;
  size_t xs = (size_t)mk_xs_floats(c, nsplit) * sizeof(float);
  if (c.weight_dtype == DEC_BF16) xs += 2 * sizeof(__nv_bfloat16) * (size_t)mk_xb_plane(c);
  size_t attn = MK_KS * (hd + ce) * kvs + MK_KS * hd * kvs + G * hd * 4 + G * MK_KS * 4;
  const size_t slots = (size_t)MK_COMPUTE_WARPS * G * (hd + 2) * 4;   // warp-task softmax states
  if (slots > attn) attn = slots;
  const size_t u = xs > attn ? xs : attn;
  return (u + 127) / 128 * 128;
}

// Attention as per-warp tasks: head_dim 64/128 (a lane owns head_dim / 32
// dims), at most 8 (head_dim 64) or 4 (head_dim 128) query heads per kv head,
// and a stage holds at least one head's K or V row; other shapes take the
// CTA-task attention.
static bool mk_attn_warp_ok(const dec_config& c) {
  const int G = c.n_heads / c.n_kv_heads;
  return (c.head_dim == 64 && G >= 1 && G <= 8) || (c.head_dim == 128 && G >= 1 && G <= 4);
}

size_t mk_smem_bytes(const dec_config& c, int nsplit) {
  return (size_t)MK_RING_BYTES + mk_u_bytes(c, nsplit) + sizeof(MkMisc);
}

size_t mk_maps_bytes(const dec_config& c) {
  return c.weight_dtype == DEC_BF16 ? sizeof(CUtensorMap) * ((size_t)c.n_layers * MAPS_PER_LAYER + 2) : 0;
}

static PFN_cuTensorMapEncodeTiled_v12000 mk_encode_fn() {
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

// A [rows][K] bf16 weight matrix as 16 x 64 tiles with 128-byte swizzling.
static bool mk_encode(CUtensorMap* m, const void* base, uint64_t rows, uint64_t K) {
  auto fn = mk_encode_fn();
  if (!fn || !base) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)MK_TK, (cuuint32_t)MK_TM};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of every bf16 weight matrix the step streams, copied to m.mk_maps.
static bool mk_build_maps(Model& m) {
  const dec_config& c = m.cfg;
  if (c.weight_dtype != DEC_BF16) return true;
  if (!m.mk_maps) return false;
  const uint64_t h = c.hidden, qd = (uint64_t)c.n_heads * c.head_dim, kd = (uint64_t)c.n_kv_heads * c.head_dim;
  const uint64_t f = c.ffn, E = c.n_experts > 0 ? c.n_experts : 1;
  std::vector<CUtensorMap> maps((size_t)c.n_layers * MAPS_PER_LAYER + 2);
  const size_t head_map = (size_t)c.n_layers * MAPS_PER_LAYER;
  if (m.wq8) {
    // 8-bit weights: codes [rows][K] in boxes of 16 rows x 128 columns (128-byte
    // swizzle), scales [rows][K / 32] f32 in boxes of 16 rows x 8 groups.
    auto fn = mk_encode_fn();
    if (!fn) return false;
    auto codes = [&](CUtensorMap* t, const QMat& q, uint64_t rows, uint64_t K) {
      const cuuint64_t dims[2] = {K, rows};
      const cuuint64_t strides[1] = {K};
      const cuuint32_t box[2] = {128, (cuuint32_t)MK_TM};
      const cuuint32_t estr[2] = {1, 1};
      return q.codes && fn(t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(q.codes), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto scales = [&](CUtensorMap* t, const QMat& q, uint64_t rows, uint64_t K) {
      const cuuint64_t dims[2] = {K / 32, rows};
      const cuuint64_t strides[1] = {K / 32 * 4};   // rejected unless a multiple of 16 bytes
      const cuuint32_t box[2] = {(cuuint32_t)(MK_QKG / 32), (cuuint32_t)MK_TM};
      const cuuint32_t estr[2] = {1, 1};
      return q.scales && fn(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(q.scales), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    for (int l = 0; l < c.n_layers; ++l) {
      const LayerPtrs& L = m.layers[l];
      CUtensorMap* t = &maps[(size_t)l * MAPS_PER_LAYER];
      if (!codes(t + MAP_QKV, L.q_wqkv, qd + 2 * kd, h) || !scales(t + MAP_QKV_S, L.q_wqkv, qd + 2 * kd, h) ||
          !codes(t + MAP_O, L.q_wo, h, qd) || !scales(t + MAP_O_S, L.q_wo, h, qd) ||
          !codes(t + MAP_GATEUP, L.q_gateup, E * 2 * f, h) || !scales(t + MAP_GATEUP_S, L.q_gateup, E * 2 * f, h) ||
          !codes(t + MAP_DOWN, L.q_down, E * h, f) || !scales(t + MAP_DOWN_S, L.q_down, E * h, f))
        return false;
    }
    if (m.q_head.codes) {
      if (!codes(&maps[head_map], m.q_head, (uint64_t)c.vocab, h) ||
          !scales(&maps[head_map + 1], m.q_head, (uint64_t)c.vocab, h))
        return false;
    } else if (!mk_encode(&maps[head_map], m.head, (uint64_t)c.vocab, h)) {
      return false;
    }
  } else {
    for (int l = 0; l < c.n_layers; ++l) {
      const LayerPtrs& L = m.layers[l];
      CUtensorMap* t = &maps[(size_t)l * MAPS_PER_LAYER];
      if (!mk_encode(t + MAP_QKV, L.wqkv, qd + 2 * kd, h) || !mk_encode(t + MAP_O, L.wo, h, qd) ||
          !mk_encode(t + MAP_GATEUP, L.w_gateup, E * 2 * f, h) || !mk_encode(t + MAP_DOWN, L.w_down, E * h, f))
        return false;
      if (L.w_down_t && !mk_encode(t + MAP_DOWN_T, L.w_down_t, E * f, h)) return false;
    }
    if (!mk_encode(&maps[head_map], m.head, (uint64_t)c.vocab, h)) return false;
  }
  // K and V rings: [slots][kv heads][head_dim], a box = one attention piece of one head.
  // int8 rings: rows of [scales][codes] (KvRowLayout); the codes map starts at the
  // codes' offset, the scales map at the row (one head's scales = HD / 32 floats),
  // both with the row as the slot stride; a box covers the piece's MK_I8_RPP keys.
  const bool kvb16 = c.kv_dtype == DEC_BF16, kvi8 = c.kv_dtype == DEC_I8;
  const uint64_t es = kvb16 ? 2 : 4, hd = (uint64_t)c.head_dim;
  const KvRowLayout rl = kv_row_layout(c);
  auto encode_ring = [&](CUtensorMap* t, const void* base) {
    auto fn = mk_encode_fn();
    if (!fn || !base) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    if (kvi8) {
      const cuuint64_t dims[3] = {hd, (cuuint64_t)c.n_kv_heads, (cuuint64_t)c.max_seq};
      const cuuint64_t strides[2] = {hd, (cuuint64_t)rl.bytes};
      const cuuint32_t box[3] = {(cuuint32_t)hd, 1, (cuuint32_t)MK_I8_RPP};
      return fn(t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<char*>((const char*)base + rl.code_off), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[3] = {hd, (cuuint64_t)c.n_kv_heads, (cuuint64_t)c.max_seq};
    const cuuint64_t strides[2] = {hd * es, kd * es};
    const cuuint32_t box[3] = {(cuuint32_t)hd, 1, (cuuint32_t)(MkRing<__nv_bfloat16>::BYTES / (hd * es))};
    return fn(t, kvb16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  auto encode_scales = [&](CUtensorMap* t, const void* base) {
    auto fn = mk_encode_fn();
    if (!fn || !base) return false;
    const cuuint64_t dims[3] = {hd / 32, (cuuint64_t)c.n_kv_heads, (cuuint64_t)c.max_seq};
    const cuuint64_t strides[2] = {hd / 32 * 4, (cuuint64_t)rl.bytes};
    const cuuint32_t box[3] = {(cuuint32_t)(hd / 32), 1, (cuuint32_t)MK_I8_RPP};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(t, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerPtrs& L = m.layers[l];
    CUtensorMap* t = &maps[(size_t)l * MAPS_PER_LAYER];
    if (kvi8) {
      if (!decode_kv_i8_persistent(c) || !encode_ring(t + MAP_K, L.kc) || !encode_ring(t + MAP_V, L.vc) ||
          !encode_scales(t + MAP_KS, L.kc) || !encode_scales(t + MAP_VS, L.vc))
        return false;
    } else if ((hd == 64 || hd == 128) && (!encode_ring(t + MAP_K, L.kc) || !encode_ring(t + MAP_V, L.vc))) {
      return false;
    }
  }
  return cudaMemcpy(m.mk_maps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice) ==
         cudaSuccess;
}

bool mk_ffn_fused_layout(const dec_config& c) {
  return c.weight_dtype == DEC_BF16 && !c.weight_quant && !decode_needs_rows(c) && c.hidden % MK_KG == 0 &&
         c.ffn % MK_FTS == 0;
}

// Fused FFN (bf16 weights, transposed down copy present): hidden in whole
// MK_KG-column blocks, ffn in MK_FTS-task steps (so no task block crosses an
// expert), at most MK_FT tasks per CTA and MK_MAX_NB partial rows.
bool mk_ffn_fused_ok(const Model& m, int nb) {
  const dec_config& c = m.cfg;
  if (m.wq8 || c.weight_dtype != DEC_BF16 || !m.layers || !m.layers[0].w_down_t || !m.s.fpart) return false;
  if (c.hidden % MK_KG != 0 || c.ffn % MK_FTS != 0 || nb < 1 || nb > MK_MAX_NB) return false;
  const int T = (c.n_experts ? c.n_experts_used : 1) * c.ffn;
  const int per = ((T + nb - 1) / nb + MK_FTS - 1) / MK_FTS * MK_FTS;
  return per <= MK_FT;
}

// dst[b][c][r] = src[b][r][c] for bf16 matrices of rows x cols (32 x 32 tiles
// through shared memory; both sides coalesced).
__global__ void __launch_bounds__(256) k_transpose_bf16(const __nv_bfloat16* __restrict__ src, int rows, int cols,
                                                        __nv_bfloat16* __restrict__ dst) {
  __shared__ __nv_bfloat16 t[32][34];
  const size_t mat = (size_t)rows * cols * blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32, tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + tx;
    if (r < rows && c < cols) t[i][tx] = src[mat + (size_t)r * cols + c];
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + tx;
    if (r < rows && c < cols) dst[mat + (size_t)c * rows + r] = t[tx][i];
  }
}

cudaError_t launch_transpose_bf16(const void* src, int rows, int cols, int batch, void* dst, cudaStream_t s) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return cudaSuccess;
  const dim3 grid((cols + 31) / 32, (rows + 31) / 32, batch);
  k_transpose_bf16<<<grid, 256, 0, s>>>((const __nv_bfloat16*)src, rows, cols, (__nv_bfloat16*)dst);
  return cudaGetLastError();
}

template <typename W, typename KV>
static void* mk_pick(int hd) {
  if (hd == 64) return (void*)k_decode_step<W, KV, 64>;
  if (hd == 128) return (void*)k_decode_step<W, KV, 128>;
  return (void*)k_decode_step<W, KV, 16>;
}

// The persistent step's instantiations: bf16 weights at every head_dim, f32
// weights only at head_dim 16 (the fp32 toy shape; larger f32 models keep the
// per-layer kernels), which keeps this file's build time in check.
static void* mk_func(const dec_config& c) {
  const bool wb = c.weight_dtype == DEC_BF16, kb = c.kv_dtype == DEC_BF16;
  if (c.kv_dtype == DEC_I8) return decode_kv_i8_persistent(c) ? (void*)k_decode_step<__nv_bfloat16, KVI8, 128> : nullptr;
  if (c.weight_quant) {
    if (!wb) return nullptr;   // 8-bit weights from f32 models decode on the row kernels
    return kb ? mk_pick<WQ8, __nv_bfloat16>(c.head_dim) : mk_pick<WQ8, float>(c.head_dim);
  }
  if (!wb) {
    if (c.head_dim != 16) return nullptr;
    return kb ? (void*)k_decode_step<float, __nv_bfloat16, 16> : (void*)k_decode_step<float, float, 16>;
  }
  if (kb) return mk_pick<__nv_bfloat16, __nv_bfloat16>(c.head_dim);
  return mk_pick<__nv_bfloat16, float>(c.head_dim);
}

// Whether the persistent step fits this configuration on this GPU; sets the
// kernel's shared-memory limit and the grid (one CTA per SM).
bool mk_prepare(Model& m, int num_sms) {
  const dec_config& c = m.cfg;
  const int es = c.weight_dtype == DEC_BF16 ? 2 : 4;
  m.mk_ok = false;
  m.mk_cluster = 0;
  (void)es;
  if (decode_needs_rows(c)) return false;   // served by the row kernels
  // Head dims 64 / 128 run the warp-task attention only.
  if ((c.head_dim == 64 || c.head_dim == 128) && !mk_attn_warp_ok(c)) return false;
  if (c.n_layers > MK_MAX_LAYERS) return false;   // the layer table travels in the kernel parameters
  // MoE down keeps one row sum per owned row (a CTA owns ceil(hidden / CTAs)
  // rows, in 16-row blocks on the tensor-core path); RoPE table of up to 64 pairs.
  auto rows_per_cta = [&](int nb) { return ((c.hidden + nb - 1) / nb + 15) / 16 * 16; };
  if (rows_per_cta(num_sms) > 256 || c.head_dim / 2 > 64) return false;
  if (!mk_build_maps(m)) return false;
  if (m.nsplit > 1 && m.attn_sps % MK_KS != 0) return false;
  const size_t smem = mk_smem_bytes(c, m.nsplit);
  if (smem > 227 * 1024) return false;
  void* fn = mk_func(c);
  if (!fn) return false;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return false;
  // The register split inside the kernel assumes exactly MK_REGS registers per thread at launch.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || fa.numRegs != MK_REGS) return false;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, MK_THREADS, smem) != cudaSuccess || per_sm < 1)
    return false;
  m.mk_smem = smem;
  m.mk_nb = num_sms;
  m.mk_ok = true;
  // One-cluster schedule: 16 CTAs (a non-portable size) or 8, if the GPU can
  // place such a cluster with this kernel's shared memory; the MoE row sums
  // need at most 256 residual rows per CTA.
  m.mk_cluster = 0;
  for (int cs = 16; cs >= 8; cs /= 2) {
    if (rows_per_cta(cs) > 256) break;
    if (cs > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(MK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, fn, &cfg) == cudaSuccess && nc >= 1) {
      m.mk_cluster = cs;
      break;
    }
    cudaGetLastError();
  }
  return true;
}

void launch_decode_mk(const Model& m, cudaStream_t s, const int32_t* d_token, int32_t token, int32_t pos,
                      float* logits, int32_t* d_argmax, bool cluster) {
  const dec_config& c = m.cfg;
  const Scratch& S = m.s;
  MkParams P;
  P.n_layers = c.n_layers;
  P.h = c.hidden;
  P.nq = c.n_heads;
  P.nkv = c.n_kv_heads;
  P.hd = c.head_dim;
  P.f = c.ffn;
  P.V = c.vocab;
  P.E = c.n_experts;
  P.k = c.n_experts ? c.n_experts_used : 1;
  P.max_seq = c.max_seq;
  P.sliding = c.sliding_window;
  P.nsplit = m.nsplit;
  P.sps = m.attn_sps;
  P.nb = cluster ? m.mk_cluster : m.mk_nb;
  P.cluster = cluster ? m.mk_cluster : 0;
  P.eps = c.rms_eps;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerPtrs& d = m.layers[l];
    P.layers[l] = MkLayer{d.attn_norm, d.wqkv,  d.bqkv, d.wo,     d.ffn_norm, d.w_gateup, d.w_down,
                          d.router,    d.kc,    d.vc,   d.q_norm, d.k_norm,   layer_rope_global(c, l) ? 0 : 1};
  }
  P.embed = m.tok_embd;
  P.out_norm = m.out_norm;
  P.head = m.head;
  P.st = S.st;
  P.inv_freq = S.inv_freq;
  P.inv_freq_local = S.inv_freq_local;
  P.x = S.x;
  P.q = S.q;
  P.attn = S.attn;
  P.act = S.act;
  P.part = S.part;
  P.amax_val = S.amax_val;
  P.amax_idx = S.amax_idx;
  P.ids_out = S.ids;
  P.logits = logits;
  P.d_argmax = d_argmax;
  P.d_token = d_token;
  P.token = token;
  P.pos = pos;
  P.trace_ids = m.trace_ids;
  P.trace_logits = m.trace_logits;
  P.trace_cap = m.trace_cap;
  P.u_bytes = (int)mk_u_bytes(c, m.nsplit);
  P.stamps = m.mk_stamps;
  P.kv_bytes = c.kv_dtype == DEC_BF16 ? 2 : c.kv_dtype == DEC_I8 ? 1 : 4;
  P.kv_cur = S.kv_cur;
  P.kv_code_off = c.kv_dtype == DEC_I8 ? kv_row_layout(c).code_off : 0;
  P.kv_row_bytes = kv_row_layout(c).bytes;
  P.qkn = decode_qkn_persistent(c) ? 1 : 0;
  P.maps = reinterpret_cast<const CUtensorMap*>(m.mk_maps);
  P.xs_floats = mk_xs_floats(c, m.nsplit);
  P.xb_plane = mk_xb_plane(c);
  P.attn_warp = mk_attn_warp_ok(c) ? 1 : 0;
  P.head_q8 = m.q_head.codes ? 1 : 0;
  P.fpart = S.fpart;
  P.ffn_fused = mk_ffn_fused_ok(m, P.nb) ? 1 : 0;
  // Warp-task attention merges each kv head's splits inside its own phase; the
  // CTA-task attention keeps a merge phase for large split sets.
  P.merge_phase = (!P.attn_warp && m.nsplit > 1 &&
                   (size_t)c.n_heads * m.nsplit * (c.head_dim + 2) * 4 > 64 * 1024) ? 1 : 0;
  P.attn_ns = (P.nb + c.n_kv_heads - 1) / c.n_kv_heads;
  if (P.attn_ns > 32) P.attn_ns = 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.nb);
  cfg.blockDim = dim3(MK_THREADS);
  cfg.dynamicSmemBytes = m.mk_smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.nb;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&P};
  timer_begin(m, DEC_K_STEP, s);
  cudaLaunchKernelExC(&cfg, mk_func(c), args);
  timer_end(m, DEC_K_STEP, s);
  count_launch(m);
}

}  // namespace dec
