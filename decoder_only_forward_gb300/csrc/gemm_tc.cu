// Prefill projection GEMM on the 5th-generation tensor cores:
//   C[M,N] = A[M,K] . B[N,K]^T, bf16 operands, f32 accumulation in TMEM.
// A (activations) may be given as a bf16 pair (hi, lo) with A = hi + lo; the
// kernel then issues two MMAs per K step so the product keeps ~16 bits of the
// activations' mantissa (bf16 weights with fp32 activations and accumulation).
//
// Persistent: one CTA per SM walks 128 x BN output tiles (tile t, t + grid,
// ...), ordered so that CTAs running at the same time share weight columns
// (B) in L2.  When there are too few tiles to occupy the SMs (few rows, the
// batched decode step), K is split into ksplit ranges: unit t is K range
// t % ksplit of tile t / ksplit, its raw f32 sum goes to a partial buffer, and
// k_splitk_epi adds the ranges in order and applies the epilogue.  Three warp
// roles:
//   warp 0 lane 0: TMA producer, K-blocks of 64 into a ring of smem stages;
//   warp 1 lane 0: MMA issuer (tcgen05.mma, cta_group::1), frees stages with
//                  tcgen05.commit, alternates between two TMEM accumulators;
//                  warp 1 also owns the TMEM allocation;
//   warps 2-5:     epilogue of the previous tile while the next one
//                  accumulates: tcgen05.ld of 32 rows x 32 columns per warp,
//                  a transpose through the warp's own smem slice, then the
//                  fused epilogue with consecutive lanes on consecutive
//                  column pairs (coalesced stores).
#include <cudaTypedefs.h>

#include <mutex>

#include "ksplit.h"
#include "prefill_common.cuh"
#include "tc.cuh"

namespace dec {

constexpr int TC_BM = 128, TC_BK = 64, TC_THREADS = 192;

template <int BN, bool SPLIT>
struct TcCfg {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;
  static constexpr int B_BYTES = BN * TC_BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES * (SPLIT ? 2 : 1) + B_BYTES;
  static constexpr int EPI_LD = 33;                          // floats per staged row
  static constexpr int EPI_BYTES = 4 * 32 * EPI_LD * 4;      // one 32 x 32 slice per epilogue warp
  static constexpr int BAR_BYTES = 256 + 1280;   // barriers and flags, then the grouped tile prefix
  static constexpr int STAGES_FIT = (232448 - 1024 - EPI_BYTES - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int SMEM = STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES + 1024;
  static constexpr int TMEM_COLS = 2 * BN;                   // two accumulators
};

template <int BN, bool SPLIT>
__global__ void __launch_bounds__(TC_THREADS, 1) k_gemm_tc(const __grid_constant__ CUtensorMap tm_ahi,
                                                           const __grid_constant__ CUtensorMap tm_alo,
                                                           const __grid_constant__ CUtensorMap tm_b, int M, int N,
                                                           int K, GemmEpi e, int groups, int m_tiles, int ksplit,
                                                           float* __restrict__ kpart, DeviceState* st) {
  using C = TcCfg<BN, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* epi_smem = reinterpret_cast<float*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES + C::EPI_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;   // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2]
  uint64_t* drained = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* progress = abort_flag + 1;  // [0] K-blocks issued, [1] K-blocks consumed
  // Grouped GEMM: tile_pref[g] = row tiles of groups before g (the rows of group g
  // are [offset[g], offset[g+1]), known on the device only).
  int* tile_pref = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(full) + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (N + BN - 1) / BN;
  const int kblocks = (K + TC_BK - 1) / TC_BK;
  const int kb_per = (kblocks + ksplit - 1) / ksplit;   // every split non-empty (host's choice)
  if (e.group_offset && threadIdx.x == 32) {
    int acc = 0;
    for (int g = 0; g < groups; ++g) {
      tile_pref[g] = acc;
      const int rg = e.group_offset[g + 1] - e.group_offset[g];
      acc += min(m_tiles, (max(rg, 0) + TC_BM - 1) / TC_BM);
    }
    tile_pref[groups] = acc;
  }
  __syncthreads();
  // Row tiles sharing one BN block of weight rows: only tiles that hold rows are
  // enumerated, so the persistent CTAs split the real work evenly.
  const int per_n = e.group_offset ? tile_pref[groups] : m_tiles;
  const int total = n_tiles * per_n * ksplit;
  // Unit u -> (K range u % ksplit of) tile (group, 128-row block, BN-column
  // block), the same answer for every role.
  auto decode_tile = [&](int u, int& row0, int& rows, int& b_row0, int& m0, int& n0) -> bool {
    const int t = u / ksplit;
    const int nb = t / per_n, rem = t % per_n;
    int g = 0, mb = rem;
    row0 = 0;
    rows = M;
    b_row0 = 0;
    if (e.group_offset) {
      while (g + 1 < groups && tile_pref[g + 1] <= rem) ++g;
      mb = rem - tile_pref[g];
      row0 = e.group_offset[g];
      rows = e.group_offset[g + 1] - row0;
      b_row0 = g * N;
    }
    m0 = mb * TC_BM;
    n0 = nb * BN;
    return m0 < rows;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);   // one arrival per epilogue warp
    }
    mbar_init(drained, 1);
    *abort_flag = 0;
    progress[0] = 0;
    progress[1] = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tm_ahi);
    if (SPLIT) tma_prefetch_desc(&tm_alo);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int kb_all = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int row0, rows, b_row0, m0, n0;
        if (!decode_tile(t, row0, rows, b_row0, m0, n0)) continue;
        const int kb0 = (t % ksplit) * kb_per, kb1 = min(kblocks, kb0 + kb_per);
        for (int kb = kb0; kb < kb1; ++kb, ++kb_all) {
          const int s = kb_all % C::STAGES;
          const uint32_t ph = (kb_all / C::STAGES) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, st, 101)) {
            ok = false;
            break;
          }
          uint8_t* base = smem + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_2d(base, &tm_ahi, &full[s], kb * TC_BK, row0 + m0);
          if (SPLIT) tma_load_2d(base + C::A_BYTES, &tm_alo, &full[s], kb * TC_BK, row0 + m0);
          tma_load_2d(base + C::A_BYTES * (SPLIT ? 2 : 1), &tm_b, &full[s], kb * TC_BK, b_row0 + n0);
          progress[0] = kb_all + 1;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
      int kb_all = 0, it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int row0, rows, b_row0, m0, n0;
        if (!decode_tile(t, row0, rows, b_row0, m0, n0)) continue;
        const int b = it & 1;
        // The epilogue must have drained this accumulator (tile it - 2).
        if (!mbar_wait(&acc_empty[b], ((it >> 1) & 1) ^ 1, abort_flag, st, 104)) break;
        tc_fence_after();
        const uint32_t acc = tmem + b * BN;
        const int kb0 = (t % ksplit) * kb_per, kb1 = min(kblocks, kb0 + kb_per);
        for (int kb = kb0; kb < kb1; ++kb, ++kb_all) {
          const int s = kb_all % C::STAGES;
          const uint32_t ph = (kb_all / C::STAGES) & 1;
          if (!mbar_wait(&full[s], ph, abort_flag, st, 102)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* base = smem + s * C::STAGE_BYTES;
          const uint64_t da = sw128_kmajor_desc(smem_u32(base));
          const uint64_t dl = sw128_kmajor_desc(smem_u32(base + C::A_BYTES));
          const uint64_t db = sw128_kmajor_desc(smem_u32(base + C::A_BYTES * (SPLIT ? 2 : 1)));
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k) {
            tc_mma_bf16(acc, da + 2 * k, db + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            if (SPLIT) tc_mma_bf16(acc, dl + 2 * k, db + 2 * k, idesc, 1u);
          }
          tc_commit(&empty[s]);
          progress[1] = kb_all + 1;
        }
        if (!ok) break;
        tc_commit(&acc_full[b]);
        ++it;
      }
      // Every MMA issued here completes before the TMEM goes back.
      tc_commit(drained);
      volatile int no_abort = 0;
      mbar_wait(drained, 0, &no_abort, nullptr, 0, 100000000ull);
    }
  } else {
    // tcgen05.ld is warp-collective: every branch around it is warp-uniform.
    const int q = warp & 3;
    float* slice = epi_smem + q * 32 * C::EPI_LD;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int row0, rows, b_row0, m0, n0;
      if (!decode_tile(t, row0, rows, b_row0, m0, n0)) continue;
      const int b = it & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[b], (it >> 1) & 1, abort_flag, st, 103))) break;
      tc_fence_after();
      const uint32_t acc = tmem + b * BN + lane_base;
      const int r_base = m0 + q * 32;          // this warp's first row within the group
      float* kp = ksplit > 1 ? kpart + (size_t)(t % ksplit) * M * N : nullptr;
      // A warp whose 32 rows are all past the tile's rows (a batch of few rows)
      // only keeps the accumulator hand-off in step.
      const bool idle = r_base >= rows;
#pragma unroll 1
      for (int c = 0; c < BN && !idle; c += 32) {
        if (n0 + c >= N) break;
        float v[32];
        tmem_ld32(acc + c, v);
        // Row `lane` of the slice <- this lane's accumulator row.
#pragma unroll
        for (int j = 0; j < 32; ++j) slice[lane * C::EPI_LD + j] = v[j];
        __syncwarp();
        // Lanes 0-15: row rr, lanes 16-31: row rr + 1; column pair (lane & 15).
        const int pc = 2 * (lane & 15);
#pragma unroll 4
        for (int rr = 0; rr < 32; rr += 2) {
          const int lr = rr + (lane >> 4);
          if (r_base + lr < rows) {
            const int row = row0 + r_base + lr, col = n0 + c + pc;
            if (kp) {
              float* d = kp + (size_t)row * N + col;
              const float v0 = slice[lr * C::EPI_LD + pc], v1 = slice[lr * C::EPI_LD + pc + 1];
              if ((N & 1) == 0) {
                if (col < N) *reinterpret_cast<float2*>(d) = make_float2(v0, v1);
              } else if (col < N) {
                d[0] = v0;
                if (col + 1 < N) d[1] = v1;
              }
            } else {
              epi_pair(e, row, col, slice[lr * C::EPI_LD + pc], slice[lr * C::EPI_LD + pc + 1]);
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Never taken when the pipeline is consistent.  Let the copies in flight
    // land (bounded) before the shared memory is released.
    volatile int no_abort = 0;
    if (threadIdx.x == 0)
      for (int kb = progress[1]; kb < progress[0]; ++kb)
        mbar_wait(&full[kb % C::STAGES], (kb / C::STAGES) & 1, &no_abort, nullptr, 0, 100000000ull);
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Sum of the ksplit partial products of every (row, column pair), in split
// order, then the GEMM's epilogue.
__global__ void __launch_bounds__(256) k_splitk_epi(const float* __restrict__ part, int ksplit, int M, int N,
                                                    GemmEpi e) {
  const int half = (N + 1) >> 1;
  const size_t pairs = (size_t)M * half, plane = (size_t)M * N;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < pairs; i += (size_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / half), col = 2 * (int)(i % half);
    const bool two = col + 1 < N;
    const float* p = part + (size_t)row * N + col;
    float a0 = p[0], a1 = two ? p[1] : 0.f;
    for (int z = 1; z < ksplit; ++z) {
      a0 += p[z * plane];
      if (two) a1 += p[z * plane + 1];
    }
    epi_pair(e, row, col, a0, a1);
  }
}

// The planes' products summed in order, then the epilogue (8-bit weights: the
// weight's hi and lo planes were multiplied separately).
cudaError_t launch_sum_planes_epi(const float* part, int planes, int M, int N, const GemmEpi& e, cudaStream_t s) {
  const long long pairs = (long long)M * ((N + 1) / 2);
  long long blocks = (pairs + 255) / 256;
  const long long cap = 8LL * device_sm_count();
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  k_splitk_epi<<<(int)blocks, 256, 0, s>>>(part, planes, M, N, e);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// A [rows, cols] bf16 row-major matrix, tiles of box_rows x 64, 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)TC_BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() { return device_sm_count(); }

template <int BN, bool SPLIT>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& al, const CUtensorMap& b, int M, int N, int K,
                             const GemmEpi& e, int groups, int max_rows, float* kpart, size_t kpart_bytes,
                             DeviceState* st, cudaStream_t s) {
  using C = TcCfg<BN, SPLIT>;
  auto kern = k_gemm_tc<BN, SPLIT>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  const int m_tiles = (max_rows + TC_BM - 1) / TC_BM;
  const long long tiles = (long long)m_tiles * groups * ((N + BN - 1) / BN);
  const int sms = num_sms();
  const int kblocks = (K + TC_BK - 1) / TC_BK;
  // Grouped GEMMs keep all M rows per split; plain ones a whole number of row tiles.
  const long long rows = groups > 1 ? (long long)M : (long long)m_tiles * TC_BM;
  const int ksplit = kpart ? pick_ksplit(tiles, kblocks, BN, TC_BK, rows, N, kpart_bytes, sms) : 1;
  const long long total = tiles * ksplit;
  const int grid = (int)(total < sms ? total : sms);
  kern<<<grid, TC_THREADS, C::SMEM, s>>>(a, al, b, M, N, K, e, groups, m_tiles, ksplit, kpart, st);
  if (ksplit > 1) {
    const long long pairs = (long long)M * ((N + 1) / 2);
    long long blocks = (pairs + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    k_splitk_epi<<<(int)blocks, 256, 0, s>>>(kpart, ksplit, M, N, e);
  }
  return cudaGetLastError();
}

// A (hi plane, optional lo plane): [a_rows, K] bf16; B: [groups * N, K] bf16.
// Grouped when e.group_offset is set (max_rows bounds any one group's rows).
// kpart (nullable): f32 scratch of kpart_bytes for split-K partial sums.
cudaError_t launch_gemm_tc(const void* a_hi, const void* a_lo, int a_rows, const void* b, int M, int N, int K,
                           const GemmEpi& e, int groups, int max_rows, float* kpart, size_t kpart_bytes,
                           DeviceState* st, cudaStream_t s) {
  if (K % 8 != 0 || a_rows <= 0 || N <= 0) return cudaErrorInvalidValue;
  const int bn = N >= 1536 ? 256 : 128;
  CUtensorMap ma, ml, mb;
  if (!make_map(&ma, a_hi, (uint64_t)a_rows, (uint64_t)K, TC_BM)) return cudaErrorInvalidValue;
  if (a_lo && !make_map(&ml, a_lo, (uint64_t)a_rows, (uint64_t)K, TC_BM)) return cudaErrorInvalidValue;
  if (!a_lo) ml = ma;
  if (!make_map(&mb, b, (uint64_t)N * groups, (uint64_t)K, (uint32_t)bn)) return cudaErrorInvalidValue;
  if (bn == 256)
    return a_lo ? launch_tc<256, true>(ma, ml, mb, M, N, K, e, groups, max_rows, kpart, kpart_bytes, st, s)
                : launch_tc<256, false>(ma, ml, mb, M, N, K, e, groups, max_rows, kpart, kpart_bytes, st, s);
  return a_lo ? launch_tc<128, true>(ma, ml, mb, M, N, K, e, groups, max_rows, kpart, kpart_bytes, st, s)
              : launch_tc<128, false>(ma, ml, mb, M, N, K, e, groups, max_rows, kpart, kpart_bytes, st, s);
}

}  // namespace dec

using namespace dec;

// C = (A_hi + A_lo) . B^T through the tensor-core kernel (C f32, row-major).
extern "C" dec_status dec_gemm_bf16(const void* a_hi, const void* a_lo, const void* b, float* c, int32_t m,
                                    int32_t n, int32_t k, void* cuda_stream) {
  if (!a_hi || !b || !c || m <= 0 || n <= 0 || k <= 0) {
    set_global_error("dec_gemm_bf16: NULL pointer or non-positive size");
    return DEC_EINVAL;
  }
  if (k % 8 != 0 || n % 2 != 0 || (((uintptr_t)a_hi | (uintptr_t)b | (uintptr_t)(a_lo ? a_lo : a_hi)) & 15u)) {
    set_global_error("dec_gemm_bf16: k must be a multiple of 8, n even, operands 16-byte aligned");
    return DEC_EINVAL;
  }
  GemmEpi e{};
  e.mode = EPI_STORE;
  e.n_out = n;
  e.out_f32 = c;
  const cudaError_t err =
      launch_gemm_tc(a_hi, a_lo, m, b, m, n, k, e, 1, m, nullptr, 0, nullptr, (cudaStream_t)cuda_stream);
  if (err != cudaSuccess) {
    set_global_error(cudaGetErrorString(err));
    return DEC_ECUDA;
  }
  return DEC_OK;
}
