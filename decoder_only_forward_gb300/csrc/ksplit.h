// Choice of the K split of the persistent tensor-core GEMM (gemm_tc.cu).
// Host-only C++, so a host test can drive it.
#pragma once

#include <stddef.h>

namespace dec {

// K splits for a GEMM whose tiles alone would leave SMs idle: the count that
// minimises (waves of units) x (K-blocks per unit) x (time of one weight
// K-block at an SM's share of HBM), plus the partial sums' round trip for
// s > 1, within the partial buffer.  rows: the rows the partial buffer holds
// per split.  A function of the GEMM's shape and the GPU only: for the same
// weights and tile rows every call takes the same split (and rounding).
inline int pick_ksplit(long long tiles, int kblocks, int BN, int BK, long long rows, int N, size_t cap_bytes, int sms) {
  const double bw = 6.0e12;                                    // bytes/s, a round HBM copy rate
  const double t_kb = (double)BN * BK * 2.0 / (bw / sms);    // one weight K-block on one SM
  double best_t = 0.0;
  int best = 1;
  for (int s = 1; s <= 16 && s <= kblocks; ++s) {
    const int kb_per = (kblocks + s - 1) / s;
    if ((kblocks + kb_per - 1) / kb_per != s) continue;         // a split would be empty
    const double part_bytes = (double)s * rows * N * 4.0;
    if (s > 1 && part_bytes > (double)cap_bytes) break;
    const long long units = tiles * s;
    double t = (double)((units + sms - 1) / sms) * kb_per * t_kb;
    if (s > 1) t += 2.0 * part_bytes / bw + 3e-6;               // partials out and back, one more launch
    if (s == 1 || t < 0.97 * best_t) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

}  // namespace dec
