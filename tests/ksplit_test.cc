// Host-only checks of the tensor-core GEMM's K-split choice (csrc/ksplit.h):
// it splits when a GEMM's tiles leave most SMs idle (few rows, the batched
// decode step), never when there are waves of tiles (prefill), never leaves a
// split empty, and respects the partial buffer.  Built and run by
// tests/test_ksplit.py; exits non-zero on a failure.
#include <cstdio>

#include "ksplit.h"

#define CHECK(c)                                                   \
  do {                                                             \
    if (!(c)) {                                                    \
      std::fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, #c); \
      return 1;                                                    \
    }                                                              \
  } while (0)

using dec::pick_ksplit;

static const int SMS = 152, BK = 64;
static const size_t CAP = (size_t)128 << 20;

static bool nonempty(int kblocks, int s) {
  const int per = (kblocks + s - 1) / s;
  return (kblocks + per - 1) / per == s;
}

int main() {
  // Mistral-7B projections with one 128-row tile (BN 256): N x K.
  const int shapes[][2] = {{6144, 4096}, {4096, 4096}, {28672, 4096}, {4096, 14336}, {32000, 4096}};
  for (auto& sh : shapes) {
    const int N = sh[0], K = sh[1], kb = K / BK;
    const long long tiles = (N + 255) / 256;
    const int s = pick_ksplit(tiles, kb, 256, BK, 128, N, CAP, SMS);
    std::printf("N=%d K=%d tiles=%lld -> ksplit %d\n", N, K, tiles, s);
    CHECK(s >= 1 && s <= 16 && nonempty(kb, s));
    if (tiles * 2 <= SMS) CHECK(s >= 2);        // at most half the SMs busy without a split
    // Batch invariance: the choice depends on the tile rows, the same for any B <= 128.
    CHECK(pick_ksplit(tiles, kb, 256, BK, 128, N, CAP, SMS) == s);
  }
  // Prefill: 4096 rows make 32 row tiles per weight block: waves of work, no split.
  CHECK(pick_ksplit(32LL * 24, 64, 256, BK, 4096, 6144, CAP, SMS) == 1);
  // A partial buffer too small for even two splits: none.
  CHECK(pick_ksplit(16, 64, 256, BK, 128, 4096, 128 * 4096 * 4, SMS) == 1);
  // Fewer K-blocks than the largest split: never more splits than K-blocks.
  CHECK(pick_ksplit(4, 3, 128, BK, 128, 512, CAP, SMS) <= 3);
  std::printf("ksplit ok\n");
  return 0;
}
