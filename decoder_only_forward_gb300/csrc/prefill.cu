// Prefill driver.
#include "runtime.h"

namespace dec {

// Positions are swept ascending, so each position's K/V is written before any
// later position reads it (sipllm "Transformer forward pass", Single-pass
// prefill).  This first driver runs the decode kernels once per position.
void launch_prefill_chunk(const Model& m, cudaStream_t s, int n, int start, float* logits,
                          int32_t* d_argmax) {
  for (int t = 0; t < n; ++t) {
    launch_set_step(m, s, m.s.tokens + t, 0, start + t);
    const bool last = t == n - 1;
    launch_decode_body(m, s, last ? logits : nullptr, last ? d_argmax : nullptr);
  }
}

}  // namespace dec
