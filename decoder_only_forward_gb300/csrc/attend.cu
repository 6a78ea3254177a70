// Standalone attention entry point: the split-K flash-decode kernel of the
// decode step, callable on any KV ring (rml "The decoder", Attend).
#include <stdint.h>

#include "runtime.h"

namespace dec {

bool attend_check(const void* q, const void* k, const void* v, const void* out, int nq, int nkv, int hd,
                  int max_seq, int sliding, int kv_dtype, int pos, AttendLayout& lay, const char** why) {
  auto bad = [&](const char* m) { *why = m; return false; };
  if (!q || !k || !v || !out) return bad("q, k, v and out must be non-NULL");
  if ((((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out) & 15u) != 0)
    return bad("q, k, v and out must be 16-byte aligned");
  if (nq <= 0 || nkv <= 0 || max_seq <= 0 || pos < 0) return bad("sizes must be positive and pos >= 0");
  if (nq % nkv != 0 || nq / nkv > MAX_GROUP) return bad("n_heads must be a multiple of n_kv_heads, at most 16 per group");
  if (nkv > MAX_KV_HEADS) return bad("at most 192 kv heads");
  if (hd != 16 && hd != 64 && hd != 128) return bad("head_dim must be 16, 64 or 128");
  if (kv_dtype != DEC_F32 && kv_dtype != DEC_BF16) return bad("kv_dtype must be DEC_F32 or DEC_BF16");
  if (sliding < 0) return bad("sliding_window must be >= 0");
  if (sliding == 0 && pos >= max_seq) return bad("without a window pos must be < max_seq");
  if (sliding > 0 && max_seq > sliding) return bad("max_seq cannot exceed the window");
  // A ring shorter than the window cannot hold the window once it wraps: like a
  // handle's cache, it then holds positions below max_seq only.
  if (sliding > max_seq && pos >= max_seq) return bad("a ring shorter than the window holds pos < max_seq only");
  int nsplit = (max_seq + 127) / 128;
  const int cap = (2 * device_sm_count()) / nkv;   // about two CTAs per SM
  if (nsplit > cap) nsplit = cap;
  if (nsplit > 64) nsplit = 64;
  if (nsplit < 1) nsplit = 1;
  lay.nsplit = nsplit;
  lay.part_offset = (sizeof(DeviceState) + 255) / 256 * 256;
  lay.total = lay.part_offset + sizeof(float) * (size_t)nq * nsplit * (hd + 2);
  return true;
}

}  // namespace dec

using namespace dec;

extern "C" {

size_t dec_attend_scratch_bytes(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_seq) {
  AttendLayout lay;
  const char* why = nullptr;
  static const float dummy[4] = {0, 0, 0, 0};
  if (!attend_check(dummy, dummy, dummy, dummy, n_heads, n_kv_heads, head_dim, max_seq, 0, DEC_F32, 0, lay, &why))
    return 0;
  return lay.total;
}

dec_status dec_attend(const float* q, const void* k, const void* v, int32_t n_heads, int32_t n_kv_heads,
                      int32_t head_dim, int32_t max_seq, int32_t sliding_window, int32_t kv_dtype, int32_t pos,
                      float* out, void* scratch, size_t scratch_bytes, void* cuda_stream) {
  AttendLayout lay;
  const char* why = nullptr;
  if (!attend_check(q, k, v, out, n_heads, n_kv_heads, head_dim, max_seq, sliding_window, kv_dtype, pos, lay,
                    &why)) {
    set_global_error(why);
    return DEC_EINVAL;
  }
  if (!scratch || ((uintptr_t)scratch & 255u) != 0) {
    set_global_error("scratch must be non-NULL and 256-byte aligned");
    return DEC_EINVAL;
  }
  if (scratch_bytes < lay.total) {
    set_global_error("scratch is smaller than dec_attend_scratch_bytes()");
    return DEC_ENOMEM;
  }
  char* base = (char*)scratch;
  launch_attend(q, k, v, n_heads, n_kv_heads, head_dim, max_seq, sliding_window, kv_dtype, pos, lay.nsplit,
                (DeviceState*)base, (float*)(base + lay.part_offset), out, (cudaStream_t)cuda_stream);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_global_error(cudaGetErrorString(e));
    return DEC_ECUDA;
  }
  return DEC_OK;
}

}  // extern "C"
