// StreamingLLM ring append (StreamingLLM article, キャッシュ構造 and 推論の流れ): token
// t's key/value goes to row t while t < S (the sink tokens, never overwritten), then to
// ring row S + (t - S) mod R, overwriting the oldest recent token.  The row index is the
// same for every unit and is computed on the host; one warp copies one unit's rows.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

__global__ void sink_append_kernel(const uint4 *k_new, const uint4 *v_new, uint4 *kc, uint4 *vc,
                                   int32_t *pos, int rows, int rv, int slot, int32_t t32) {
  const int u = blockIdx.x;
  const int lane = threadIdx.x;
  const size_t dst = ((size_t)u * rows + slot) * rv;
  for (int e = lane; e < rv; e += 32) {
    kc[dst + e] = k_new[(size_t)u * rv + e];
    vc[dst + e] = v_new[(size_t)u * rv + e];
  }
  if (lane == 0 && pos) pos[(size_t)u * rows + slot] = t32;
}

}  // namespace

cudaError_t launch_sink_append(const Ctx &c, const void *k_new, const void *v_new, void *k_cache,
                               void *v_cache, int32_t *pos, int units, int D, int rows, int slot,
                               int64_t t) {
  sink_append_kernel<<<units, 32, 0, c.stream>>>(
      reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
      reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), pos, rows, D / 8,
      slot, (int32_t)t);
  return cudaGetLastError();
}

}  // namespace kvc
