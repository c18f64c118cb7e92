// compressed_decode_attn_noalloc: the decode-attention entry point for callers that
// cannot hand this library a device workspace.  A serving engine that owns all device
// memory through its own pool passes only the tensors of the step down to the
// attention call; it has no allocator to give us, and a cudaMalloc in the middle of a
// decode step would also synchronise the device.  This entry point therefore keeps the
// split-K scratch (per-unit counters and partial results) in a fixed device array of
// this file, which every GPU that loads the library holds until the process exits.
//
// * The array is KVC_NOALLOC_SCRATCH_BYTES (8 MiB).  A call whose scratch need
//   (compressed_decode_attn_workspace_bytes) is larger is rejected with
//   KVC_ERR_WORKSPACE before anything is launched.
// * Host code cannot use the array's name as a device address.  The first call on a
//   device looks the address up with cudaGetSymbolAddress, with that device current,
//   and caches it; that first call should therefore come before any stream capture.
// * Every call shares the array.  Once its arguments have passed every check, each call
//   clears the counters it will use before its launch, so a call starts clean even after
//   an earlier one gave up on a wait; a rejected call leaves the array untouched.  Calls
//   that overlap on the GPU (other streams, other threads) race on the array: order them.
// * Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "kvc_internal.cuh"

#define KVC_NOALLOC_SCRATCH_BYTES (8u << 20)

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVC_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_ptr[64];

// Device address of the scratch array on the current device (looked up once per device,
// after the device has been found supported).  A failed lookup clears CUDA's last error
// so that the caller's own error checks do not see it.
kvc_status scratch_address(kvc_stream_t stream, void **out) {
  const kvc_status st = kvc::device_check(stream);
  if (st != KVC_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) {
      (void)cudaGetLastError();
      return KVC_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" kvc_status compressed_decode_attn_noalloc(const kvc_decode_params *p, const void *q,
                                                     const void *k_new, const void *v_new,
                                                     void *k_cache, void *v_cache, int32_t *pos,
                                                     int32_t *n_valid, void *out,
                                                     kvc_stream_t stream) {
  const kvc::TraceRange trace_range("compressed_decode_attn_noalloc");
  if (!p) return KVC_ERR_NULL;
  const size_t need = compressed_decode_attn_workspace_bytes(p);
  if (need > KVC_NOALLOC_SCRATCH_BYTES) return KVC_ERR_WORKSPACE;
  void *scratch = nullptr;
  const kvc_status st = scratch_address(stream, &scratch);
  if (st != KVC_OK) return st;
  // every argument check of the decode runs first; only then are the split-K counters
  // at the start of the scratch cleared, right before the launch
  return kvc::decode_call(p, q, k_new, v_new, k_cache, v_cache, pos, n_valid, out, scratch,
                          KVC_NOALLOC_SCRATCH_BYTES, stream, true);
}
