// Self-test of the bounded device waits: a global flag that nothing sets and an mbarrier
// that nothing arrives on.  Both waits must give up after their limit, raise
// KVC_DEV_TIMEOUT and let the kernel return normally; the kernel records which of the
// two gave up.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

__device__ int g_never_set;    // nothing in the library ever writes it
__device__ int g_selftest_result;

__global__ void selftest_wait_kernel(uint32_t *status, unsigned long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    flag = 0;
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int result = 0;
    if (!spin_count_bounded(&g_never_set, 1, status, limit)) {
      set_status(status, KVC_DEV_TIMEOUT);
      result |= 1;
    }
    const Abort ab{&flag, status, limit};
    if (!ab.wait(b, 0)) result |= 2;  // phase 0 never completes
    g_selftest_result = result;
  }
  __syncthreads();
}

}  // namespace

// Runs the kernel and returns the bits of the waits that gave up (1 = flag, 2 = mbarrier)
// in *result (synchronises the stream).
cudaError_t run_selftest_wait(const Ctx &c, int *result) {
  selftest_wait_kernel<<<1, 32, 0, c.stream>>>(c.status, c.timeout_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(result, g_selftest_result, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                c.stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(c.stream);
}

}  // namespace kvc
