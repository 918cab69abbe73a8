// Self-test of the bounded-wait path that every tcgen05/TMA kernel of this library uses: one
// CTA initialises an mbarrier that nothing ever arrives at and waits on it with mbar_wait and
// a caller-given limit.  The wait runs out, records DEV_ERR_TIMEOUT in the context's error
// word and returns; no copy or MMA is in flight, so the kernel simply exits.  This shows that
// a wait that gives up ends the kernel and reaches the host as MLA_ERR_TIMEOUT, with the
// context still usable, without making any real kernel lose its data.
#include "tc_common.cuh"

namespace mla {

namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, err, &abort_flag, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace mla
