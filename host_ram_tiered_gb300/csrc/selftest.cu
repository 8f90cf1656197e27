// kvo_selftest_wait_timeout: the library's bounded barrier wait, run on a
// barrier that nothing completes, so that its failure path -- give up after
// the limit, set kErrWaitTimeout, return -- can be tested without a fault.
#include "kvo_internal.cuh"
#include "sync.cuh"

namespace kvo {

namespace {

__global__ void wait_timeout_kernel(uint32_t *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);                      // one arrival completes phase 0; none comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, err, limit_ns);
}

}  // namespace

}  // namespace kvo

using namespace kvo;

extern "C" int kvo_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
  clear_error();
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fail(KVO_ERR_ARG, "kvo_selftest_wait_timeout: limit_ns must be in (0, 10 s]");
  uint32_t *err = device_error_word();
  if (!err) return fail(KVO_ERR_CUDA, "kvo_selftest_wait_timeout: device error word unavailable");
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, limit_ns);
  return cuda_status(cudaGetLastError(), "kvo_selftest_wait_timeout launch");
}
