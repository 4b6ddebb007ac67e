// selftest.cu -- device-side check of the bounded wait used by the bulk-copy
// kernel: a CTA waits on an mbarrier that nothing will ever complete and must
// give up after the limit, record the timeout in the error word and return.
#include "ssu_launch.cuh"

namespace ssu {
namespace {

__global__ void bounded_wait_probe(uint64_t limit_ns, unsigned* err,
                                   unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint64_t t0 = global_ns();
  const bool done = mbar_wait_for(&bar, 0, limit_ns);
  const uint64_t t1 = global_ns();
  __syncthreads();
  if (threadIdx.x == 0) {
    *waited_ns = (unsigned long long)(t1 - t0);
    if (!done) atomicOr(err, kErrFullTimeout);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_probe(uint64_t limit_ns, unsigned long long* waited_ns,
                                      cudaStream_t stream) {
  unsigned* err = device_error_word();
  if (!err) return cudaErrorInvalidSymbol;
  bounded_wait_probe<<<1, 32, 0, stream>>>(limit_ns, err, waited_ns);
  return cudaGetLastError();
}

}  // namespace ssu
