// Self-test of the failure path every kernel's waits share: a bounded
// mbarrier wait that gives up, records KVP_ERR_DEVICE_TIMEOUT in the device
// status word and returns, leaving the context usable.  One thread waits on a
// shared-memory barrier with a 2 ms limit through the same wait the kernels
// use (their limit is 2 s).  With arrive set it arrives on the barrier first
// and the wait succeeds; otherwise nothing ever arrives and the wait expires.
// No fault, no trap, no unbounded loop.
#include "kvp_device.cuh"

namespace kvp {
namespace {

constexpr unsigned long long kSelftestWaitNs = 2000000ull;  // 2 ms

__global__ void __launch_bounds__(1) selftest_wait_kernel(int arrive, int* status) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (arrive) mbar_arrive(&bar);
  mbar_wait<kSelftestWaitNs>(&bar, 0, status);
}

}  // namespace

cudaError_t launch_selftest_wait(int arrive, int* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 1, 0, stream>>>(arrive ? 1 : 0, status);
  return cudaGetLastError();
}

}  // namespace kvp
