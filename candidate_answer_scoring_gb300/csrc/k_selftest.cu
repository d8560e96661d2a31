// Diagnostic: exercise the bounded device-side wait on a barrier that nothing
// ever completes, so that tests can check that a wait which runs out returns
// JET_ERR_TIMEOUT through the error word and leaves the context usable.
#include "jet_internal.cuh"
#include "jet_wait.cuh"

namespace jet {
namespace {

__global__ void wait_selftest_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    err[0] = 0;
    err[2] = 0;
    abort_flag = 0;
    mbar_init(&bar, 1);                       // expects one arrival that never comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, err, 99, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, unsigned long long limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace jet
