// Self-test of the device-side failure path shared by the pipelined kernels: a bounded
// mbarrier wait that runs out, the abort flag that releases the other waiting roles,
// and the timeout bit in the workspace status word that the host then reads. The
// kernel is a two-role pipeline whose barriers nothing ever arrives on, so every wait
// in it runs out, without a fault: the same helpers as the grouped GEMM and the gate
// (mbar_wait with its wall-clock limit kWaitLimitNs), nothing else.
#include <cstdint>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(int32_t* status) {
  __shared__ uint64_t full_bar, empty_bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&full_bar, 1);
    mbar_init(&empty_bar, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort = &s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    // Producer: waits for its first slot to be released (parity 0 of a fresh barrier,
    // which completes only on an arrival that never comes). After kWaitLimitNs it sets
    // the timeout bit and the abort flag, as the grouped GEMM's roles do.
    if (!mbar_wait(&empty_bar, 0, abort)) {
      *abort = 1;
      atomicOr(status, MOE_DEVICE_FLAG_TIMEOUT);
    }
  } else if (warp == 1 && lane == 0) {
    // Consumer: starts waiting for data half a limit later, so its own limit would run
    // out half a limit after the producer's; the abort flag ends its wait first.
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kWaitLimitNs / 2) __nanosleep(1000000);
    const uint64_t t1 = globaltimer_ns();
    const bool got = mbar_wait(&full_bar, 0, abort);
    // status[1]: 1 when the wait ended through the abort flag before its own limit.
    if (!got && globaltimer_ns() - t1 < kWaitLimitNs) atomicOr(status + 1, 1);
  }
  __syncthreads();
}

}  // namespace

moe_status launch_wait_selftest(int32_t* status, cudaStream_t s) {
  wait_selftest_kernel<<<1, 64, 0, s>>>(status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe
