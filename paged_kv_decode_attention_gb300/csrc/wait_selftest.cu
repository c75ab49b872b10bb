// wait_selftest.cu -- pkv_selftest_bounded_wait: a check of the kernels'
// fail-fast path.
//
// Every pipeline wait in libpkv gives up after a wall-time limit and sets
// PKV_DEVERR_TIMEOUT instead of hanging the GPU.  In a healthy kernel no wait
// ever comes near that limit, so ordinary calls cannot show that the path
// works.  This entry point runs the same bounded wait (mbar_wait_limited, the
// helper behind every kernel's mbar_wait) in a one-CTA kernel with the
// producer/consumer shape of the decode kernels: a producer warp arms the
// ring's stage 0 and, unless asked to, never stage 1; the consumer warp waits
// for both with the caller's short limit.  The wait on the unarmed stage then
// runs out, the consumer records PKV_DEVERR_TIMEOUT and the kernel returns
// normally: nothing is in flight (no bulk copy or TMA is issued), and the
// CUDA context stays usable for the next call.
#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_common.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(64) bounded_wait_selftest_kernel(uint64_t limit_ns, int arm_all,
                                                                   unsigned int* err) {
  __shared__ __align__(8) uint64_t full_bar[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 1) {
    // producer: stage 0 always, stage 1 only when asked
    if (lane == 0) {
      mbar_arrive(&full_bar[0]);
      if (arm_all) mbar_arrive(&full_bar[1]);
    }
  } else if (lane == 0) {
    // consumer: both stages, each wait bounded by the caller's limit
    bool ok = mbar_wait_limited(&full_bar[0], 0, limit_ns);
    if (ok) ok = mbar_wait_limited(&full_bar[1], 0, limit_ns);
    if (!ok) report(err, PKV_DEVERR_TIMEOUT);
  }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_selftest_bounded_wait(uint32_t wait_limit_us, int32_t arm_all, void* stream) {
  if (wait_limit_us == 0 || wait_limit_us > 1000000u) return PKV_ERR_SHAPE;
  unsigned int* err = pkv::device_error_word();
  if (err == nullptr) return PKV_ERR_CUDA;
  pkv::bounded_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(wait_limit_us) * 1000ull, arm_all != 0, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
