// Failure-detection self-test: makes the kernels' bounded mbarrier waits run out on purpose,
// on a barrier that nothing arrives at, so that the timeout path (error word, host status,
// a context that stays usable) can be checked without any fault.
#include <cuda_runtime.h>

#include "paged_attn.h"
#include "pa_kernels.h"
#include "pa_tc.cuh"

static_assert(pa::kWaitLimit == PA_WAIT_LIMIT && pa::kSpinLimit == PA_SPIN_LIMIT,
              "the header states the limits the kernels use");

namespace pa {
namespace {

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// One warp.  helper 0: mbar_wait (the decode kernels' wait); helper 1: wait_or_abort (the
// tcgen05 kernels' wait, which records the timeout itself); helper 2: a loop of
// non-suspending probes, the form of the tensor-core issuers' idle loops.  Writes the wall time
// the wait took to *elapsed_ns.
__global__ void __launch_bounds__(32) wait_selftest_kernel(int helper, uint32_t polls, unsigned* err,
                                                           unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);  // one arrival expected; none ever comes
  fence_mbar_init();
  abort_flag = 0u;
  const unsigned long long t0 = global_ns();
  bool ok;
  if (helper == 0) {
    ok = mbar_wait(b, 0, polls);
    if (!ok) record_error(err, kErrTimeout);
  } else if (helper == 1) {
    ok = wait_or_abort(b, 0, &abort_flag, err, polls);
  } else {
    ok = false;
    for (uint32_t it = 0; it < polls && !ok; ++it) ok = mbar_test_wait(b, 0);
    if (!ok) record_error(err, kErrTimeout);
  }
  const unsigned long long t1 = global_ns();
  *elapsed_ns = ok ? 0ull : (t1 - t0);
}

}  // namespace
}  // namespace pa

extern "C" int paged_attn_selftest_wait(int helper, unsigned int polls, unsigned long long* elapsed_ns,
                                        void* stream) {
  if (helper < 0 || helper > 2 || !elapsed_ns) return PA_ERR_INVALID_ARG;
  if (polls < 1 || polls > (helper == 2 ? pa::kSpinLimit : pa::kWaitLimit)) return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(elapsed_ns) % 8 != 0) return PA_ERR_INVALID_ARG;
  unsigned* err = nullptr;
  if (pa::error_word_address(&err) != cudaSuccess) return PA_ERR_CUDA;
  pa::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(helper, polls, err, elapsed_ns);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
