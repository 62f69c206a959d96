// dsa_selftest_wait_timeout: the bounded-wait abort path, run on purpose.
//
// Every pipeline of the library (the scorer's TMA ring, the attention pair's
// exchange, the top-k's staged chunk copy) waits on mbarriers through
// ptx::mbar_wait, which gives up after a poll limit instead of spinning for
// ever; the kernel then ORs DSA_DEVERR_TIMEOUT into the workspace's error word
// and unwinds. On valid inputs no wait ever runs out, so this entry point makes
// one run out: a single warp waits on an mbarrier that nothing arrives on, with
// a short poll limit, and reports through the same helper and the same error
// word. Nothing asynchronous is in flight (no copy, no MMA, no tensor memory),
// so the kernel returns with the context and the workspace usable.
#include "dsa_internal.cuh"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t* err, uint32_t poll_limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // Phase 0 of `bar` needs one arrival and gets none: the wait gives up.
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, poll_limit)) atomicOr(err, DSA_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status_t dsa_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t poll_limit,
                                                  cudaStream_t stream) {
  if (!ws || ws_bytes < sizeof(int32_t) || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return DSA_ERR_INVALID;
  if (poll_limit == 0 || poll_limit > (1u << 20)) return DSA_ERR_INVALID;
  dsa::wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<int32_t*>(ws), poll_limit);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
