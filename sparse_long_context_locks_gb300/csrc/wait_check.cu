// wait_check.cu -- locks_check_bounded_wait: a diagnostic launch that makes
// the library's bounded mbarrier wait run out, so a test can see the timeout
// reported without any fault.
//
// The kernel runs mbar_wait (common.cuh), the same bounded wait every decode
// kernel uses, on a barrier that waits for two arrivals and gets one: the
// phase never completes, the wait gives up after the caller's limit and
// records LOCKS_FLAG_TIMEOUT in the status word.  Before returning, the kernel
// waits (with the default one-second bound) for the one bulk copy it issued,
// so no copy is in flight into shared memory when the CTA exits.

#include <cstdint>

#include "../../include/locks.h"
#include "common.cuh"

namespace locks {
namespace {

constexpr int kCheckBytes = 256;

__global__ void __launch_bounds__(32) wait_check_kernel(const uint8_t* src, uint32_t* result, uint32_t* status,
                                                        uint64_t limit_ns) {
  __shared__ __align__(128) uint8_t buf[kCheckBytes];
  __shared__ uint64_t bar_copy, bar_never;
  const int lane = threadIdx.x;
  if (lane == 0) {
    mbar_init(&bar_copy, 1);
    mbar_init(&bar_never, 2);
    fence_mbar_init();
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive_expect_tx(&bar_copy, kCheckBytes);
    bulk_g2s(buf, src, kCheckBytes, &bar_copy);
    mbar_arrive(&bar_never);   // one of the two arrivals this barrier waits for
  }
  __syncwarp();
  const bool never = mbar_wait(&bar_never, 0, status, limit_ns);
  const uint64_t t_gave_up = globaltimer_ns();
  const bool copied = mbar_wait(&bar_copy, 0, status);
  uint32_t sum = 0;
  if (copied) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(buf);
    sum = w[lane] + w[lane + 32];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) {
    result[0] = never ? 0u : 1u;     // 1: the never-completing wait ran out
    result[1] = copied ? 1u : 0u;    // 1: the issued copy landed before exit
    result[2] = sum;                 // sum of the 64 copied words
    result[3] = (uint32_t)(t_gave_up & 0xffffffffu);
  }
}

}  // namespace
}  // namespace locks

extern "C" locks_status locks_check_bounded_wait(const void* src, uint32_t* result, uint32_t limit_us,
                                                 void* workspace, size_t workspace_bytes,
                                                 locks_stream_t stream) {
  using namespace locks;
  if (src == nullptr || result == nullptr || workspace == nullptr) return LOCKS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0 || (reinterpret_cast<uintptr_t>(result) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 || workspace_bytes < sizeof(uint32_t))
    return LOCKS_ERR_INVALID_ARG;
  if (limit_us == 0 || limit_us > 100000) return LOCKS_ERR_INVALID_ARG;   // 1 us .. 100 ms
  wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(src), result, static_cast<uint32_t*>(workspace), (uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}
