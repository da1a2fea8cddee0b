// Self-test of the bounded mbarrier wait that every kernel of the library uses
// when it waits for staged data: a wait that is never satisfied must give up
// after its poll limit, report KVQ_DEVERR_TIMEOUT and let the kernel return,
// leaving the context usable.  Nothing is copied while it waits.
#include "kvq_common.cuh"
#include "kvq_internal.h"

namespace kvq {

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Two warps wait on one mbarrier (expected arrivals: 1).  With `arrive`, thread
// 0 arrives first and the wait succeeds; without, nothing ever arrives and the
// wait gives up after max_polls polls.
__global__ void bounded_wait_kernel(int32_t* error_flags, uint32_t max_polls, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  const bool ok = mbar_wait(&bar, 0, max_polls);
  if (!ok && (threadIdx.x & 31) == 0) atomicOr(error_flags, KVQ_DEVERR_TIMEOUT);
}

}  // namespace kvq

extern "C" kvq_status kvq_selftest_bounded_wait(int32_t* error_flags, uint32_t max_polls, int32_t arrive,
                                                void* stream) {
  if (error_flags == nullptr || !kvq::aligned(error_flags, 4) || max_polls == 0) return KVQ_ERR_INVALID;
  kvq::bounded_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(error_flags, max_polls, arrive);
  return kvq::launch_status();
}
