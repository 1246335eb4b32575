// Diagnostic kernels behind pkv_check_bounded_wait (the per-warp ring check
// sits beside the partition kernel in pkv_decode.cu).
//
// Shared-ring check: the kernels whose warps share one ring of stages (the
// FP8 head-group partition kernel) decide a timed-out wait for the whole CTA
// with a CTA-wide vote after every step, so that no warp waits at a barrier
// the others have left.  Here four warps share two stage barriers.  Barrier
// 0 completes its first phase through a plain arrival (no copy is involved);
// barrier 1 never does.  Warps 1-3 wait on barrier 0 and pass at once; warp
// 0 waits on barrier 1 with the bounded wait until its limit runs out.  Every
// wait ends by itself, so every warp reaches the vote; the vote then sends
// every warp out, and warp 0 sets PKV_DEV_ERR_TIMEOUT.
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__global__ void __launch_bounds__(128) bounded_wait_vote_check_kernel(int32_t* status, long long timeout_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t done = smem_u32(&bars[0]), open = smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    mbar_init(open, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(done);  // phase 0 of `done` completes; `open` never does
  __syncthreads();
  const bool ok = __all_sync(kFull, mbar_wait_bounded(warp == 0 ? open : done, 0, timeout_ns));
  if (__syncthreads_or(!ok) && warp == 0 && lane == 0) flag(status, 16u);  // PKV_DEV_ERR_TIMEOUT
}

}  // namespace

cudaError_t launch_bounded_wait_vote_check(int32_t* status, long long timeout_ns, cudaStream_t stream) {
  bounded_wait_vote_check_kernel<<<1, 128, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace pkv
