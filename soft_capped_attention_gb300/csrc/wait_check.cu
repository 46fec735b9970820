// Self-check of the bounded-wait protocol that every tcgen05 kernel follows.
//
// Each CTA takes the shape of the attention kernels: warp 1 allocates all 512
// TMEM columns, warp 0 (the producer's role) waits on an mbarrier that nothing
// will ever arrive on, with a caller-given limit, and warps 2..3 (a consumer's
// role) wait on a second such barrier with the normal limit.  When warp 0's
// limit runs out it records the timeout bit in the status word and raises the
// CTA's abort flag; the consumers see the flag and leave their wait; every warp
// meets at the final barrier and warp 1 frees TMEM.  No copy or MMA is in
// flight, so nothing needs draining.  The dynamic shared memory request keeps
// one CTA per SM, as in the attention kernels, so that a TMEM column left
// allocated would stall the next attention kernel on that SM.
#include "capattn_internal.h"
#include "tc_common.cuh"

namespace capattn {

namespace {

constexpr int kWaitCheckSmem = 160 * 1024;

__global__ void __launch_bounds__(128, 1) wait_check_kernel(uint32_t* status, uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  const uint32_t bar_never0 = smem_u32(&bars[0]), bar_never1 = smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_never0, 1);
    mbar_init(bar_never1, 1);
    fence_mbar_init();
    smem_raw[0] = 0;  // the dynamic request only reserves the SM
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  pdl_trigger();
  pdl_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (warp == 0) {
    mbar_wait_warp(bar_never0, 0, status, &abort_flag, limit_ns);
  } else if (warp >= 2) {
    mbar_wait_warp(bar_never1, 0, status, &abort_flag);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, int ctas, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(wait_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kWaitCheckSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(wait_check_kernel, dim3(ctas), dim3(128), kWaitCheckSmem, s, status, limit_ns);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace capattn
