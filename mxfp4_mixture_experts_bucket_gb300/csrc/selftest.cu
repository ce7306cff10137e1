// Self-test of the failure path shared by the pipelined kernels: a bounded
// mbarrier wait that runs out. One CTA with the roles of a real pipeline, on a
// small scale: warp 0 owns 32 columns of tensor memory, warp 1 (lane 0) lands
// one bulk copy in shared memory, warp 2 waits for a barrier that nothing ever
// arrives at. The wait gives up after the library's time limit (2 s), records
// the timeout in the device status word with its site, and raises the CTA's
// abort flag; the copy is waited for before the CTA leaves and tensor memory is
// freed, so the context stays usable. No fault, trap or unbounded wait is
// involved: the same primitive (tc::mbar_wait) bounds every wait of the
// library's kernels.
#include "tcgen05.cuh"

namespace moe {

constexpr int kSelftestKernel = 15;  // the kernel field of the timeout site
constexpr uint32_t kSelftestCopy = 1024;

__global__ void __launch_bounds__(96, 1) selftest_wait_timeout_kernel(const uint8_t* __restrict__ src, int* status) {
  __shared__ __align__(128) uint8_t buf[kSelftestCopy];
  __shared__ __align__(8) uint64_t full_bar, never_bar, tfree_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&full_bar), 1);
    tc::mbar_init(tc::smem_u32(&never_bar), 1);  // nothing arrives here
    tc::mbar_init(tc::smem_u32(&tfree_bar), 1);
    s_abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), 32);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const volatile int* abort_flag = &s_abort;
  if (warp == 1) {
    if (lane == 0) {
      tc::mbar_expect_tx(tc::smem_u32(&full_bar), kSelftestCopy);
      tc::bulk_load(tc::smem_u32(buf), src, kSelftestCopy, tc::smem_u32(&full_bar));
      // the copy lands before this CTA may leave, whatever the other roles do
      tc::mbar_wait(tc::smem_u32(&full_bar), 0, nullptr);
    }
  } else if (warp == 2) {
    const bool ok = tc::mbar_wait(tc::smem_u32(&never_bar), 0, abort_flag);
    if (!__all_sync(0xffffffffu, ok) && lane == 0) {
      s_abort = 1;
      report_timeout(status, kSelftestKernel, 2, 0, 0);
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&tfree_bar));  // done with tensor memory
  } else {
    tc::mbar_wait_sleep(tc::smem_u32(&tfree_bar), 0, nullptr, 256);
    tc::fence_after_sync();
    tc::tmem_dealloc(s_tmem, 32);
  }
}

cudaError_t launch_selftest_wait_timeout(const uint8_t* src, int* status, Launch L) {
  return launch_kernel(selftest_wait_timeout_kernel, dim3(1), dim3(96), 0, L, src, status);
}

}  // namespace moe
