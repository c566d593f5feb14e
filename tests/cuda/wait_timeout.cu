// Test-only kernel: waits, with the library's bounded mbarrier wait, on a barrier that
// nothing arrives on, and reports what the library's kernels report when a pipeline wait
// runs out: PDA_DEVERR_TIMEOUT, with the kernel returning normally.
#include "pda_device.cuh"

__global__ void wait_for_nothing(int32_t* status, unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    pda::mbar_init(&bar, 1);
    pda::fence_mbar_init();
  }
  __syncwarp();
  const unsigned long long t0 = pda::global_timer_ns();
  const bool done = __all_sync(pda::kFullMask, pda::mbar_wait_bounded(&bar, 0));
  if (lane == 0) {
    *elapsed_ns = pda::global_timer_ns() - t0;
    if (!done) pda::atomic_or_error(status, PDA_DEVERR_TIMEOUT);
  }
}

extern "C" int pda_test_wait_timeout(int32_t* status, unsigned long long* elapsed_ns,
                                     cudaStream_t stream) {
  wait_for_nothing<<<1, 32, 0, stream>>>(status, elapsed_ns);
  return static_cast<int>(cudaGetLastError());
}
