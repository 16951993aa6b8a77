// Failure-detection probe: one bounded wait that is meant to run out.
//
// Every kernel of the layer waits on mbarriers (copies landed, MMAs done, stages free) through
// ptx::mbar_wait, which gives up after a time limit and lets the kernel raise a bit in the device
// status word, stop, drain and return, so that a lost arrival shows up as a status bit on the host
// instead of a hung GPU.  This kernel runs that same wait on an mbarrier that nothing arrives on,
// with a short limit, and raises kStatusWaitProbe when it gives up: the host can check the whole
// path (the wait's time limit, the status word, the context staying usable) without any fault.
#include "tcgen05_ptx.cuh"

namespace colibri {
namespace {

__global__ void __launch_bounds__(32) wait_probe_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int never;  // the abort flag of the wait: never set
  if (threadIdx.x != 0) return;
  never = 0;
  ptx::mbar_init(ptx::smem_u32(&bar), 1);
  ptx::fence_mbar_init();
  if (!ptx::mbar_wait(ptx::smem_u32(&bar), 0, &never, timeout_ns)) atomicOr(status, kStatusWaitProbe);
}

}  // namespace

cudaError_t launch_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace colibri
