// Probe of the bounded mbarrier wait that every pipeline in the library uses:
// a wait on a phase that nothing completes gives up after its limit and says
// so, which turns a lost copy or commit into an error status while the CUDA
// context stays usable.  Test infrastructure only.
#include <stdint.h>

#include "ptx.cuh"

using namespace minipic;

// status[0]: wait on a barrier that nothing arrives on (1 = completed, 2 = gave up)
// status[1]: wait on a barrier that thread 0 arrives on (1 = completed, 2 = gave up)
// status[2]: global-timer nanoseconds thread 0 spent in the first wait
__global__ void __launch_bounds__(32) wait_probe_kernel(long long* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  const uint32_t never = ptx::smem_addr(&bars[0]), once = ptx::smem_addr(&bars[1]);
  if (threadIdx.x == 0) {
    ptx::mbar_init(never, 1);
    ptx::mbar_init(once, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = ptx::globaltimer();
  const bool a = ptx::mbar_wait(never, 0, limit_ns);  // phase 0 of a fresh barrier: never completes
  const uint64_t t1 = ptx::globaltimer();
  if (threadIdx.x == 0) ptx::mbar_arrive(once);  // completes phase 0 of the other barrier
  const bool b = ptx::mbar_wait(once, 0, limit_ns);
  if (threadIdx.x == 0) {
    status[0] = a ? 1 : 2;
    status[1] = b ? 1 : 2;
    status[2] = (long long)(t1 - t0);
  }
}

extern "C" int wait_probe(long long* status, unsigned long long limit_ns, void* stream) {
  wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
