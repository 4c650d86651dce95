// Throughput probe for the tcgen05 shapes the prefill kernel issues: one CTA
// per SM, one thread issues `iters` x 8 back-to-back M = 128, K = 16 MMAs into a
// TMEM accumulator (operands: constant bf16 tiles; values do not matter) and
// records the SM cycles until their commit lands.  Test infrastructure only.
//   mode 0: A and B from shared memory (the QK^T form), N = n
//   mode 1: A from TMEM, B from shared memory (the P.V form), N = n
#include <stdint.h>

#include "ptx.cuh"
#include "umma.cuh"

using namespace minipic;

namespace {

constexpr int kSmem = 70000;  // A tile (16 KB) + B tile (up to 32 KB) + 1 KB alignment slack

__global__ void __launch_bounds__(128, 1) rate_kernel(long long* cycles, int n, int mode, int iters, int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tslot;
  __shared__ __align__(8) uint64_t mbar;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sb = (ptx::smem_addr(smem) + 1023u) & ~1023u;
  uint8_t* sg = smem + (sb - ptx::smem_addr(smem));
  for (int i = tid; i < 65536 / 4; i += 128) reinterpret_cast<uint32_t*>(sg)[i] = 0x3f803f80u;
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(&mbar), 1);
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    umma::tmem_alloc(ptx::smem_addr(&tslot), 512);
    umma::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = tslot;
  if (tid == 0) {
    const uint32_t id = umma::idesc_bf16_f32(128, n, false, mode == 1);
    const uint64_t ad = umma::smem_desc_sw128(sb, 16, 1024);
    const uint64_t bd = mode == 0 ? umma::smem_desc_sw128(sb + 32768, 16, 1024)
                                  : umma::smem_desc_sw128(sb + 32768, 2048, 1024);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // accumulator at column 256 (N <= 256); A in TMEM at columns 0..31
        if (mode == 0)
          umma::mma_ss(tmem + 256, ad + (uint64_t)(2 * (ks & 3)), bd + (uint64_t)(2 * (ks & 3)), id, 1u);
        else
          umma::mma_ts(tmem + 256, tmem + 8 * (ks & 3), bd + (uint64_t)(64 * (ks & 3)), id, 1u);
      }
    }
    umma::commit(ptx::smem_addr(&mbar));
    if (!ptx::mbar_wait(ptx::smem_addr(&mbar), 0)) atomicOr(err, 1);
    cycles[blockIdx.x] = clock64() - t0;
  }
  __syncwarp();
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, 512);
}

}  // namespace

// cycles: device array of `ctas` entries.  Returns a cudaError_t value.
extern "C" int mma_rate(long long* cycles, int ctas, int n, int mode, int iters, int* err, cudaStream_t s) {
  if (n < 16 || n > 256 || n % 16 != 0 || (mode != 0 && mode != 1) || iters < 1 || ctas < 1) return 1;
  cudaError_t e = cudaFuncSetAttribute(rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return (int)e;
  rate_kernel<<<ctas, 128, kSmem, s>>>(cycles, n, mode, iters, err);
  return (int)cudaGetLastError();
}
