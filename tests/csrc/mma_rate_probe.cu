// Throughput probe for the tcgen05 shapes the prefill kernel issues: one CTA
// per SM, one thread issues `iters` x 8 back-to-back M = 128, K = 16 MMAs into a
// TMEM accumulator (operands: constant bf16 tiles; values do not matter) and
// records the SM cycles until their commit lands.  Test infrastructure only.
//   mode 0: A and B from shared memory (the QK^T form), N = n
//   mode 1: A from TMEM, B from shared memory (the P.V form), N = n
// mma_rate2 does the same with CTA pairs (cta_group::2, M = 256 across a
// 2-CTA cluster, each CTA holding 128 rows of A and N / 2 columns of B); the
// even CTA issues.  A kernel uses one cta_group throughout, so the pair form
// is a kernel of its own.
#include <cuda_runtime.h>
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

// ---- cta_group::2 forms (this kernel issues no cta_group::1 instruction)
__device__ __forceinline__ void alloc2(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma2_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(id)
      : "memory");
}
__device__ __forceinline__ void commit2_both(uint32_t mbar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(mbar),
      "h"((uint16_t)3)
      : "memory");
}

__global__ void __launch_bounds__(128, 1) rate_kernel2(long long* cycles, int n, int mode, int iters, int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tslot;
  __shared__ __align__(8) uint64_t mbar;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t rank = ptx::cluster_rank();
  const uint32_t sb = (ptx::smem_addr(smem) + 1023u) & ~1023u;
  uint8_t* sg = smem + (sb - ptx::smem_addr(smem));
  for (int i = tid; i < 65536 / 4; i += 128) reinterpret_cast<uint32_t*>(sg)[i] = 0x3f803f80u;
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(&mbar), 1);
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    alloc2(ptx::smem_addr(&tslot), 512);
    relinquish2();
  }
  ptx::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' operands, barriers and TMEM exist
  umma::fence_after_sync();
  const uint32_t tmem = tslot;
  if (tid == 0) {
    const long long t0 = clock64();
    if (rank == 0) {
      const uint32_t id = umma::idesc_bf16_f32(256, n, false, mode == 1);
      const uint64_t ad = umma::smem_desc_sw128(sb, 16, 1024);
      const uint64_t bd = mode == 0 ? umma::smem_desc_sw128(sb + 32768, 16, 1024)
                                    : umma::smem_desc_sw128(sb + 32768, 2048, 1024);
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if (mode == 0)
            mma2_ss(tmem + 256, ad + (uint64_t)(2 * (ks & 3)), bd + (uint64_t)(2 * (ks & 3)), id);
          else
            mma2_ts(tmem + 256, tmem + 8 * (ks & 3), bd + (uint64_t)(64 * (ks & 3)), id);
        }
      }
      commit2_both(ptx::smem_addr(&mbar));
    }
    if (!ptx::mbar_wait(ptx::smem_addr(&mbar), 0)) atomicOr(err, 1);
    if (rank == 0) cycles[blockIdx.x >> 1] = clock64() - t0;
  }
  __syncwarp();
  umma::fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();
  umma::fence_after_sync();
  if (warp == 0) dealloc2(tmem, 512);
  ptx::cluster_sync();
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

// Pair form: ctas (even) CTAs in clusters of two; cycles has ctas / 2 entries
// (one per pair, M = 256 x N = n x K = 16 per MMA).
extern "C" int mma_rate2(long long* cycles, int ctas, int n, int mode, int iters, int* err, cudaStream_t s) {
  if (n < 32 || n > 256 || n % 32 != 0 || (mode != 0 && mode != 1) || iters < 1 || ctas < 2 || ctas % 2)
    return 1;
  cudaError_t e = cudaFuncSetAttribute(rate_kernel2, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = (size_t)kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, rate_kernel2, cycles, n, mode, iters, err);
  return (int)e;
}
