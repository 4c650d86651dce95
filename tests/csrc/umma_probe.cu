// Single-CTA probe of the tcgen05 path used by the prefill kernel: shared-memory
// descriptors with 128-byte swizzle (K-major and MN-major operands), the bf16
// instruction descriptor, commit-to-mbarrier, TMEM loads and stores, and the
// TMEM-A form of the MMA.  Test infrastructure only.
//   S    = A B^T          (A, B: 128 x 128, K-major)
//   O_ss = P V            (P K-major from shared memory, V MN-major)
//   O_ts = P V            (P from TMEM)
#include <cuda_bf16.h>
#include <stdint.h>

#include "ptx.cuh"
#include "umma.cuh"

using namespace minipic;

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// copy a row-major [128][128] bf16 matrix into [2 halves][128 rows][128 B] swizzled
__device__ void fill(uint8_t* dst, const __nv_bfloat16* src) {
  const int r = threadIdx.x;
  for (int h = 0; h < 2; ++h)
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + r * 128 + h * 64 + c * 8);
      *reinterpret_cast<uint4*>(dst + h * 16384 + swz(r, c)) = v;
    }
}

__global__ void __launch_bounds__(128) probe_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B,
                                                    const __nv_bfloat16* P, const __nv_bfloat16* V, float* S_out,
                                                    float* O_ss, float* O_ts, int* err) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = raw + ((1024 - (ptx::smem_addr(raw) & 1023)) & 1023);
  uint8_t* sA = sm;
  uint8_t* sB = sm + 32768;
  uint8_t* sP = sm + 65536;
  uint8_t* sV = sm + 98304;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 131072);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + 131072 + 64);
  const int tid = threadIdx.x, warp = tid >> 5;

  fill(sA, A);
  fill(sB, B);
  fill(sP, P);
  fill(sV, V);
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(bar), 1);
    ptx::mbar_init(ptx::smem_addr(bar + 1), 1);
    ptx::fence_barrier_init();
  }
  ptx::fence_proxy_async_smem();
  if (warp == 0) {
    umma::tmem_alloc(ptx::smem_addr(tslot), 512);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;

  // P rows into TMEM columns [256, 320): two bf16 per 32-bit column
  {
    const int r = tid;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16) + 256;
    for (int part = 0; part < 4; ++part) {
      uint32_t v[16];
      for (int j = 0; j < 16; ++j) {
        const int k = part * 32 + 2 * j;
        __nv_bfloat162 p2 = __halves2bfloat162(P[r * 128 + k], P[r * 128 + k + 1]);
        v[j] = *reinterpret_cast<uint32_t*>(&p2);
      }
      umma::tmem_st16(lane_addr + part * 16, v);
    }
    umma::tmem_wait_st();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();

  if (tid == 0) {
    const uint32_t idk = umma::idesc_bf16_f32(128, 128, false, false);
    const uint32_t idv = umma::idesc_bf16_f32(128, 128, false, true);
    for (int k = 0; k < 8; ++k) {
      const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
      umma::mma_ss(tmem, umma::smem_desc_sw128(ptx::smem_addr(sA) + off, 16, 1024),
                   umma::smem_desc_sw128(ptx::smem_addr(sB) + off, 16, 1024), idk, k > 0);
    }
    for (int k = 0; k < 8; ++k) {
      const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
      const uint64_t vdesc = umma::smem_desc_sw128(ptx::smem_addr(sV) + k * 2048, 16384, 1024);
      umma::mma_ss(tmem + 128, umma::smem_desc_sw128(ptx::smem_addr(sP) + off, 16, 1024), vdesc, idv, k > 0);
      umma::mma_ts(tmem + 384, tmem + 256 + 8 * k, vdesc, idv, k > 0);
    }
    umma::commit(ptx::smem_addr(bar));
  }
  if (!ptx::mbar_wait(ptx::smem_addr(bar), 0)) atomicOr(err, 1);
  umma::fence_after_sync();

  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  const int row = tid;
  for (int which = 0; which < 3; ++which) {
    float* out = which == 0 ? S_out : (which == 1 ? O_ss : O_ts);
    const uint32_t col0 = which == 0 ? 0 : (which == 1 ? 128 : 384);
    for (int part = 0; part < 4; ++part) {
      uint32_t v[32];
      umma::tmem_ld32(lane_base + col0 + part * 32, v);
      umma::tmem_wait_ld();
      for (int j = 0; j < 32; ++j) out[row * 128 + part * 32 + j] = __uint_as_float(v[j]);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, 512);
}

extern "C" int umma_probe(const void* A, const void* B, const void* P, const void* V, float* S, float* O_ss,
                          float* O_ts, int* err, void* stream) {
  const int smem = 131072 + 128 + 1024;
  if (cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 1;
  probe_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
      (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, (const __nv_bfloat16*)P, (const __nv_bfloat16*)V, S, O_ss,
      O_ts, err);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
