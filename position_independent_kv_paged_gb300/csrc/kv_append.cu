// Appending new tokens to the position-free paged cache (MiniPIC summary,
// section 2.1: the cache holds unrotated key vectors, so a new key is stored
// exactly as produced).  Token i of request r becomes key index
// j = kv_start[r] + i: block block_tables[r][j / 16], slot j % 16.
//
// An HBM-bound copy: a thread moves 16-byte chunks of (token, head) rows of K
// and the same chunks of V, four per pass with every load issued first.
// Consecutive threads walk a row, then the heads of a token, so the reads of
// k_new / v_new are contiguous and every 128-byte line of a pool row is
// written whole.  blockIdx.y is the request.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace minipic {
namespace {

constexpr int kThreads = 256;

constexpr int kUnroll = 4;  // chunks per thread and pass, loads issued before stores

template <int CPR>  // 16-byte chunks per (token, head) row
__global__ void __launch_bounds__(kThreads) kv_append_kernel(AppendArgs a) {
  const int r = blockIdx.y;
  const int t0 = a.cu_new[r];
  const int n = a.cu_new[r + 1] - t0;
  if (n <= 0) return;
  const int js = a.kv_start[r];
  const int* bt = a.block_tables + (size_t)r * a.max_blocks;
  const long long per_tok = (long long)a.Hkv * CPR;
  const long long total = (long long)n * per_tok;
  const long long row_chunks = 16LL * CPR;  // chunks of one (block, head) tile
  const long long stride = (long long)gridDim.x * kThreads;
  for (long long base = (long long)blockIdx.x * kThreads + threadIdx.x; base < total; base += stride * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
    long long dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long idx = base + u * stride;
      dst[u] = -1;
      if (idx >= total) continue;
      const int i = (int)(idx / per_tok);
      const int rem = (int)(idx - (long long)i * per_tok);
      const int h = rem / CPR, c = rem - h * CPR;
      const int j = js + i;
      const int blk = j >> 4;
      if (js < 0 || blk >= a.max_blocks) {
        if (h == 0 && c == 0) atomicOr(a.err, kErrSeqLen);
        continue;
      }
      const int phys = __ldg(bt + blk);
      if (phys < 0 || phys >= a.num_blocks) {
        if (h == 0 && c == 0) atomicOr(a.err, kErrBlockId);
        continue;
      }
      const size_t src = ((size_t)(t0 + i) * a.Hkv + h) * CPR + c;
      dst[u] = (long long)(((size_t)phys * a.Hkv + h) * row_chunks + (size_t)(j & 15) * CPR + c);
      kv[u] = __ldcs(static_cast<const uint4*>(a.k_new) + src);
      vv[u] = __ldcs(static_cast<const uint4*>(a.v_new) + src);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] < 0) continue;
      static_cast<uint4*>(a.k_pool)[dst[u]] = kv[u];
      static_cast<uint4*>(a.v_pool)[dst[u]] = vv[u];
    }
  }
}

template <int CPR>
cudaError_t launch_t(const AppendArgs& a, cudaStream_t s) {
  const long long per_req = (long long)a.max_new * a.Hkv * CPR;
  long long gx = (per_req + (long long)kThreads * kUnroll - 1) / ((long long)kThreads * kUnroll);
  if (gx < 1) gx = 1;
  if (gx > 65535) gx = 65535;  // grid-stride beyond this
  dim3 grid((unsigned)gx, (unsigned)a.batch);
  kv_append_kernel<CPR><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t s) {
  const int row_bytes = a.D * a.elem;
  switch (row_bytes / 16) {
    case 8: return launch_t<8>(a, s);    // bf16, d 64
    case 16: return launch_t<16>(a, s);  // bf16 d 128, f32 d 64
    case 32: return launch_t<32>(a, s);  // f32, d 128
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace minipic
