// Whole-block copies between the paged pools and page-locked host memory
// (MiniPIC summary, section 3, item 5: unrotated blocks move between GPU and
// host with nothing to track or adjust, so offload is a plain copy).
//
// One kernel gathers (swap-out) or scatters (swap-in) the listed blocks; it
// reaches the host buffer directly by its address (page-locked memory is
// mapped into the device's address space), so n blocks take one launch instead
// of 2n copy calls.  A thread moves 16-byte chunks, four per pass with every
// load issued first; consecutive threads walk a block's contiguous bytes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace minipic {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// to_host: pool[ids[i]] -> host[i]; otherwise host[i] -> pool[ids[i]].  K and V.
__global__ void __launch_bounds__(kThreads) kv_offload_kernel(OffloadArgs a, bool to_host) {
  const long long per_blk = a.block_chunks;           // 16-byte chunks of one block (all heads)
  const long long total = (long long)a.n * per_blk;   // of K (V the same)
  const long long stride = (long long)gridDim.x * kThreads;
  uint4* pk = static_cast<uint4*>(a.k_pool);
  uint4* pv = static_cast<uint4*>(a.v_pool);
  uint4* hk = static_cast<uint4*>(a.host_k);
  uint4* hv = static_cast<uint4*>(a.host_v);
  for (long long base = (long long)blockIdx.x * kThreads + threadIdx.x; base < total; base += stride * kUnroll) {
    uint4 kx[kUnroll], vx[kUnroll];
    long long dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long idx = base + u * stride;
      dst[u] = -1;
      if (idx >= total) continue;
      const long long i = idx / per_blk;
      const long long c = idx - i * per_blk;
      const int b = __ldg(a.block_ids + i);
      if (b < 0 || b >= a.num_blocks) {
        if (c == 0) atomicOr(a.err, kErrBlockId);
        continue;
      }
      const long long p = (long long)b * per_blk + c;  // chunk in the pool
      if (to_host) {
        kx[u] = __ldcs(pk + p);
        vx[u] = __ldcs(pv + p);
        dst[u] = idx;
      } else {
        kx[u] = __ldcs(hk + idx);
        vx[u] = __ldcs(hv + idx);
        dst[u] = p;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] < 0) continue;
      if (to_host) {
        __stcs(hk + dst[u], kx[u]);
        __stcs(hv + dst[u], vx[u]);
      } else {
        pk[dst[u]] = kx[u];
        pv[dst[u]] = vx[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_offload(const OffloadArgs& a, bool to_host, int num_sms, cudaStream_t s) {
  const long long total = (long long)a.n * a.block_chunks;
  long long grid = (total + (long long)kThreads * kUnroll - 1) / ((long long)kThreads * kUnroll);
  const long long cap = (long long)num_sms * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  kv_offload_kernel<<<(unsigned)grid, kThreads, 0, s>>>(a, to_host);
  return cudaGetLastError();
}

}  // namespace minipic
