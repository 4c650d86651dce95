// Allocation-free variant of the decode entry point.
//
// Some callers cannot allocate device memory when they call attention: code
// running inside a memory pool that must not grow, a runtime that forbids
// cudaMalloc on its serving path (an allocation can synchronize the device or
// fail under fragmentation), or a plain C host without an allocator of its
// own.  For them this file keeps the split-KV partial results of decode in a
// fixed device array that is part of the library image: every GPU that loads
// the library holds kNoAllocScratchBytes for it until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Only the split-completion counters at its start must be zero when
// a call begins, so each call clears them on its stream first; partial results
// are always written before they are read.  Calls whose work overlaps on the
// GPU (two streams, or concurrent host threads) race on the array; serialize
// them.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/minipic.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MINIPIC_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current and reused afterwards.
minipic_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MINIPIC_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MINIPIC_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MINIPIC_OK;
}

}  // namespace

extern "C" {

minipic_status minipic_attn_decode_noalloc(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                                           const minipic_rope* rope, const minipic_decode_batch* batch,
                                           float scale, minipic_stream_t stream) {
  if (!kv || !batch) return MINIPIC_ERR_INVALID;
  if (batch->batch > 0) {
    const size_t need = minipic_attn_decode_workspace_size(batch->batch, num_q_heads, kv->num_kv_heads,
                                                           kv->head_dim, batch->max_blocks_per_seq,
                                                           kv->block_size);
    if (need > kNoAllocScratchBytes) return MINIPIC_ERR_WORKSPACE;  // shape too large for the fixed scratch
  }
  void* scratch = nullptr;
  const minipic_status st = scratch_address(&scratch);
  if (st != MINIPIC_OK) return st;
  // the split-completion counters (the first batch * kv-heads words, padded to
  // 256 bytes) must start at zero; clear them rather than trust the last call
  if (batch->batch > 0 && kv->num_kv_heads > 0) {
    const size_t cnt = (((size_t)batch->batch * kv->num_kv_heads * sizeof(int)) + 255) / 256 * 256;
    if (cnt <= kNoAllocScratchBytes && cudaMemsetAsync(scratch, 0, cnt, (cudaStream_t)stream) != cudaSuccess)
      return MINIPIC_ERR_CUDA;
  }
  return minipic_attn_decode(dtype, num_q_heads, kv, rope, batch, scale, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
