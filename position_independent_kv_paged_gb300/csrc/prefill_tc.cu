// Prefill kernel wrapper and launcher for head dim 64 (the CTA body is in
// prefill2_body.cuh; head dim 128 goes to the CTA-pair kernel).
#include "prefill2_body.cuh"
#include "tmap.cuh"

namespace minipic {
namespace {

using namespace prefill2_impl;

// Launched in clusters of two along x: CTAs 2c and 2c + 1 (adjacent query-tile
// pairs of one request and kv head) share every K~/V tile through multicast.
template <int D, bool ROPE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const PrefillLaunch2 L) {
  extern __shared__ uint8_t smem_raw[];
  // heaviest (latest) query-tile pairs first
  const int n = gridDim.x;
  prefill2_cta<D, ROPE, true>(&kmap, &vmap, L, n - 1 - (int)blockIdx.x, n - 1 - (int)(blockIdx.x ^ 1u), n,
                              blockIdx.y, blockIdx.z, smem_raw);
}

template <int D, bool ROPE>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  const int smem = PG2<D>::TOTAL + 1024;
  static bool done[64] = {false};
  cudaError_t e = set_smem_once(prefill_tc_kernel<D, ROPE>, smem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.Hkv * 16;
  if (!make_pool_map(&km, a.k_pool, rows, D) || !make_pool_block_map(&vm, a.v_pool, rows, D))
    return cudaErrorInvalidValue;
  PrefillLaunch2 L{a, 128 / a.G};
  const int n_pairs = (a.max_q_len + 2 * L.tq - 1) / (2 * L.tq);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((n_pairs + 1) & ~1), (unsigned)a.Hkv, (unsigned)a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, ROPE>, km, vm, L);
}

}  // namespace

// Head dim 128 runs the CTA-pair kernel; head dim 64 this single-CTA kernel.
cudaError_t launch_prefill_tc(const PrefillArgs& a, bool rotate, cudaStream_t s) {
  if (a.D == 128) return launch_prefill_pair(a, rotate, s);
  if (a.D != 64) return cudaErrorInvalidValue;
  return rotate ? launch_t<64, true>(a, s) : launch_t<64, false>(a, s);
}

}  // namespace minipic
