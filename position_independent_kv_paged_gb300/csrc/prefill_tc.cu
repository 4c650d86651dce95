// Prefill kernel wrapper and launcher (the CTA body is in prefill2_body.cuh).
#include "prefill2_body.cuh"
#include "tmap.cuh"

namespace minipic {
namespace {

using namespace prefill2_impl;

template <int D, bool ROPE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const PrefillLaunch2 L) {
  extern __shared__ uint8_t smem_raw[];
  // heaviest (latest) query-tile pairs first
  prefill2_cta<D, ROPE>(&kmap, &vmap, L, gridDim.x - 1 - blockIdx.x, gridDim.x, blockIdx.y, blockIdx.z, smem_raw);
}

template <int D, bool ROPE>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  const int smem = PG2<D>::TOTAL + 1024;
  static bool done[64] = {false};
  cudaError_t e = set_smem_once(prefill_tc_kernel<D, ROPE>, smem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.Hkv * 16;
  if (!make_pool_map(&km, a.k_pool, rows, D) || !make_pool_map(&vm, a.v_pool, rows, D)) return cudaErrorInvalidValue;
  PrefillLaunch2 L{a, 128 / a.G};
  const int n_pairs = (a.max_q_len + 2 * L.tq - 1) / (2 * L.tq);
  dim3 grid(n_pairs, a.Hkv, a.batch);
  prefill_tc_kernel<D, ROPE><<<grid, kThreads, smem, s>>>(km, vm, L);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs& a, bool rotate, cudaStream_t s) {
  if (rotate) return a.D == 128 ? launch_t<128, true>(a, s) : launch_t<64, true>(a, s);
  return a.D == 128 ? launch_t<128, false>(a, s) : launch_t<64, false>(a, s);
}

}  // namespace minipic
