// Prefill kernel wrapper and launcher for head dim 64 (the CTA body is in
// prefill2_body.cuh; head dim 128 goes to the CTA-pair kernel).
#include "prefill2_body.cuh"
#include "tmap.cuh"

namespace minipic {
namespace {

using namespace prefill2_impl;

// One CTA per (query-tile pair, kv head, request); each CTA loads its own K~/V
// tiles.
template <int D, bool ROPE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const PrefillLaunch2 L) {
  extern __shared__ uint8_t smem_raw[];
  // heaviest (latest) query-tile pairs first
  const int n = gridDim.x;
  prefill2_cta<D, ROPE>(&kmap, &vmap, L, n - 1 - (int)blockIdx.x, n, blockIdx.y, blockIdx.z, smem_raw);
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
  if (n_pairs <= 0) return cudaSuccess;
  prefill_tc_kernel<D, ROPE>
      <<<dim3((unsigned)n_pairs, (unsigned)a.Hkv, (unsigned)a.batch), kThreads, smem, s>>>(km, vm, L);
  return cudaGetLastError();
}

}  // namespace

// Head dim 128 runs the CTA-pair kernel; head dim 64 this single-CTA kernel.
cudaError_t launch_prefill_tc(const PrefillArgs& a, bool rotate, cudaStream_t s) {
  if (a.D == 128) return launch_prefill_pair(a, rotate, s);
  if (a.D != 64) return cudaErrorInvalidValue;
  return rotate ? launch_t<64, true>(a, s) : launch_t<64, false>(a, s);
}

}  // namespace minipic
