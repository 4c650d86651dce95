// Decode kernel wrapper and launcher (the CTA body is in decode_body.cuh).
#include "decode_body.cuh"
#include "tmap.cuh"

namespace minipic {
namespace {

using namespace decode_impl;

// CPS resident CTAs per SM: 3 with 2 stages per warp, else 3 stages.
template <int D, int NT, bool ROPE, int CPS>
__global__ void __launch_bounds__(kWarps * 32, CPS)
    decode_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  decode_cta<D, NT, ROPE, kWarps, CPS == 3 ? 2 : kStages, 0, D == 128>(&kmap, &vmap, a, blockIdx.x, blockIdx.y,
                                                                     blockIdx.z, smem_raw);
}

template <int D, int NT, bool ROPE, int CPS>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
  const int smem = Smem<D, kWarps, CPS == 3 ? 2 : kStages>::TOTAL + 1024;
  static bool done[64] = {false};
  cudaError_t e = set_smem_once(decode_mma_kernel<D, NT, ROPE, CPS>, smem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.Hkv * 16;
  const bool ok = D == 128 ? make_pool_block_map(&km, a.k_pool, rows, D) && make_pool_block_map(&vm, a.v_pool, rows, D)
                           : make_pool_map(&km, a.k_pool, rows, D) && make_pool_map(&vm, a.v_pool, rows, D);
  if (!ok) return cudaErrorInvalidValue;
  dim3 grid(a.n_split, a.Hkv, a.batch);
  decode_mma_kernel<D, NT, ROPE, CPS><<<grid, kWarps * 32, smem, s>>>(km, vm, a);
  return cudaGetLastError();
}

template <int D, bool ROPE>
cudaError_t launch_d(const DecodeArgs& a, cudaStream_t s) {
  if (a.G > 8) return launch_t<D, 2, ROPE, 1>(a, s);
  return a.ctas_per_sm == 3 ? launch_t<D, 1, ROPE, 3>(a, s) : launch_t<D, 1, ROPE, 2>(a, s);
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeArgs& a, bool rotate, cudaStream_t s) {
  if (a.num_blocks <= 0) return launch_decode_simt(a, true, rotate, s);  // nothing to map; all keys masked
  if (a.D == 128) return rotate ? launch_d<128, true>(a, s) : launch_d<128, false>(a, s);
  return rotate ? launch_d<64, true>(a, s) : launch_d<64, false>(a, s);
}

}  // namespace minipic
