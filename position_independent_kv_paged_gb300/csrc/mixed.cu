// Mixed continuous batch in one launch: the grid holds the span-prefill query
// tiles first (heaviest first) and then the decode splits, so that the
// tensor-core-bound prefill CTAs and the HBM-bound decode CTAs share the SMs
// (the device side of interleaved span-prefill scheduling, MiniPIC summary
// section 2.2 "Scheduling": span prefills pipelined with ongoing decodes).
// Both CTA bodies are the ones of the standalone kernels; decode CTAs take the
// prefill CTA's shape (16 warps, ~226 KB shared memory) and run 12 decode
// warps with 2 stages each.
#include "decode_body.cuh"
#include "prefill2_body.cuh"
#include "tmap.cuh"

namespace minipic {
namespace {

constexpr int kMixThreads = prefill2_impl::kThreads;  // 16 warps; decode CTAs use 12 of them
constexpr int kDecWarps = 12, kDecStages = 2;

template <int D, int NT>
__global__ void __launch_bounds__(kMixThreads, 1)
    mixed_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const __grid_constant__ CUtensorMap vblk, const prefill2_impl::PrefillLaunch2 P, const DecodeArgs Dd, const int n_pre, const int n_pairs) {
  extern __shared__ uint8_t smem_raw[];
  const int i = blockIdx.x;
  if (i < n_pre) {
    const int per = P.a.Hkv * P.a.batch;
    const int pr_rev = i / per, rem = i - pr_rev * per;
    const int hk = rem / P.a.batch, r = rem - hk * P.a.batch;
    prefill2_impl::prefill2_cta<D, true>(&kmap, &vblk, P, n_pairs - 1 - pr_rev, n_pairs, hk, r, smem_raw);
  } else {
    const int j = i - n_pre;
    const int split = j % Dd.n_split, rest = j / Dd.n_split;
    const int hk = rest % Dd.Hkv, r = rest / Dd.Hkv;
    decode_impl::decode_cta<D, NT, true, kDecWarps, kDecStages>(&kmap, &vmap, Dd, split, hk, r, smem_raw);
  }
}

template <int D, int NT>
cudaError_t launch_t(const PrefillArgs& p, const DecodeArgs& d, cudaStream_t s) {
  constexpr int a = decode_impl::Smem<D, kDecWarps, kDecStages>::TOTAL, b = prefill2_impl::PG2<D>::TOTAL;
  const int smem = (a > b ? a : b) + 1024;
  static bool done[64] = {false};
  cudaError_t e = set_smem_once(mixed_kernel<D, NT>, smem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap km, vm, vb;
  const long long rows = (long long)p.num_blocks * p.Hkv * 16;
  if (!make_pool_map(&km, p.k_pool, rows, D) || !make_pool_map(&vm, p.v_pool, rows, D) ||
      !make_pool_block_map(&vb, p.v_pool, rows, D))
    return cudaErrorInvalidValue;
  prefill2_impl::PrefillLaunch2 P{p, 128 / p.G};
  const int n_pairs = (p.max_q_len + 2 * P.tq - 1) / (2 * P.tq);
  const long long n_pre = (long long)n_pairs * p.Hkv * p.batch;
  const long long n_dec = (long long)d.n_split * d.Hkv * d.batch;
  if (n_pre + n_dec > 0x7fffffffLL) return cudaErrorInvalidValue;
  mixed_kernel<D, NT><<<(unsigned)(n_pre + n_dec), kMixThreads, smem, s>>>(km, vm, vb, P, d, (int)n_pre, n_pairs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mixed(const PrefillArgs& p, const DecodeArgs& d, cudaStream_t s) {
  if (p.D == 128) return launch_mixed_pair(p, d, s);
  return d.G <= 8 ? launch_t<64, 1>(p, d, s) : launch_t<64, 2>(p, d, s);
}

}  // namespace minipic
