// Decode attention over the position-free paged cache, SIMT form (fp32 and
// bf16 inputs, fp32 arithmetic throughout).  This is the exact-precision path:
// the fp32 workload needs errors far below what bf16 tensor-core operands give.
//
// One CTA = (split, kv head, request); its 4 warps take the split's blocks
// round robin and keep an online softmax per query head of the GQA group; the
// warps are merged through shared memory at the end.  Lane l owns head
// dimensions l, l+32, ... so each rotary pair (i, i + d/2) is lane-local and a
// key is rotated with two multiply-adds per element from the cos/sin table
// row of its logical position (MiniPIC summary section 2.1: pi(j) =
// start of the key's block in this request + slot).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"

namespace minipic {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}
template <typename T>
__device__ __forceinline__ void st_f(T* p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int D, int MAXG, bool ROPE>
__global__ void __launch_bounds__(128) decode_simt_kernel(DecodeArgs a) {
  constexpr int E = D / 32;  // elements per lane
  constexpr int H = E / 2;   // rotary pairs per lane
  constexpr int NW = 4;
  __shared__ float sm_m[NW][MAXG];
  __shared__ float sm_l[NW][MAXG];
  __shared__ float sm_o[NW][MAXG][D];

  const int s = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;
  const T* __restrict__ kpool = static_cast<const T*>(a.k_pool);
  const T* __restrict__ vpool = static_cast<const T*>(a.v_pool);
  const T* __restrict__ qg = static_cast<const T*>(a.q);

  int L = a.seq_lens[r];
  const int Lmax = a.max_blocks * a.BS;
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0 && s == 0) atomicOr(a.err, kErrSeqLen);
    L = L < 0 ? 0 : Lmax;
  }
  const int nblk = (L + a.BS - 1) / a.BS;
  const int n_valid = max(1, (nblk + a.split_blocks - 1) / a.split_blocks);
  if (s >= n_valid) return;
  const int b_begin = s * a.split_blocks;
  const int b_end = min(nblk, b_begin + a.split_blocks);

  // Rotated queries of the group: qr[h][e] holds dim lane + 32 e of head g*G + h.
  float qr[MAXG][E];
  int tq = 0;
  if (ROPE) {
    tq = a.q_pos[r];
    if (tq < 0 || tq >= a.max_pos) {
      if (threadIdx.x == 0 && s == 0) atomicOr(a.err, kErrPosition);
      tq = 0;
    }
  }
#pragma unroll
  for (int h = 0; h < MAXG; ++h) {
    if (h < G) {
      const T* qp = qg + ((size_t)r * a.Hq + (size_t)g * G + h) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) qr[h][e] = ld_f(qp + lane + 32 * e);
      if (ROPE) {
        const float* row = a.cos_sin + (size_t)tq * D;
#pragma unroll
        for (int e = 0; e < H; ++e) {
          const float c = __ldg(row + lane + 32 * e);
          const float sn = __ldg(row + D / 2 + lane + 32 * e);
          const float x = qr[h][e], y = qr[h][e + H];
          qr[h][e] = fmaf(x, c, -y * sn);
          qr[h][e + H] = fmaf(y, c, x * sn);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) qr[h][e] = 0.f;
    }
  }

  float m[MAXG], l[MAXG], o[MAXG][E];
#pragma unroll
  for (int h = 0; h < MAXG; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[h][e] = 0.f;
  }
  const float sl2 = a.scale * kLog2e;

  for (int b = b_begin + warp; b < b_end; b += NW) {
    const int phys = a.block_tables[(size_t)r * a.max_blocks + b];
    if (phys < 0 || phys >= a.num_blocks) {
      if (lane == 0) atomicOr(a.err, kErrBlockId);
      continue;
    }
    const int start = ROPE ? a.block_starts[(size_t)r * a.max_blocks + b] : 0;
    const int nk = min(a.BS, L - b * a.BS);
    const size_t tile = ((size_t)phys * a.Hkv + g) * a.BS;
    for (int slot = 0; slot < nk; ++slot) {
      const T* kp = kpool + (tile + slot) * D;
      const T* vp = vpool + (tile + slot) * D;
      float k[E], v[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        k[e] = ld_f(kp + lane + 32 * e);
        v[e] = ld_f(vp + lane + 32 * e);
      }
      if (ROPE) {
        const int pos = start + slot;
        if (pos < 0 || pos >= a.max_pos) {
          if (lane == 0) atomicOr(a.err, kErrPosition);
          continue;
        }
        const float* row = a.cos_sin + (size_t)pos * D;
#pragma unroll
        for (int e = 0; e < H; ++e) {
          const float c = __ldg(row + lane + 32 * e);
          const float sn = __ldg(row + D / 2 + lane + 32 * e);
          const float x = k[e], y = k[e + H];
          k[e] = fmaf(x, c, -y * sn);
          k[e + H] = fmaf(y, c, x * sn);
        }
      }
#pragma unroll
      for (int h = 0; h < MAXG; ++h) {
        if (h < G) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) dot = fmaf(qr[h][e], k[e], dot);
          dot = warp_sum(dot) * sl2;
          const float mn = fmaxf(m[h], dot);
          const float corr = exp2f(m[h] - mn);
          const float p = exp2f(dot - mn);
          l[h] = fmaf(l[h], corr, p);
#pragma unroll
          for (int e = 0; e < E; ++e) o[h][e] = fmaf(o[h][e], corr, p * v[e]);
          m[h] = mn;
        }
      }
    }
  }

  // merge the warps of this CTA
#pragma unroll
  for (int h = 0; h < MAXG; ++h) {
    if (lane == 0) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = l[h];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sm_o[warp][h][lane + 32 * e] = o[h][e];
  }
  __syncthreads();
  const bool direct = (n_valid == 1);
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, dim = idx - h * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w][h]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = (sm_m[w][h] == -CUDART_INF_F) ? 0.f : exp2f(sm_m[w][h] - M);
      Ls = fmaf(sm_l[w][h], f, Ls);
      O = fmaf(sm_o[w][h][dim], f, O);
    }
    const int hq = g * G + h;
    if (direct) {
      T* out = static_cast<T*>(a.out) + ((size_t)r * a.Hq + hq) * D + dim;
      st_f<T>(out, Ls > 0.f ? O / Ls : 0.f);
      if (dim == 0 && a.lse) a.lse[(size_t)r * a.Hq + hq] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
    } else {
      const size_t pi = ((size_t)r * a.Hq + hq) * a.n_split + s;
      a.part_o[pi * D + dim] = O;
      if (dim == 0) {
        a.part_ml[pi * 2] = M;
        a.part_ml[pi * 2 + 1] = Ls;
      }
    }
  }
}

// Log-sum-exp merge of the split partials of one (request, query head).
template <typename T>
__global__ void decode_merge_kernel(DecodeArgs a) {
  const int r = blockIdx.x / a.Hq, hq = blockIdx.x % a.Hq;
  int L = a.seq_lens[r];
  const int Lmax = a.max_blocks * a.BS;
  L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  const int nblk = (L + a.BS - 1) / a.BS;
  const int n_valid = max(1, (nblk + a.split_blocks - 1) / a.split_blocks);
  if (n_valid <= 1) return;  // written directly by the split kernel
  const size_t base = ((size_t)r * a.Hq + hq) * a.n_split;
  float M = -CUDART_INF_F;
  for (int s = 0; s < n_valid; ++s) M = fmaxf(M, a.part_ml[(base + s) * 2]);
  for (int dim = threadIdx.x; dim < a.D; dim += blockDim.x) {
    float Ls = 0.f, O = 0.f;
    for (int s = 0; s < n_valid; ++s) {
      const float ms = a.part_ml[(base + s) * 2];
      const float f = (ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
      Ls = fmaf(a.part_ml[(base + s) * 2 + 1], f, Ls);
      O = fmaf(a.part_o[(base + s) * a.D + dim], f, O);
    }
    T* out = static_cast<T*>(a.out) + ((size_t)r * a.Hq + hq) * a.D + dim;
    st_f<T>(out, Ls > 0.f ? O / Ls : 0.f);
    if (dim == 0 && a.lse) a.lse[(size_t)r * a.Hq + hq] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
  }
}

template <typename T, int D, bool ROPE>
cudaError_t dispatch_g(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.n_split, a.Hkv, a.batch);
  if (a.G <= 4)
    decode_simt_kernel<T, D, 4, ROPE><<<grid, 128, 0, s>>>(a);
  else if (a.G <= 8)
    decode_simt_kernel<T, D, 8, ROPE><<<grid, 128, 0, s>>>(a);
  else
    decode_simt_kernel<T, D, 16, ROPE><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T, bool ROPE>
cudaError_t dispatch_d(const DecodeArgs& a, cudaStream_t s) {
  return a.D == 64 ? dispatch_g<T, 64, ROPE>(a, s) : dispatch_g<T, 128, ROPE>(a, s);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, bool bf16, bool rotate, cudaStream_t s) {
  if (bf16)
    return rotate ? dispatch_d<__nv_bfloat16, true>(a, s) : dispatch_d<__nv_bfloat16, false>(a, s);
  return rotate ? dispatch_d<float, true>(a, s) : dispatch_d<float, false>(a, s);
}

cudaError_t launch_decode_merge(const DecodeArgs& a, bool bf16, cudaStream_t s) {
  if (a.n_split <= 1) return cudaSuccess;
  const int threads = a.D;
  if (bf16)
    decode_merge_kernel<__nv_bfloat16><<<a.batch * a.Hq, threads, 0, s>>>(a);
  else
    decode_merge_kernel<float><<<a.batch * a.Hq, threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace minipic
