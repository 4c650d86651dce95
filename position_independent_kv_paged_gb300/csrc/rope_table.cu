// Rotary cos/sin table (MiniPIC summary, section 2.1: the kernel rotates keys
// with "a cosine/sine table lookup" and multiply-adds per element).
//
// Row p holds cos(p * theta_i) in columns [0, d/2) and sin(p * theta_i) in
// columns [d/2, d), theta_i = base^(-2 i / d).  The angle is formed in double
// precision (fp32 angles would be off by ~1e-2 rad at p ~ 1.3e5) and CUDA's
// double-precision sincos is called; the results are rounded once to the
// table's type (fp32, or fp16 for the prefill's packed-fp16 key rotation).
#include <cuda_fp16.h>

#include "internal.h"

namespace minipic {
namespace {

__device__ __forceinline__ void store_val(float* p, double v) { *p = (float)v; }
__device__ __forceinline__ void store_val(uint16_t* p, double v) { *p = __half_as_ushort(__double2half(v)); }

template <typename T>
__global__ void __launch_bounds__(256) rope_table_kernel(T* __restrict__ cs, int max_pos, int d, double base) {
  const int half = d >> 1;
  const long long total = (long long)max_pos * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(idx / half);
    const int i = (int)(idx - (long long)p * half);
    const double theta = pow(base, -2.0 * (double)i / (double)d);
    const double ang = (double)p * theta;
    double s, c;
    sincos(ang, &s, &c);
    store_val(cs + (long long)p * d + i, c);
    store_val(cs + (long long)p * d + half + i, s);
  }
}

template <typename T>
cudaError_t launch_t(T* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s) {
  const long long total = (long long)max_pos * (head_dim / 2);
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  rope_table_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(cos_sin, max_pos, head_dim, base);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_table(float* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s) {
  return launch_t(cos_sin, max_pos, head_dim, base, s);
}

cudaError_t launch_rope_table_f16(uint16_t* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s) {
  return launch_t(cos_sin, max_pos, head_dim, base, s);
}

}  // namespace minipic
