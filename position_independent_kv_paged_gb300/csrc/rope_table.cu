// Rotary cos/sin table (MiniPIC summary, section 2.1: the kernel rotates keys
// with "a cosine/sine table lookup" and multiply-adds per element).
//
// Row p holds cos(p * theta_i) in columns [0, d/2) and sin(p * theta_i) in
// columns [d/2, d), theta_i = base^(-2 i / d).  The angle is formed in double
// precision (fp32 angles would be off by ~1e-2 rad at p ~ 1.3e5) and CUDA's
// double-precision sincos is called; the results are rounded once to the
// table's type (fp32, or fp16 for the prefill's packed-fp16 key rotation).
// The bf16 form for the decode's packed-bf16 rotation holds, for each position
// p, two rows of 3 d/2 values: cos | sin | -sin of the angle +p theta_i and of
// -p theta_i (that is cos | -sin | sin), each the fp32 value rounded to the
// nearest bf16.  A rotation by a signed angle then reads one row, with no
// conversion and no sign logic.
#include <cuda_bf16.h>
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

__global__ void __launch_bounds__(256) rope_table_bf16_kernel(uint16_t* __restrict__ cs, int max_pos, int d,
                                                              double base) {
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
    const float cf = (float)c, sf = (float)s;
    const uint16_t cb = __bfloat16_as_ushort(__float2bfloat16_rn(cf));
    const uint16_t sp = __bfloat16_as_ushort(__float2bfloat16_rn(sf));
    const uint16_t sn = __bfloat16_as_ushort(__float2bfloat16_rn(-sf));
    uint16_t* row = cs + (long long)p * 6 * half;  // angle +p theta: cos | sin | -sin
    row[i] = cb;
    row[half + i] = sp;
    row[2 * half + i] = sn;
    row += 3 * half;                                // angle -p theta: cos | -sin | sin
    row[i] = cb;
    row[half + i] = sn;
    row[2 * half + i] = sp;
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

cudaError_t launch_rope_table_bf16(uint16_t* cs, int max_pos, int head_dim, double base, cudaStream_t s) {
  const long long total = (long long)max_pos * (head_dim / 2);
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  rope_table_bf16_kernel<<<(unsigned)blocks, 256, 0, s>>>(cs, max_pos, head_dim, base);
  return cudaGetLastError();
}

}  // namespace minipic
