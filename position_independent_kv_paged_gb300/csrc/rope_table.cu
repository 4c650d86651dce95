// Rotary cos/sin table (MiniPIC summary, section 2.1: the kernel rotates keys
// with "a cosine/sine table lookup" and multiply-adds per element).
//
// Row p holds cos(p * theta_i) in columns [0, d/2) and sin(p * theta_i) in
// columns [d/2, d), theta_i = base^(-2 i / d).  The angle is formed in double
// precision (fp32 angles would be off by ~1e-2 rad at p ~ 1.3e5) and CUDA's
// double-precision sincos is called; the results are rounded once to the
// table's type (fp32, or fp16 for the prefill's packed-fp16 key rotation);
// one pass can write all three forms.
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

// One pass over (position p, frequency i): the angle p theta_i in fp64 and
// CUDA's double sincos, written to every table the caller asked for (null
// pointers are skipped): fp32 cos | sin; fp16 cos | sin (the fp64 values
// rounded once); bf16 rows of cos | sin | -sin for +p and for -p (the fp32
// values rounded to the nearest bf16).
__global__ void __launch_bounds__(256) rope_tables_kernel(float* __restrict__ f32, uint16_t* __restrict__ f16,
                                                          uint16_t* __restrict__ b16, int max_pos, int d,
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
    if (f32) {
      f32[(long long)p * d + i] = (float)c;
      f32[(long long)p * d + half + i] = (float)s;
    }
    if (f16) {
      f16[(long long)p * d + i] = __half_as_ushort(__double2half(c));
      f16[(long long)p * d + half + i] = __half_as_ushort(__double2half(s));
    }
    if (b16) {
      const float cf = (float)c, sf = (float)s;
      const uint16_t cb = __bfloat16_as_ushort(__float2bfloat16_rn(cf));
      const uint16_t sp = __bfloat16_as_ushort(__float2bfloat16_rn(sf));
      const uint16_t sn = __bfloat16_as_ushort(__float2bfloat16_rn(-sf));
      uint16_t* row = b16 + (long long)p * 6 * half;  // angle +p theta: cos | sin | -sin
      row[i] = cb;
      row[half + i] = sp;
      row[2 * half + i] = sn;
      row += 3 * half;                                 // angle -p theta: cos | -sin | sin
      row[i] = cb;
      row[half + i] = sn;
      row[2 * half + i] = sp;
    }
  }
}

}  // namespace

cudaError_t launch_rope_tables(float* f32, uint16_t* f16, uint16_t* b16, int max_pos, int head_dim, double base,
                               cudaStream_t s) {
  const long long total = (long long)max_pos * (head_dim / 2);
  long long blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  rope_tables_kernel<<<(unsigned)blocks, 256, 0, s>>>(f32, f16, b16, max_pos, head_dim, base);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s) {
  return launch_rope_tables(cos_sin, nullptr, nullptr, max_pos, head_dim, base, s);
}

cudaError_t launch_rope_table_f16(uint16_t* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s) {
  return launch_rope_tables(nullptr, cos_sin, nullptr, max_pos, head_dim, base, s);
}

cudaError_t launch_rope_table_bf16(uint16_t* cs, int max_pos, int head_dim, double base, cudaStream_t s) {
  return launch_rope_tables(nullptr, nullptr, cs, max_pos, head_dim, base, s);
}

}  // namespace minipic
