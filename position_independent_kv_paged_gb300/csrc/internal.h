// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace minipic {

// Arguments of one decode launch (built by the C-ABI layer after validation).
struct DecodeArgs {
  const void* q;             // [B][Hq][D]
  const void* k_pool;        // [num_blocks][Hkv][BS][D]
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* block_starts;
  const int32_t* seq_lens;
  const int32_t* q_pos;
  const float* cos_sin;      // [max_pos][D] or null when rotation is compiled out
  const uint16_t* cs_bf16;   // [max_pos][2][3 D/2] bf16 cos | sin | -sin of +-p (tensor-core path), or null
  int max_pos;
  void* out;                 // [B][Hq][D]
  float* lse;                // [B][Hq] or null
  float* part_o;             // [B][Hq][n_split][D] (unnormalised), null when n_split == 1
  float* part_ml;            // [B][Hq][n_split][2] (max, sum) in log2 units
  int* counters;             // [B][Hkv] finished splits (zero between calls), null when n_split == 1
  int batch, Hq, Hkv, G, D, BS, num_blocks, max_blocks;
  int split_blocks;          // blocks per split
  int n_split;               // splits per (request, kv head)
  int ctas_per_sm;           // tensor-core decode: 3 (2 stages per warp) or 2 (3 stages) CTAs per SM
  float scale;               // softmax scale (1/sqrt(D) by default)
  int* err;                  // device error word
};

// Arguments of one prefill launch.
struct PrefillArgs {
  const void* q;             // [total_q][Hq][D]
  const int32_t* cu_q_lens;  // [B+1]
  const int32_t* q_pos;      // [total_q]
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* block_starts;
  const int32_t* kv_lens;
  const float* cos_sin;       // [max_pos][D] fp32 (query rotation)
  const uint16_t* cos_sin16;  // [max_pos][D] fp16 (key rotation in the CTA-pair kernel)
  int max_pos;
  void* out;
  float* lse;
  int batch, total_q, max_q_len, Hq, Hkv, G, D, BS, num_blocks, max_blocks;
  float scale;
  int* err;
};

// Error bits (mirror MINIPIC_DEVERR_* of the public header).
enum : int { kErrBlockId = 1, kErrPosition = 2, kErrSeqLen = 4, kErrTimeout = 8, kErrRange = 16 };

// Launchers; return cudaSuccess or the launch error.
cudaError_t launch_rope_table(float* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s);
cudaError_t launch_rope_table_f16(uint16_t* cos_sin, int max_pos, int head_dim, double base, cudaStream_t s);
cudaError_t launch_rope_table_bf16(uint16_t* cs, int max_pos, int head_dim, double base, cudaStream_t s);
cudaError_t launch_rope_tables(float* f32, uint16_t* f16, uint16_t* b16, int max_pos, int head_dim, double base,
                               cudaStream_t s);

// Split planning of the decode kernels (same plan used for workspace sizing).
struct DecodePlan {
  int split_blocks;
  int n_split;
  bool use_mma;
  int ctas_per_sm;  // tensor-core path: resident CTAs per SM (3 or 2; 1 for more than 8 heads per group)
};
DecodePlan plan_decode(int batch, int Hkv, int G, int D, int max_blocks, int bs, bool bf16, int num_sms);

cudaError_t launch_decode(const DecodeArgs& a, bool bf16, bool rotate, const DecodePlan& plan, cudaStream_t s);
cudaError_t launch_decode_simt(const DecodeArgs& a, bool bf16, bool rotate, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeArgs& a, bool rotate, cudaStream_t s);
cudaError_t launch_decode_merge(const DecodeArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs& a, bool rotate, cudaStream_t s);
// Head dim 128: CTA-pair (cta_group::2) form, called by launch_prefill_tc.
cudaError_t launch_prefill_pair(const PrefillArgs& a, bool rotate, cudaStream_t s);
// One grid of prefill tiles followed by decode splits (both with rotation).
cudaError_t launch_mixed(const PrefillArgs& p, const DecodeArgs& d, cudaStream_t s);
// Head dim 128: one grid of CTA-pair prefill clusters and decode clusters.
cudaError_t launch_mixed_pair(const PrefillArgs& p, const DecodeArgs& d, cudaStream_t s);

// Cache append: token i of request r -> key index kv_start[r] + i.
struct AppendArgs {
  const void* k_new;  // [total_new][Hkv][D]
  const void* v_new;
  const int32_t* cu_new;      // [batch + 1]
  const int32_t* kv_start;    // [batch]
  const int32_t* block_tables;  // [batch][max_blocks]
  void* k_pool;  // [num_blocks][Hkv][16][D]
  void* v_pool;
  int batch, max_new, max_blocks, num_blocks, Hkv, D, elem;
  int* err;
};
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t s);

// Whole-block copies between the pools and page-locked host memory.
struct OffloadArgs {
  void* k_pool;  // [num_blocks][Hkv][16][D]
  void* v_pool;
  void* host_k;  // device-side address of the host buffer, [n][Hkv][16][D]
  void* host_v;
  const int32_t* block_ids;  // [n]
  int n, num_blocks;
  long long block_chunks;  // 16-byte chunks of one block (all kv heads)
  int* err;
};
cudaError_t launch_kv_offload(const OffloadArgs& a, bool to_host, int num_sms, cudaStream_t s);

// Byte layout of the decode workspace: one completion counter per (request,
// kv head) first, then partial outputs and partial (max, sum) pairs.
struct DecodeWs {
  size_t o_bytes, ml_bytes, cnt_bytes, total;
};
DecodeWs decode_ws_layout(int batch, int Hq, int Hkv, int D, int n_split);

}  // namespace minipic
