// C-ABI layer: argument validation, split planning, workspace sizing and
// launches.  No allocation, no state except the per-device error word.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>

#include "../../include/minipic.h"
#include "internal.h"

namespace minipic {

// Device error word (MINIPIC_DEVERR_* bits); one per device that loads the library.
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {nullptr};
int g_num_sms[kMaxDevices] = {0};
std::mutex g_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device lookups done once: the device address of the error word and the SM count.
cudaError_t device_info(int** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = n;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  if (err) *err = g_err_ptr[dev];
  if (sms) *sms = g_num_sms[dev];
  return cudaSuccess;
}

int current_sms() {
  int sms = 0;
  if (device_info(nullptr, &sms) != cudaSuccess || sms <= 0) sms = 152;
  return sms;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

DecodeWs decode_ws(int batch, int Hq, int Hkv, int D, int n_split) {
  return decode_ws_layout(batch, Hq, Hkv, D, n_split);
}

minipic_status check_pool(const minipic_kv_pool* kv, int32_t num_q_heads, bool need_ptrs) {
  if (!kv) return MINIPIC_ERR_INVALID;
  if (kv->num_blocks < 0 || kv->num_kv_heads <= 0 || num_q_heads <= 0) return MINIPIC_ERR_INVALID;
  if (num_q_heads % kv->num_kv_heads != 0) return MINIPIC_ERR_INVALID;
  if (kv->head_dim <= 0 || (kv->head_dim & 1)) return MINIPIC_ERR_INVALID;
  if (kv->block_size <= 0) return MINIPIC_ERR_INVALID;
  if (need_ptrs && kv->num_blocks > 0) {
    if (!kv->k_pool || !kv->v_pool) return MINIPIC_ERR_INVALID;
    if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return MINIPIC_ERR_INVALID;
  }
  if (kv->head_dim != 64 && kv->head_dim != 128) return MINIPIC_ERR_UNSUPPORTED;
  if (kv->block_size != 16) return MINIPIC_ERR_UNSUPPORTED;
  if (num_q_heads / kv->num_kv_heads > 16) return MINIPIC_ERR_UNSUPPORTED;
  return MINIPIC_OK;
}

minipic_status check_rope(const minipic_rope* rope, int head_dim) {
  if (!rope || !rope->cos_sin || !aligned16(rope->cos_sin)) return MINIPIC_ERR_INVALID;
  if (rope->max_pos <= 0 || rope->head_dim != head_dim) return MINIPIC_ERR_INVALID;
  return MINIPIC_OK;
}

// Validate a decode batch and fill the launch arguments (no launch).
minipic_status build_decode(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                            const minipic_rope* rope, const minipic_decode_batch* b, float scale, void* workspace,
                            size_t workspace_bytes, bool rotate, DecodeArgs* out_args, DecodePlan* out_plan,
                            bool* empty) {
  *empty = false;
  if (dtype != MINIPIC_F32 && dtype != MINIPIC_BF16) return MINIPIC_ERR_INVALID;
  if (!b) return MINIPIC_ERR_INVALID;
  minipic_status st = check_pool(kv, num_q_heads, b->batch > 0);
  if (st != MINIPIC_OK) return st;
  if (b->batch < 0 || b->max_blocks_per_seq < 0) return MINIPIC_ERR_INVALID;
  if (rotate) {
    st = check_rope(rope, kv->head_dim);
    if (st != MINIPIC_OK) return st;
    // the tensor-core path reads the bf16 cos | sin | -sin rows
    if (dtype == MINIPIC_BF16 && (!rope->cos_sin_bf16 || !aligned16(rope->cos_sin_bf16))) return MINIPIC_ERR_INVALID;
  }
  if (b->batch == 0) {
    *empty = true;
    return MINIPIC_OK;
  }
  if (b->max_blocks_per_seq == 0) return MINIPIC_ERR_INVALID;
  if (!b->q || !b->block_tables || !b->block_starts || !b->seq_lens || !b->q_pos || !b->out)
    return MINIPIC_ERR_INVALID;
  if (!aligned16(b->q) || !aligned16(b->out) || !aligned16(b->block_tables) ||
      !aligned16(b->block_starts))
    return MINIPIC_ERR_INVALID;
  if (!isfinite(scale)) return MINIPIC_ERR_INVALID;

  int* err = nullptr;
  int sms = 0;
  if (device_info(&err, &sms) != cudaSuccess) return MINIPIC_ERR_CUDA;
  const bool bf16 = dtype == MINIPIC_BF16;
  const int G = num_q_heads / kv->num_kv_heads;
  DecodePlan plan = plan_decode(b->batch, kv->num_kv_heads, G, kv->head_dim, b->max_blocks_per_seq,
                                kv->block_size, bf16, sms);
  DecodeWs ws = decode_ws(b->batch, num_q_heads, kv->num_kv_heads, kv->head_dim, plan.n_split);
  if (ws.total > 0) {
    if (!workspace || workspace_bytes < ws.total || !aligned16(workspace)) return MINIPIC_ERR_WORKSPACE;
  }

  DecodeArgs a{};
  a.q = b->q;
  a.k_pool = kv->k_pool;
  a.v_pool = kv->v_pool;
  a.block_tables = b->block_tables;
  a.block_starts = b->block_starts;
  a.seq_lens = b->seq_lens;
  a.q_pos = b->q_pos;
  a.cos_sin = rotate ? rope->cos_sin : nullptr;
  a.cs_bf16 = rotate && bf16 ? rope->cos_sin_bf16 : nullptr;
  a.max_pos = rotate ? rope->max_pos : 0;
  a.out = b->out;
  a.lse = b->lse;
  char* wsb = static_cast<char*>(workspace);
  a.counters = ws.total ? reinterpret_cast<int*>(wsb) : nullptr;
  a.part_o = ws.total ? reinterpret_cast<float*>(wsb + ws.cnt_bytes) : nullptr;
  a.part_ml = ws.total ? reinterpret_cast<float*>(wsb + ws.cnt_bytes + ws.o_bytes) : nullptr;
  a.batch = b->batch;
  a.Hq = num_q_heads;
  a.Hkv = kv->num_kv_heads;
  a.G = G;
  a.D = kv->head_dim;
  a.BS = kv->block_size;
  a.num_blocks = kv->num_blocks;
  a.max_blocks = b->max_blocks_per_seq;
  a.split_blocks = plan.split_blocks;
  a.n_split = plan.n_split;
  a.ctas_per_sm = plan.ctas_per_sm;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)kv->head_dim);
  a.err = err;
  *out_args = a;
  *out_plan = plan;
  return MINIPIC_OK;
}

minipic_status decode_common(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                             const minipic_rope* rope, const minipic_decode_batch* b, float scale,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream, bool rotate) {
  DecodeArgs a{};
  DecodePlan plan{};
  bool empty = false;
  const minipic_status st =
      build_decode(dtype, num_q_heads, kv, rope, b, scale, workspace, workspace_bytes, rotate, &a, &plan, &empty);
  if (st != MINIPIC_OK || empty) return st;
  const cudaError_t e = launch_decode(a, dtype == MINIPIC_BF16, rotate, plan, stream);
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

// Validate a prefill batch and fill the launch arguments (no launch).
minipic_status build_prefill(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                             const minipic_rope* rope, const minipic_prefill_batch* b, float scale, bool rotate,
                             PrefillArgs* out_args, bool* empty) {
  *empty = false;
  if (dtype != MINIPIC_F32 && dtype != MINIPIC_BF16) return MINIPIC_ERR_INVALID;
  if (!b) return MINIPIC_ERR_INVALID;
  minipic_status st = check_pool(kv, num_q_heads, b->batch > 0);
  if (st != MINIPIC_OK) return st;
  if (rotate) {
    st = check_rope(rope, kv->head_dim);
    if (st != MINIPIC_OK) return st;
  }
  if (dtype != MINIPIC_BF16) return MINIPIC_ERR_UNSUPPORTED;
  if (rotate && (!rope->cos_sin_f16 || !aligned16(rope->cos_sin_f16))) return MINIPIC_ERR_INVALID;
  if (b->batch < 0 || b->total_q < 0 || b->max_q_len < 0 || b->max_blocks_per_seq < 0) return MINIPIC_ERR_INVALID;
  if (b->batch == 0 || b->total_q == 0) {
    *empty = true;
    return MINIPIC_OK;
  }
  if (b->max_q_len == 0 || b->max_blocks_per_seq == 0 || kv->num_blocks == 0) return MINIPIC_ERR_INVALID;
  if (!b->q || !b->cu_q_lens || !b->q_pos || !b->block_tables || !b->block_starts || !b->kv_lens || !b->out)
    return MINIPIC_ERR_INVALID;
  if (!aligned16(b->q) || !aligned16(b->out)) return MINIPIC_ERR_INVALID;
  if (!isfinite(scale)) return MINIPIC_ERR_INVALID;
  int* err = nullptr;
  if (device_info(&err, nullptr) != cudaSuccess) return MINIPIC_ERR_CUDA;
  PrefillArgs a{};
  a.q = b->q;
  a.cu_q_lens = b->cu_q_lens;
  a.q_pos = b->q_pos;
  a.k_pool = kv->k_pool;
  a.v_pool = kv->v_pool;
  a.block_tables = b->block_tables;
  a.block_starts = b->block_starts;
  a.kv_lens = b->kv_lens;
  a.cos_sin = rotate ? rope->cos_sin : nullptr;
  a.cos_sin16 = rotate ? rope->cos_sin_f16 : nullptr;
  a.max_pos = rotate ? rope->max_pos : 0;
  a.out = b->out;
  a.lse = b->lse;
  a.batch = b->batch;
  a.total_q = b->total_q;
  a.max_q_len = b->max_q_len;
  a.Hq = num_q_heads;
  a.Hkv = kv->num_kv_heads;
  a.G = num_q_heads / kv->num_kv_heads;
  a.D = kv->head_dim;
  a.BS = kv->block_size;
  a.num_blocks = kv->num_blocks;
  a.max_blocks = b->max_blocks_per_seq;
  a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)kv->head_dim);
  a.err = err;
  *out_args = a;
  return MINIPIC_OK;
}

minipic_status prefill_common(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                              const minipic_rope* rope, const minipic_prefill_batch* b, float scale,
                              cudaStream_t stream, bool rotate) {
  PrefillArgs a{};
  bool empty = false;
  const minipic_status st = build_prefill(dtype, num_q_heads, kv, rope, b, scale, rotate, &a, &empty);
  if (st != MINIPIC_OK || empty) return st;
  const cudaError_t e = launch_prefill_tc(a, rotate, stream);
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

// The mixed grid runs each decode split as one CTA of 8-12 warps that holds a
// whole SM (the CTA shape is the prefill's), where the standalone kernel keeps
// 2-3 CTAs of 4 warps resident per SM.  Short splits then leave their fixed
// cost (metadata staging, pipeline fill, merge) exposed, so the mixed grid
// plans fewer, longer splits: about four waves of one CTA per SM, 64 to 512
// blocks each.  Fewer splits need less of the caller's workspace, whose
// partial-result regions are laid out again for the new split count.
void replan_mixed_decode(DecodeArgs& a, int num_sms) {
  if (a.n_split <= 1) return;
  const long long total = (long long)a.batch * a.Hkv * a.max_blocks;
  const long long slots = (long long)num_sms * 4;
  long long est = (total + slots - 1) / slots;
  if (est < 64) est = 64;
  if (est > 512) est = 512;  // the decode CTA stages a split's block metadata in shared memory
  if (est <= a.split_blocks) return;
  int split_blocks = a.max_blocks, n_split = 1;
  if (est < a.max_blocks) {
    const long long n = (a.max_blocks + est - 1) / est;
    split_blocks = (int)((a.max_blocks + n - 1) / n);
    n_split = (a.max_blocks + split_blocks - 1) / split_blocks;
  }
  if (n_split >= a.n_split) return;
  const DecodeWs ws = decode_ws_layout(a.batch, a.Hq, a.Hkv, a.D, n_split);
  char* base = reinterpret_cast<char*>(a.counters);  // the workspace start (counters first)
  a.split_blocks = split_blocks;
  a.n_split = n_split;
  if (n_split > 1) {
    a.part_o = reinterpret_cast<float*>(base + ws.cnt_bytes);
    a.part_ml = reinterpret_cast<float*>(base + ws.cnt_bytes + ws.o_bytes);
  }
}

}  // namespace

DecodeWs decode_ws_layout(int batch, int Hq, int Hkv, int D, int n_split) {
  DecodeWs w{0, 0, 0, 0};
  if (n_split <= 1) return w;
  w.cnt_bytes = align_up((size_t)batch * Hkv * sizeof(int), 256);
  w.o_bytes = align_up((size_t)batch * Hq * n_split * D * sizeof(float), 256);
  w.ml_bytes = align_up((size_t)batch * Hq * n_split * 2 * sizeof(float), 256);
  w.total = w.cnt_bytes + w.o_bytes + w.ml_bytes;
  return w;
}

DecodePlan plan_decode(int batch, int Hkv, int G, int D, int max_blocks, int bs, bool bf16, int num_sms) {
  (void)D;
  (void)bs;
  DecodePlan p{max_blocks, 1, bf16, 0};
  const long long pairs = (long long)batch * Hkv;
  if (!bf16) {
    // SIMT path: aim for ~4 CTAs per SM, splits of at least 8 blocks
    const long long target = (long long)num_sms * 4;
    const int min_split_blocks = 8;
    if (pairs >= target || max_blocks <= min_split_blocks) return p;
    long long n = (target + pairs - 1) / pairs;
    const long long cap = (max_blocks + min_split_blocks - 1) / min_split_blocks;
    if (n > cap) n = cap;
    if (n < 1) n = 1;
    p.split_blocks = (int)((max_blocks + n - 1) / n);
    p.n_split = (max_blocks + p.split_blocks - 1) / p.split_blocks;
    return p;
  }
  // tensor-core path: CTAs of 4 warps; with many (request, kv head) pairs, 3
  // resident per SM with 2 stages per warp (more warps to hide the per-block
  // latency when blocks come from L2), else 2 per SM with 3 stages (deeper
  // per-warp prefetch for HBM-bound long contexts); 1 for groups > 8.  Splits
  // of at least 32 blocks (8 per warp), as long as about 4 waves of CTAs (3
  // with 2 CTAs per SM) allow: each split pays a fixed cost (metadata
  // staging, pipeline fill, the merge), so longer splits won over the ~12 waves
  // used before (Zipf-shared RAG batch 0.259 -> 0.221 ms, long contexts 0.631
  // -> 0.565 ms); groups > 8 keep ~12 waves.  The table width stands in for
  // the lengths, which stay on the device.
  p.ctas_per_sm = G > 8 ? 1 : (pairs >= 2LL * num_sms ? 3 : 2);
  const long long resident = (long long)num_sms * p.ctas_per_sm;
  const long long total = pairs * max_blocks;
  const long long waves = p.ctas_per_sm == 3 ? 4 : (p.ctas_per_sm == 2 ? 3 : 12);
  long long est = (total + resident * waves - 1) / (resident * waves);
  if (est < 32) est = 32;
  if (est > 512) est = 512;  // the kernel stages a split's block metadata in shared memory
  if (est >= max_blocks) return p;
  const long long n = (max_blocks + est - 1) / est;
  p.split_blocks = (int)((max_blocks + n - 1) / n);
  p.n_split = (max_blocks + p.split_blocks - 1) / p.split_blocks;
  return p;
}

cudaError_t launch_decode(const DecodeArgs& a, bool bf16, bool rotate, const DecodePlan& plan,
                          cudaStream_t s) {
  // the tensor-core kernel merges its splits itself; the SIMT path merges in a second kernel
  if (plan.use_mma) return launch_decode_mma(a, rotate, s);
  cudaError_t e = launch_decode_simt(a, bf16, rotate, s);
  if (e != cudaSuccess) return e;
  return launch_decode_merge(a, bf16, s);
}

}  // namespace minipic

using namespace minipic;

extern "C" {

const char* minipic_status_string(minipic_status status) {
  switch (status) {
    case MINIPIC_OK: return "ok";
    case MINIPIC_ERR_INVALID: return "invalid argument";
    case MINIPIC_ERR_UNSUPPORTED: return "unsupported configuration";
    case MINIPIC_ERR_WORKSPACE: return "workspace missing or too small";
    case MINIPIC_ERR_CUDA: return "CUDA error";
    case MINIPIC_ERR_DEVICE_CHECK: return "device data out of range";
    case MINIPIC_ERR_CAPACITY: return "prefix cache full";
  }
  return "unknown status";
}

minipic_status minipic_rope_table(float* cos_sin, int32_t max_pos, int32_t head_dim, double rope_base,
                                  minipic_stream_t stream) {
  if (!cos_sin || !aligned16(cos_sin) || max_pos <= 0 || head_dim <= 0 || (head_dim & 1))
    return MINIPIC_ERR_INVALID;
  if (!(rope_base > 0.0) || !isfinite(rope_base)) return MINIPIC_ERR_INVALID;
  cudaError_t e = launch_rope_table(cos_sin, max_pos, head_dim, rope_base, (cudaStream_t)stream);
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

minipic_status minipic_rope_table_f16(uint16_t* cos_sin_f16, int32_t max_pos, int32_t head_dim, double rope_base,
                                      minipic_stream_t stream) {
  if (!cos_sin_f16 || !aligned16(cos_sin_f16) || max_pos <= 0 || head_dim <= 0 || (head_dim & 1))
    return MINIPIC_ERR_INVALID;
  if (!(rope_base > 0.0) || !isfinite(rope_base)) return MINIPIC_ERR_INVALID;
  cudaError_t e = launch_rope_table_f16(cos_sin_f16, max_pos, head_dim, rope_base, (cudaStream_t)stream);
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

minipic_status minipic_rope_tables(float* cos_sin, uint16_t* cos_sin_f16, uint16_t* cos_sin_bf16, int32_t max_pos,
                                   int32_t head_dim, double rope_base, minipic_stream_t stream) {
  if (!cos_sin && !cos_sin_f16 && !cos_sin_bf16) return MINIPIC_ERR_INVALID;
  if ((cos_sin && !aligned16(cos_sin)) || (cos_sin_f16 && !aligned16(cos_sin_f16)) ||
      (cos_sin_bf16 && !aligned16(cos_sin_bf16)))
    return MINIPIC_ERR_INVALID;
  if (max_pos <= 0 || head_dim <= 0 || (head_dim & 1) || (cos_sin_bf16 && (head_dim & 15))) return MINIPIC_ERR_INVALID;
  if (!(rope_base > 0.0) || !isfinite(rope_base)) return MINIPIC_ERR_INVALID;
  cudaError_t e = launch_rope_tables(cos_sin, cos_sin_f16, cos_sin_bf16, max_pos, head_dim, rope_base,
                                     (cudaStream_t)stream);
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

minipic_status minipic_rope_table_bf16(uint16_t* cos_sin_bf16, int32_t max_pos, int32_t head_dim,
                                      double rope_base, minipic_stream_t stream) {
  if (!cos_sin_bf16 || !aligned16(cos_sin_bf16) || max_pos <= 0 || head_dim <= 0 || (head_dim & 15))
    return MINIPIC_ERR_INVALID;
  if (!(rope_base > 0.0) || !isfinite(rope_base)) return MINIPIC_ERR_INVALID;
  cudaError_t e = launch_rope_table_bf16(cos_sin_bf16, max_pos, head_dim, rope_base, (cudaStream_t)stream);
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

size_t minipic_attn_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t max_blocks_per_seq,
                                          int32_t block_size) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
      block_size <= 0 || num_q_heads % num_kv_heads)
    return 0;
  const int G = num_q_heads / num_kv_heads;
  DecodePlan p = plan_decode(batch, num_kv_heads, G, head_dim, max_blocks_per_seq, block_size, true,
                             current_sms());
  DecodePlan p32 = plan_decode(batch, num_kv_heads, G, head_dim, max_blocks_per_seq, block_size, false,
                               current_sms());
  const size_t a = decode_ws(batch, num_q_heads, num_kv_heads, head_dim, p.n_split).total;
  const size_t b = decode_ws(batch, num_q_heads, num_kv_heads, head_dim, p32.n_split).total;
  return a > b ? a : b;
}

minipic_status minipic_attn_decode(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                                   const minipic_rope* rope, const minipic_decode_batch* batch, float scale,
                                   void* workspace, size_t workspace_bytes, minipic_stream_t stream) {
  return decode_common(dtype, num_q_heads, kv, rope, batch, scale, workspace, workspace_bytes,
                       (cudaStream_t)stream, true);
}

minipic_status minipic_attn_decode_prerotated(minipic_dtype dtype, int32_t num_q_heads,
                                              const minipic_kv_pool* kv, const minipic_decode_batch* batch,
                                              float scale, void* workspace, size_t workspace_bytes,
                                              minipic_stream_t stream) {
  return decode_common(dtype, num_q_heads, kv, nullptr, batch, scale, workspace, workspace_bytes,
                       (cudaStream_t)stream, false);
}

size_t minipic_attn_prefill_workspace_size(int32_t, int32_t, int32_t, int32_t, int32_t, int32_t, int32_t) {
  return 0;
}

minipic_status minipic_attn_prefill(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                                    const minipic_rope* rope, const minipic_prefill_batch* batch, float scale,
                                    void* workspace, size_t workspace_bytes, minipic_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  return prefill_common(dtype, num_q_heads, kv, rope, batch, scale, (cudaStream_t)stream, true);
}

minipic_status minipic_attn_prefill_prerotated(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                                               const minipic_prefill_batch* batch, float scale,
                                               minipic_stream_t stream) {
  return prefill_common(dtype, num_q_heads, kv, nullptr, batch, scale, (cudaStream_t)stream, false);
}

minipic_status minipic_attn_mixed(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                                  const minipic_rope* rope, const minipic_prefill_batch* prefill,
                                  const minipic_decode_batch* decode, float scale, void* workspace,
                                  size_t workspace_bytes, minipic_stream_t stream) {
  if (dtype != MINIPIC_BF16) return (dtype == MINIPIC_F32) ? MINIPIC_ERR_UNSUPPORTED : MINIPIC_ERR_INVALID;
  PrefillArgs p{};
  DecodeArgs d{};
  DecodePlan plan{};
  bool p_empty = false, d_empty = false;
  minipic_status st = build_prefill(dtype, num_q_heads, kv, rope, prefill, scale, true, &p, &p_empty);
  if (st != MINIPIC_OK) return st;
  st = build_decode(dtype, num_q_heads, kv, rope, decode, scale, workspace, workspace_bytes, true, &d, &plan,
                    &d_empty);
  if (st != MINIPIC_OK) return st;
  cudaError_t e = cudaSuccess;
  if (p_empty && d_empty) return MINIPIC_OK;
  if (d_empty) {
    e = launch_prefill_tc(p, true, (cudaStream_t)stream);
  } else if (p_empty) {
    e = launch_decode(d, true, true, plan, (cudaStream_t)stream);
  } else {
    if (kv->num_blocks == 0) return MINIPIC_ERR_INVALID;
    replan_mixed_decode(d, current_sms());
    e = launch_mixed(p, d, (cudaStream_t)stream);
  }
  return e == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

minipic_status minipic_kv_append(minipic_dtype dtype, const minipic_kv_pool_mut* kv,
                                 const minipic_kv_append_batch* b, minipic_stream_t stream) {
  if (dtype != MINIPIC_F32 && dtype != MINIPIC_BF16) return MINIPIC_ERR_INVALID;
  if (!kv || !b) return MINIPIC_ERR_INVALID;
  if (kv->num_blocks < 0 || kv->num_kv_heads <= 0 || kv->block_size <= 0 || kv->head_dim <= 0)
    return MINIPIC_ERR_INVALID;
  if (b->batch < 0 || b->total_new < 0 || b->max_new_len < 0 || b->max_blocks_per_seq < 0)
    return MINIPIC_ERR_INVALID;
  if (kv->head_dim != 64 && kv->head_dim != 128) return MINIPIC_ERR_UNSUPPORTED;
  if (kv->block_size != 16) return MINIPIC_ERR_UNSUPPORTED;
  if (b->batch == 0 || b->total_new == 0 || b->max_new_len == 0) return MINIPIC_OK;
  if (b->batch > 65535 || b->max_blocks_per_seq == 0 || kv->num_blocks == 0) return MINIPIC_ERR_INVALID;
  if (!b->k_new || !b->v_new || !b->cu_new_lens || !b->kv_start || !b->block_tables || !kv->k_pool ||
      !kv->v_pool)
    return MINIPIC_ERR_INVALID;
  if (!aligned16(b->k_new) || !aligned16(b->v_new) || !aligned16(kv->k_pool) || !aligned16(kv->v_pool))
    return MINIPIC_ERR_INVALID;
  int* err = nullptr;
  if (device_info(&err, nullptr) != cudaSuccess) return MINIPIC_ERR_CUDA;
  AppendArgs a{};
  a.k_new = b->k_new;
  a.v_new = b->v_new;
  a.cu_new = b->cu_new_lens;
  a.kv_start = b->kv_start;
  a.block_tables = b->block_tables;
  a.k_pool = kv->k_pool;
  a.v_pool = kv->v_pool;
  a.batch = b->batch;
  a.max_new = b->max_new_len;
  a.max_blocks = b->max_blocks_per_seq;
  a.num_blocks = kv->num_blocks;
  a.Hkv = kv->num_kv_heads;
  a.D = kv->head_dim;
  a.elem = dtype == MINIPIC_BF16 ? 2 : 4;
  a.err = err;
  return launch_kv_append(a, (cudaStream_t)stream) == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

namespace {

// Device-side address of page-locked host memory (nullptr if it is not).
void* host_device_ptr(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky error of a failed query
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

minipic_status offload(minipic_dtype dtype, void* k_pool, void* v_pool, int32_t num_blocks, int32_t Hkv,
                       int32_t bs, int32_t D, const int32_t* ids, int32_t n, const void* host_k,
                       const void* host_v, bool to_host, cudaStream_t stream) {
  if (dtype != MINIPIC_F32 && dtype != MINIPIC_BF16) return MINIPIC_ERR_INVALID;
  if (num_blocks < 0 || Hkv <= 0 || bs <= 0 || D <= 0 || n < 0) return MINIPIC_ERR_INVALID;
  if (D != 64 && D != 128) return MINIPIC_ERR_UNSUPPORTED;
  if (bs != 16) return MINIPIC_ERR_UNSUPPORTED;
  if (n == 0) return MINIPIC_OK;
  if (num_blocks == 0 || !k_pool || !v_pool || !ids || !host_k || !host_v) return MINIPIC_ERR_INVALID;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(host_k) || !aligned16(host_v))
    return MINIPIC_ERR_INVALID;
  void* dk = host_device_ptr(host_k);
  void* dv = host_device_ptr(host_v);
  if (!dk || !dv || !aligned16(dk) || !aligned16(dv)) return MINIPIC_ERR_INVALID;
  int* err = nullptr;
  int sms = 0;
  if (device_info(&err, &sms) != cudaSuccess) return MINIPIC_ERR_CUDA;
  OffloadArgs a{};
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.host_k = dk;
  a.host_v = dv;
  a.block_ids = ids;
  a.n = n;
  a.num_blocks = num_blocks;
  a.block_chunks = (long long)Hkv * bs * D * (dtype == MINIPIC_BF16 ? 2 : 4) / 16;
  a.err = err;
  return launch_kv_offload(a, to_host, sms, stream) == cudaSuccess ? MINIPIC_OK : MINIPIC_ERR_CUDA;
}

}  // namespace

minipic_status minipic_kv_swap_out(minipic_dtype dtype, const minipic_kv_pool* kv, const int32_t* block_ids,
                                   int32_t n, void* host_k, void* host_v, minipic_stream_t stream) {
  if (!kv) return MINIPIC_ERR_INVALID;
  return offload(dtype, const_cast<void*>(kv->k_pool), const_cast<void*>(kv->v_pool), kv->num_blocks,
                 kv->num_kv_heads, kv->block_size, kv->head_dim, block_ids, n, host_k, host_v, true,
                 (cudaStream_t)stream);
}

minipic_status minipic_kv_swap_in(minipic_dtype dtype, const minipic_kv_pool_mut* kv, const int32_t* block_ids,
                                  int32_t n, const void* host_k, const void* host_v, minipic_stream_t stream) {
  if (!kv) return MINIPIC_ERR_INVALID;
  return offload(dtype, kv->k_pool, kv->v_pool, kv->num_blocks, kv->num_kv_heads, kv->block_size, kv->head_dim,
                 block_ids, n, host_k, host_v, false, (cudaStream_t)stream);
}

minipic_status minipic_device_error(int32_t* flags_out, int32_t clear, minipic_stream_t stream) {
  int* err = nullptr;
  if (device_info(&err, nullptr) != cudaSuccess) return MINIPIC_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MINIPIC_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MINIPIC_ERR_CUDA;
  if (clear && v) {
    if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return MINIPIC_ERR_CUDA;
  }
  if (flags_out) *flags_out = v;
  return v ? MINIPIC_ERR_DEVICE_CHECK : MINIPIC_OK;
}

}  // extern "C"
