/*
 * minipic.h -- C ABI of the position-free paged attention library (GB300, sm_103a).
 *
 * The library implements the attention step of MiniPIC's position-free KV cache
 * (MiniPIC summary, gist.science/it/paper/2606.13126, section 2.1): keys are
 * stored unrotated (k~_j) in a paged block pool, and the kernels apply rotary
 * position embedding on the fly at each request's logical key position pi(j):
 *
 *     score(t, j) = (R_t q_t)^T (R_{pi(j)} k~_j) / sqrt(d)
 *     out_t       = sum_j softmax_j(score(t, .)) v_j
 *
 * The rotation is applied with a cosine/sine table lookup and multiply-adds per
 * key element (same section, "Implementazione"), so one physical block can be
 * read by several concurrent requests at different offsets without being
 * rewritten ("Vantaggio").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Rotary form: half rotation.  For i < d/2 and angle a = p * theta_i with
 *    theta_i = base^(-2 i / d):
 *        x'_i       = x_i       cos a - x_{i+d/2} sin a
 *        x'_{i+d/2} = x_{i+d/2} cos a + x_i       sin a
 *  - KV pool: k_pool and v_pool are device arrays [num_blocks][num_kv_heads]
 *    [block_size][head_dim] of the call's dtype; keys are NOT rotated.
 *  - Request r's key with request-local index j lives in physical block
 *    block_tables[r*max_blocks_per_seq + j/block_size], slot j % block_size,
 *    at logical position pi(j) = block_starts[r*max_blocks_per_seq + j/block_size]
 *    + j % block_size.  Both tables are device int32 [batch][max_blocks_per_seq].
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Queries are passed unrotated with their positions; the kernels rotate them.
 *  - The rotary table is the device array written by minipic_rope_table:
 *    float [max_pos][head_dim], cos(p theta_i) in columns [0, d/2) and
 *    sin(p theta_i) in columns [d/2, d), plus (for the prefill and mixed calls)
 *    the same values rounded to fp16 in a second array of that layout, written
 *    by minipic_rope_table_f16, and (for the bf16 decode and the mixed call)
 *    rows of cos | sin | -sin rounded to bf16, written by
 *    minipic_rope_table_bf16.  Every position used must be < max_pos.
 *  - scale <= 0 selects 1/sqrt(head_dim).
 *  - Outputs: out has the layout of q and the call's dtype; lse (optional, may
 *    be NULL) is float, natural-log log-sum-exp of the scaled scores per
 *    (query token, query head).  A query with no key gets out = 0, lse = -inf.
 *  - Supported: head_dim 64 or 128, block_size 16, num_q_heads a multiple of
 *    num_kv_heads with num_q_heads / num_kv_heads <= 16, dtype f32 or bf16
 *    (prefill and mixed: bf16 only).  All device pointers 16-byte aligned.
 *
 * Ownership and execution
 * -----------------------
 *  The caller owns every buffer.  The library allocates no device memory; entry
 *  points that need scratch take a caller-provided workspace whose size is given
 *  by the matching *_workspace_size query.  The decode workspace starts with
 *  one completion counter per (request, kv head): zero the workspace once after
 *  allocating it; every call leaves those counters zero again (after a call that
 *  reports MINIPIC_DEVERR_TIMEOUT, zero it again before reuse).  All calls are asynchronous on the
 *  given stream (cudaStream_t; NULL = legacy default stream) and act on the
 *  device current at the call.  Inputs must stay valid until the work completes.
 *  The library looks up the device address of its error word once per device
 *  and keeps it: do not use it across cudaDeviceReset on that device.
 *
 * Errors
 * ------
 *  Every entry point returns a minipic_status; nothing aborts or throws across
 *  the ABI and no kernel traps.  Host-side validation failures return before
 *  any launch.  Device data (block ids, positions, lengths) is checked inside
 *  the kernels: an out-of-range block id or position is skipped (treated as a
 *  masked key) and a bit is set in a device error word that
 *  minipic_device_error() reads and clears.
 */
#ifndef MINIPIC_H
#define MINIPIC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* minipic_stream_t; /* identical to cudaStream_t */

typedef enum {
  MINIPIC_OK = 0,
  MINIPIC_ERR_INVALID = 1,      /* an argument is null, negative, misaligned or inconsistent */
  MINIPIC_ERR_UNSUPPORTED = 2,  /* a valid configuration this build has no kernel for */
  MINIPIC_ERR_WORKSPACE = 3,    /* workspace is NULL or smaller than the size query returned */
  MINIPIC_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  MINIPIC_ERR_DEVICE_CHECK = 5, /* a kernel recorded out-of-range device data (see below) */
  MINIPIC_ERR_CAPACITY = 6      /* prefix cache: no free or released block left (or host memory ran out) */
} minipic_status;

typedef enum { MINIPIC_F32 = 0, MINIPIC_BF16 = 1 } minipic_dtype;

/* Bits of the device error word. */
#define MINIPIC_DEVERR_BLOCK_ID   1  /* a block table entry outside [0, num_blocks) */
#define MINIPIC_DEVERR_POSITION   2  /* a key or query position outside [0, max_pos) */
#define MINIPIC_DEVERR_SEQ_LEN    4  /* a length above max_blocks_per_seq * block_size or negative */
#define MINIPIC_DEVERR_TIMEOUT    8  /* a bounded wait for an asynchronous copy gave up (results invalid) */
#define MINIPIC_DEVERR_RANGE     16  /* prefill: a rotated key or scaled, rotated query element is outside the
                                        fp16 range of the QK^T operands (|x| > 65504); the score rows that
                                        use it are undefined (inf or NaN), all other rows are unaffected */

/* The paged KV pool (device memory, caller-owned). */
typedef struct {
  const void* k_pool;     /* [num_blocks][num_kv_heads][block_size][head_dim], unrotated keys */
  const void* v_pool;     /* same layout, values */
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t block_size;     /* must be 16 */
  int32_t head_dim;       /* 64 or 128 */
} minipic_kv_pool;

/* The rotary cos/sin table (device memory, caller-owned). */
typedef struct {
  const float* cos_sin;          /* [max_pos][head_dim] fp32, written by minipic_rope_table */
  int32_t max_pos;
  int32_t head_dim;              /* must equal the pool's head_dim */
  const uint16_t* cos_sin_f16;   /* [max_pos][head_dim] fp16 bit patterns, written by
                                    minipic_rope_table_f16 with the same max_pos, head_dim
                                    and base; read by the prefill and mixed calls (NULL
                                    there returns INVALID), ignored by decode (may be NULL) */
  const uint16_t* cos_sin_bf16;  /* [max_pos][2][3 head_dim / 2] bf16 bit patterns, written by
                                    minipic_rope_table_bf16 with the same max_pos, head_dim
                                    and base; read by the bf16 decode and the mixed call's
                                    decode part (NULL there returns INVALID), ignored by the
                                    fp32 decode and by prefill (may be NULL) */
} minipic_rope;

/* One decode token per request (MiniPIC section 2.1 score equation with the
 * query at position q_pos[r] over all seq_lens[r] stored keys of request r). */
typedef struct {
  const void* q;                /* [batch][num_q_heads][head_dim], unrotated */
  const int32_t* block_tables;  /* [batch][max_blocks_per_seq] physical block ids */
  const int32_t* block_starts;  /* [batch][max_blocks_per_seq] logical start position of each block */
  const int32_t* seq_lens;      /* [batch] number of stored keys of each request */
  const int32_t* q_pos;         /* [batch] position of each decode token */
  int32_t batch;
  int32_t max_blocks_per_seq;   /* row stride of the tables; seq_lens[r] <= this * block_size */
  void* out;                    /* [batch][num_q_heads][head_dim] */
  float* lse;                   /* [batch][num_q_heads] or NULL */
} minipic_decode_batch;

/* Chunked prefill: request r's query chunk is rows cu_q_lens[r] .. cu_q_lens[r+1]-1
 * of q; it attends to the request's kv_lens[r] stored keys, which include the
 * chunk's own keys as the last q_len ones.  Query i of the chunk sees keys
 * j <= kv_lens[r] - q_len + i (causal, bottom-right aligned by key index). */
typedef struct {
  const void* q;                /* [total_q][num_q_heads][head_dim], unrotated */
  const int32_t* cu_q_lens;     /* [batch + 1], cu_q_lens[0] = 0 */
  const int32_t* q_pos;         /* [total_q] position of each query token */
  const int32_t* block_tables;  /* [batch][max_blocks_per_seq] */
  const int32_t* block_starts;  /* [batch][max_blocks_per_seq] */
  const int32_t* kv_lens;       /* [batch], kv_lens[r] >= q_len of request r */
  int32_t batch;
  int32_t total_q;              /* cu_q_lens[batch] */
  int32_t max_q_len;            /* an upper bound of every chunk length (grid planning) */
  int32_t max_blocks_per_seq;
  void* out;                    /* [total_q][num_q_heads][head_dim] */
  float* lse;                   /* [total_q][num_q_heads] or NULL */
} minipic_prefill_batch;

/* Human-readable name of a status code (static string). */
const char* minipic_status_string(minipic_status status);

/* Fill the rotary table (MiniPIC section 2.1, "a cosine/sine table"):
 * cos_sin[p*head_dim + i] = cos(p theta_i), cos_sin[p*head_dim + d/2 + i] =
 * sin(p theta_i), theta_i = rope_base^(-2 i / head_dim), for 0 <= p < max_pos.
 * The angle p * theta_i is formed in double precision and the result rounded
 * to float.  cos_sin: device, at least max_pos * head_dim floats, caller-owned.
 * Errors: INVALID for null/misaligned/non-positive sizes/odd head_dim or
 * rope_base <= 0; CUDA on launch failure. */
minipic_status minipic_rope_table(float* cos_sin, int32_t max_pos, int32_t head_dim,
                                  double rope_base, minipic_stream_t stream);

/* The same table rounded to fp16 (MiniPIC section 2.1, the cosine/sine table
 * the key rotation reads): cos_sin_f16[p*head_dim + i] and [p*head_dim + d/2 + i]
 * hold cos and sin of p theta_i, formed in double precision and rounded once to
 * the nearest fp16 (IEEE binary16 bit patterns; values below 2^-14 become
 * subnormals, whose absolute error is at most 2^-25).  The chunked-prefill
 * kernels rotate keys with it in packed fp16 arithmetic, sixteen consecutive
 * positions of a block being sixteen consecutive rows.  cos_sin_f16: device,
 * at least max_pos * head_dim uint16 values, 16-byte aligned, caller-owned.
 * Errors as for minipic_rope_table. */
minipic_status minipic_rope_table_f16(uint16_t* cos_sin_f16, int32_t max_pos, int32_t head_dim,
                                      double rope_base, minipic_stream_t stream);

/* The table in the form the bf16 decode's packed-bf16 rotation reads (MiniPIC
 * section 2.1, the cosine/sine table), over signed angles: for position p and
 * sign sg (0: +p, 1: -p), row [p][sg] holds 3 head_dim / 2 values, cos, sin and
 * -sin of the angle (-1)^sg p theta_i at [i], [d/2 + i] and [d + i], i < d/2.
 * Each is the fp32 table's value (fp64 angle, CUDA's double sincos, rounded to
 * float) rounded to the nearest bf16 (bit patterns).  A rotation by a signed
 * angle reads one row: no conversion and no sign logic in the kernel.
 * cos_sin_bf16: device, at least max_pos * 3 * head_dim uint16 values, 16-byte
 * aligned, caller-owned; head_dim a multiple of 16.  Errors as for
 * minipic_rope_table. */
minipic_status minipic_rope_table_bf16(uint16_t* cos_sin_bf16, int32_t max_pos, int32_t head_dim,
                                       double rope_base, minipic_stream_t stream);

/* The three forms of the table in one pass (one fp64 sincos per entry):
 * any of cos_sin (as minipic_rope_table), cos_sin_f16 (as _f16) and
 * cos_sin_bf16 (as _bf16) may be NULL, not all three; the values are those of
 * the single-form calls.  Errors as for those calls. */
minipic_status minipic_rope_tables(float* cos_sin, uint16_t* cos_sin_f16, uint16_t* cos_sin_bf16,
                                   int32_t max_pos, int32_t head_dim, double rope_base,
                                   minipic_stream_t stream);

/* Workspace bytes minipic_attn_decode needs for this shape on the current
 * device (split-KV partial results).  0 means no workspace is needed.  The
 * value depends only on the arguments and the device's SM count. */
size_t minipic_attn_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t max_blocks_per_seq,
                                          int32_t block_size);

/* Decode attention over the position-free paged cache (split-KV with a
 * log-sum-exp merge of the splits).  Rotates q at q_pos and every gathered key
 * at its pi(j) from the table.  dtype selects f32 or bf16 for q, pools and out
 * (arithmetic is fp32; bf16 uses tensor-core products with bf16 operands).
 * workspace: device, >= minipic_attn_decode_workspace_size(...) bytes
 * (may be NULL when that size is 0).  Errors: INVALID, UNSUPPORTED, WORKSPACE,
 * CUDA; device-data problems are reported by minipic_device_error. */
minipic_status minipic_attn_decode(minipic_dtype dtype, int32_t num_q_heads,
                                   const minipic_kv_pool* kv, const minipic_rope* rope,
                                   const minipic_decode_batch* batch, float scale,
                                   void* workspace, size_t workspace_bytes,
                                   minipic_stream_t stream);

/* Mixed continuous batch in ONE launch: span-prefill chunks (as for
 * minipic_attn_prefill) and decode tokens (as for minipic_attn_decode) over the
 * same pool and table, scheduled in one grid so that tensor-core-bound prefill
 * tiles and HBM-bound decode splits share the SMs (the device side of MiniPIC's
 * interleaved span-prefill scheduling, section 2.2 "Scheduling").  Either batch
 * may be empty (batch 0).  Workspace: as for the decode batch
 * (minipic_attn_decode_workspace_size).  bf16 only.  Errors as above. */
minipic_status minipic_attn_mixed(minipic_dtype dtype, int32_t num_q_heads, const minipic_kv_pool* kv,
                                  const minipic_rope* rope, const minipic_prefill_batch* prefill,
                                  const minipic_decode_batch* decode, float scale, void* workspace,
                                  size_t workspace_bytes, minipic_stream_t stream);

/* The same decode kernel with the rotation compiled out: keys in the pool and
 * q are taken as already rotated (standard paged attention over a pre-rotated
 * cache).  It exists to measure what on-the-fly rotation costs against
 * identical memory traffic; rope may be NULL.  Same errors as above. */
minipic_status minipic_attn_decode_prerotated(minipic_dtype dtype, int32_t num_q_heads,
                                              const minipic_kv_pool* kv,
                                              const minipic_decode_batch* batch, float scale,
                                              void* workspace, size_t workspace_bytes,
                                              minipic_stream_t stream);

/* Decode for callers that cannot allocate device memory at the call: code
 * inside a fixed memory pool that must not grow, a serving loop where an
 * allocation could synchronize the device or fail under fragmentation, or a
 * plain C host with no device allocator of its own.  The paper has no
 * counterpart; this is a deployment convenience.  Same computation, arguments
 * and errors as minipic_attn_decode, except that the split-KV partial results
 * go to a fixed device array inside the library (MINIPIC_NOALLOC_SCRATCH_BYTES,
 * held on every GPU that loads the library until the process exits) instead of
 * a caller workspace.  Nothing is allocated by this call.
 *  - Shapes whose partial results exceed the fixed array (as reported by
 *    minipic_attn_decode_workspace_size) return MINIPIC_ERR_WORKSPACE.
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (no part of it needs to start at zero).  Calls whose work
 *    overlaps on the GPU race on it: serialize them.
 *  - The looked-up address is kept for the life of the process: do not use
 *    the library across cudaDeviceReset (or any teardown of the device's
 *    primary context) on that device. */
#define MINIPIC_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
minipic_status minipic_attn_decode_noalloc(minipic_dtype dtype, int32_t num_q_heads,
                                           const minipic_kv_pool* kv, const minipic_rope* rope,
                                           const minipic_decode_batch* batch, float scale,
                                           minipic_stream_t stream);

/* Workspace bytes minipic_attn_prefill needs (0 in this build). */
size_t minipic_attn_prefill_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t max_q_len,
                                           int32_t max_blocks_per_seq, int32_t block_size);

/* Chunked prefill over cached span blocks plus the chunk's own keys (the
 * uncached-span prefill of MiniPIC section 4 and the final-prompt prefill that
 * reads cached spans).  Keys are rotated at pi(j) into shared memory and the
 * products run on the tcgen05 tensor cores with TMEM accumulators.  Keys are
 * rotated in packed fp16 arithmetic with the fp16 table (rope->cos_sin_f16,
 * required); the query is rotated in fp32 with the fp32 table.  The rotated q
 * and k are fp16 for the QK^T product (10-bit mantissa: rotated elements must
 * stay within +-65504; an element outside sets MINIPIC_DEVERR_RANGE and the
 * rows that read it are undefined); softmax weights and V are bf16 for the P.V product;
 * accumulation is fp32.  bf16 only (f32 returns UNSUPPORTED).  The workspace
 * is not used (size 0).  Errors as for decode. */
minipic_status minipic_attn_prefill(minipic_dtype dtype, int32_t num_q_heads,
                                    const minipic_kv_pool* kv, const minipic_rope* rope,
                                    const minipic_prefill_batch* batch, float scale,
                                    void* workspace, size_t workspace_bytes,
                                    minipic_stream_t stream);

/* The same prefill kernel with the rotation compiled out: keys in the pool and
 * q are taken as already rotated (standard paged prefill over a pre-rotated
 * cache, bf16 products).  It exists to measure what on-the-fly rotation costs;
 * no table is needed.  bf16 only.  Errors as for minipic_attn_prefill. */
minipic_status minipic_attn_prefill_prerotated(minipic_dtype dtype, int32_t num_q_heads,
                                               const minipic_kv_pool* kv, const minipic_prefill_batch* batch,
                                               float scale, minipic_stream_t stream);

/* ------------------------------------------------------------------ cache append
 * Storing new tokens in the position-free cache (MiniPIC summary, section 2.1:
 * the cache holds unrotated key vectors k~_j, so a token's key is written
 * exactly as produced, with no rotation at any position; a block written this
 * way can later be read at any offset). */

/* Writable view of the pools (same layout as minipic_kv_pool). */
typedef struct {
  void* k_pool;           /* [num_blocks][num_kv_heads][block_size][head_dim] */
  void* v_pool;
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t block_size;     /* must be 16 */
  int32_t head_dim;       /* 64 or 128 */
} minipic_kv_pool_mut;

/* New tokens: token i of request r is row cu_new_lens[r] + i of k_new / v_new
 * and becomes the request's key index j = kv_start[r] + i, stored in block
 * block_tables[r][j / 16], slot j % 16, for every kv head. */
typedef struct {
  const void* k_new;            /* [total_new][num_kv_heads][head_dim], unrotated keys */
  const void* v_new;            /* [total_new][num_kv_heads][head_dim] */
  const int32_t* cu_new_lens;   /* [batch + 1], cu_new_lens[0] = 0 */
  const int32_t* kv_start;      /* [batch] key index of each request's first new token */
  const int32_t* block_tables;  /* [batch][max_blocks_per_seq] */
  int32_t batch;
  int32_t total_new;            /* cu_new_lens[batch] */
  int32_t max_new_len;          /* an upper bound of every request's new-token count (grid planning) */
  int32_t max_blocks_per_seq;
} minipic_kv_append_batch;

/* Copy the new keys and values into their slots (for a prefill chunk's own
 * tokens or one decode token per request).  Device memory throughout,
 * 16-byte aligned rows; dtype f32 or bf16 (the pools' and the new rows' type).
 * A block id outside [0, num_blocks) sets MINIPIC_DEVERR_BLOCK_ID, a key index
 * outside the table (or a negative kv_start) sets MINIPIC_DEVERR_SEQ_LEN; such
 * tokens are skipped, the rest are written.  Every slot must be the target of
 * at most one token of a call (two tokens mapped to one slot race).
 * Asynchronous on `stream`. */
minipic_status minipic_kv_append(minipic_dtype dtype, const minipic_kv_pool_mut* kv,
                                 const minipic_kv_append_batch* batch, minipic_stream_t stream);

/* ------------------------------------------------------------------ host offload
 * Moving whole blocks between the pools and host memory (MiniPIC summary,
 * section 3, item 5: unrotated blocks move between GPU and host with no
 * position to track or adjust).  A block's logical positions live in the
 * requests' block_starts, so a block may come back to any free physical id:
 * only the block tables change.
 *
 * host_k / host_v: page-locked host memory (cudaHostAlloc, cudaHostRegister or
 * a pinned torch tensor) of n blocks, [n][num_kv_heads][block_size][head_dim]
 * each, 16-byte aligned; the kernel reads or writes it directly over the
 * host link.  block_ids: device int32 [n].  An id outside [0, num_blocks) sets
 * MINIPIC_DEVERR_BLOCK_ID and that block is skipped.  Host memory that is not
 * page-locked returns MINIPIC_ERR_INVALID.  Asynchronous on `stream`: the host
 * buffer is complete (swap-out) or may be reused (swap-in) once the stream
 * reaches this point.  Within a swap-in call the ids must be distinct. */
minipic_status minipic_kv_swap_out(minipic_dtype dtype, const minipic_kv_pool* kv, const int32_t* block_ids,
                                   int32_t n, void* host_k, void* host_v, minipic_stream_t stream);
minipic_status minipic_kv_swap_in(minipic_dtype dtype, const minipic_kv_pool_mut* kv, const int32_t* block_ids,
                                  int32_t n, const void* host_k, const void* host_v, minipic_stream_t stream);

/* ------------------------------------------------------------------ span reuse (host)
 * The step that feeds the attention its tables (MiniPIC summary, section 2.2):
 * KV blocks are cached by a hash chain over their tokens, and two special
 * tokens at the start of a block change the chain.  For full block i of a
 * prompt (tokens x_i):
 *   default  h_i = H(h_{i-1}, x_i), with h_{-1} = h_0
 *   SSEP     h_i = H(h_0, x_i)        the chain restarts: the span is cached
 *                                     whatever precedes it
 *   PDEP     h_i = H(h_0, x_{<=i})    the block depends on the whole prompt
 *                                     before it, across restarts
 * H(p, t) is 64-bit FNV-1a over p (8 bytes, little endian) and then the tokens
 * (4 bytes each, little endian).  Users pad spans to block boundaries so that
 * the special tokens open blocks.  Only full blocks are hashed; a trailing
 * partial block stays private to its request.  Host memory and host code
 * only; no GPU is involved. */

/* Hashes of the n_tokens / block_size full blocks of one prompt into hashes
 * (host, max_hashes capacity); *n_hashes receives their count.  Errors:
 * INVALID for null pointers, a non-positive block size or too small a
 * capacity. */
minipic_status minipic_block_hashes(const int32_t* tokens, int32_t n_tokens, int32_t block_size, int32_t ssep_token,
                                    int32_t pdep_token, uint64_t h0, uint64_t* hashes, int32_t max_hashes,
                                    int32_t* n_hashes);

/* A prefix cache over a pool of num_blocks physical blocks: maps a block hash
 * to the physical block that holds (or will hold) its unrotated keys and
 * values.  Not thread-safe; the caller serializes calls on one cache. */
typedef struct minipic_prefix_cache minipic_prefix_cache;
minipic_status minipic_prefix_cache_create(int32_t num_blocks, minipic_prefix_cache** cache);
void minipic_prefix_cache_destroy(minipic_prefix_cache* cache);

/* Blocks of one request with n_blocks blocks, the first n_hashed of them full
 * and hashed (minipic_block_hashes), the rest private: block_table[b] receives
 * the physical block, block_starts[b] = b * block_size its logical start in
 * this request, and is_new[b] = 1 when the block's keys and values still have
 * to be computed and appended (a miss), 0 when the cache already holds them
 * (one physical block may appear in many requests at different starts, which
 * the position-free attention reads correctly).  Each listed block gains one
 * reference.  A miss takes a never-used block, else evicts the unreferenced
 * cached block released longest ago; when neither exists the call returns
 * CAPACITY and leaves the cache as it was.  Host arrays of n_blocks entries. */
minipic_status minipic_prefix_cache_assign(minipic_prefix_cache* cache, const uint64_t* hashes, int32_t n_hashed,
                                           int32_t n_blocks, int32_t block_size, int32_t* block_table,
                                           int32_t* block_starts, uint8_t* is_new);

/* Drop one reference per listed block id (a block listed k times loses k).
 * An unreferenced cached block stays findable until a miss evicts it; a
 * private one just becomes free.  INVALID (and no change) when an id is out
 * of range or has fewer references than listed. */
minipic_status minipic_prefix_cache_release(minipic_prefix_cache* cache, const int32_t* block_ids, int32_t n);

/* Read the device error word (MINIPIC_DEVERR_* bits, 0 if none) of the current
 * device after the work queued on `stream` has finished (this call
 * synchronizes the stream), and reset it to 0 when `clear` is nonzero.
 * Returns DEVICE_CHECK if any bit was set, OK otherwise, CUDA on failure. */
minipic_status minipic_device_error(int32_t* flags_out, int32_t clear, minipic_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MINIPIC_H */
