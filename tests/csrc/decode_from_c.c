/* A plain C (C11) program that runs the decode hot path through include/minipic.h
 * and the CUDA runtime only: it reads a decode batch from binary files (fp32
 * q, pools and rope base; int32 tables), allocates device memory, builds the
 * rotary table, sizes the workspace, calls minipic_attn_decode, reads the
 * device error word and writes out and lse back.  Usage:
 *   decode_from_c <dir>   (dir holds shape.i32 and the arrays named below) */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "minipic.h"

static void* slurp(const char* dir, const char* name, size_t bytes) {
  char path[1024];
  FILE* f;
  void* p = malloc(bytes ? bytes : 1);
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "rb");
  if (!f || !p || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %s\n", path);
    exit(10);
  }
  fclose(f);
  return p;
}

static void* upload(const void* h, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess || cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "upload failed\n");
    exit(11);
  }
  return d;
}

int main(int argc, char** argv) {
  const char* dir;
  int32_t* shape;
  int32_t B, Hq, Hkv, d, nblk, mb, max_pos;
  double base;
  size_t qn, pn, tn;
  minipic_kv_pool kv;
  minipic_rope rope;
  minipic_decode_batch batch;
  float *cos_sin = NULL, *out_h, *lse_h;
  int32_t flags = 0;
  void* ws = NULL;
  size_t ws_bytes;
  minipic_status st;
  FILE* f;
  char path[1024];

  if (argc != 2) return 2;
  dir = argv[1];
  shape = (int32_t*)slurp(dir, "shape.i32", 7 * sizeof(int32_t));
  B = shape[0]; Hq = shape[1]; Hkv = shape[2]; d = shape[3]; nblk = shape[4]; mb = shape[5]; max_pos = shape[6];
  base = *(double*)slurp(dir, "base.f64", sizeof(double));
  qn = (size_t)B * Hq * d;
  pn = (size_t)nblk * Hkv * 16 * d;
  tn = (size_t)B * mb;

  kv.k_pool = upload(slurp(dir, "k.f32", pn * 4), pn * 4);
  kv.v_pool = upload(slurp(dir, "v.f32", pn * 4), pn * 4);
  kv.num_blocks = nblk;
  kv.num_kv_heads = Hkv;
  kv.block_size = 16;
  kv.head_dim = d;

  if (cudaMalloc((void**)&cos_sin, (size_t)max_pos * d * 4) != cudaSuccess) return 12;
  if (minipic_rope_table(cos_sin, max_pos, d, base, NULL) != MINIPIC_OK) return 13;
  rope.cos_sin = cos_sin;
  rope.max_pos = max_pos;
  rope.head_dim = d;
  rope.cos_sin_f16 = NULL;   /* not read by the fp32 decode */
  rope.cos_sin_bf16 = NULL;  /* read by the bf16 decode only */

  batch.q = upload(slurp(dir, "q.f32", qn * 4), qn * 4);
  batch.block_tables = (const int32_t*)upload(slurp(dir, "tables.i32", tn * 4), tn * 4);
  batch.block_starts = (const int32_t*)upload(slurp(dir, "starts.i32", tn * 4), tn * 4);
  batch.seq_lens = (const int32_t*)upload(slurp(dir, "seq_lens.i32", (size_t)B * 4), (size_t)B * 4);
  batch.q_pos = (const int32_t*)upload(slurp(dir, "q_pos.i32", (size_t)B * 4), (size_t)B * 4);
  batch.batch = B;
  batch.max_blocks_per_seq = mb;
  if (cudaMalloc(&batch.out, qn * 4) != cudaSuccess || cudaMalloc((void**)&batch.lse, (size_t)B * Hq * 4) != cudaSuccess)
    return 14;

  ws_bytes = minipic_attn_decode_workspace_size(B, Hq, Hkv, d, mb, 16);
  if (ws_bytes && (cudaMalloc(&ws, ws_bytes) != cudaSuccess || cudaMemset(ws, 0, ws_bytes) != cudaSuccess)) return 15;
  st = minipic_attn_decode(MINIPIC_F32, Hq, &kv, &rope, &batch, 0.0f, ws, ws_bytes, NULL);
  if (st != MINIPIC_OK) {
    fprintf(stderr, "decode: %s\n", minipic_status_string(st));
    return 16;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return 17;
  out_h = (float*)malloc(qn * 4);
  lse_h = (float*)malloc((size_t)B * Hq * 4);
  if (cudaMemcpy(out_h, batch.out, qn * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(lse_h, batch.lse, (size_t)B * Hq * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 18;
  snprintf(path, sizeof path, "%s/out.f32", dir);
  f = fopen(path, "wb");
  if (!f || fwrite(out_h, 4, qn, f) != qn) return 19;
  fclose(f);
  snprintf(path, sizeof path, "%s/lse.f32", dir);
  f = fopen(path, "wb");
  if (!f || fwrite(lse_h, 4, (size_t)B * Hq, f) != (size_t)B * Hq) return 20;
  fclose(f);
  if (minipic_device_error(&flags, 1, NULL) != MINIPIC_OK) return 21;
  printf("device_error %d\n", flags);
  return 0;
}
