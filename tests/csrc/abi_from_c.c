/* A plain C99 program that uses the library through include/minipic.h only:
 * status names, workspace sizing, the SSEP/PDEP block-hash chain and the prefix
 * cache (the host calls, which need no GPU).  It prints what it gets; the test
 * that builds and runs it compares the hashes and tables with the oracle. */
#include <stdint.h>
#include <stdio.h>

#include "minipic.h"

static int put_tables(const char* tag, const int32_t* t, const int32_t* s, const uint8_t* f, int n) {
  printf("%s", tag);
  for (int i = 0; i < n; ++i) printf(" %d:%d:%d", t[i], s[i], (int)f[i]);
  printf("\n");
  return 0;
}

int main(void) {
  const int32_t ssep = -7, pdep = -9, bs = 4;
  /* block 0 plain, block 1 opens with SSEP, block 2 with PDEP, 2 trailing tokens */
  const int32_t p1[14] = {1, 2, 3, 4, ssep, 11, 12, 13, pdep, 21, 22, 23, 5, 6};
  /* the same SSEP block one block later, after a different prefix */
  const int32_t p2[16] = {7, 7, 7, 7, 8, 8, 8, 8, ssep, 11, 12, 13, pdep, 31, 32, 33};
  uint64_t h1[3], h2[4];
  int32_t n1 = 0, n2 = 0;
  minipic_prefix_cache* cache = NULL;
  int32_t t1[4], s1[4], t2[4], s2[4];
  uint8_t f1[4], f2[4];

  printf("status %s\n", minipic_status_string(MINIPIC_ERR_INVALID));
  printf("workspace %d\n", minipic_attn_decode_workspace_size(64, 32, 8, 128, 512, 16) > 0);
  if (minipic_block_hashes(p1, 14, bs, ssep, pdep, 0x1234u, h1, 3, &n1) != MINIPIC_OK || n1 != 3) return 1;
  if (minipic_block_hashes(p2, 16, bs, ssep, pdep, 0x1234u, h2, 4, &n2) != MINIPIC_OK || n2 != 4) return 2;
  printf("hashes1 %llu %llu %llu\n", (unsigned long long)h1[0], (unsigned long long)h1[1],
         (unsigned long long)h1[2]);
  printf("hashes2 %llu %llu %llu %llu\n", (unsigned long long)h2[0], (unsigned long long)h2[1],
         (unsigned long long)h2[2], (unsigned long long)h2[3]);
  if (minipic_prefix_cache_create(16, &cache) != MINIPIC_OK) return 3;
  if (minipic_prefix_cache_assign(cache, h1, n1, 4, bs, t1, s1, f1) != MINIPIC_OK) return 4;
  if (minipic_prefix_cache_assign(cache, h2, n2, 4, bs, t2, s2, f2) != MINIPIC_OK) return 5;
  put_tables("tables1", t1, s1, f1, 4);
  put_tables("tables2", t2, s2, f2, 4);
  if (minipic_prefix_cache_release(cache, t1, 4) != MINIPIC_OK) return 6;
  minipic_prefix_cache_destroy(cache);
  printf("done\n");
  return 0;
}
