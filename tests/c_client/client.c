/* A plain C11 client of libcsa2: includes the public header, links the shared library,
 * and checks host-side behaviour that needs no GPU (argument checks answered before any
 * launch, the size queries, the status strings).  Prints "ok" and exits 0 on success;
 * otherwise prints the failed check and exits 1. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "csa2.h"

static int failures = 0;
#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__); \
      ++failures;                                                \
    }                                                            \
  } while (0)

int main(void) {
  /* a fake, 16-byte aligned device address: nothing is dereferenced before the checks */
  void* fake = (void*)(uintptr_t)4096;
  const int32_t* fi = (const int32_t*)fake;
  csa2_pages pages = {1, fi, fi, 1, 1, 64};
  csa2_index_args ia;
  memset(&ia, 0, sizeof ia);

  CHECK(csa2_version() >= 10000);
  CHECK(strlen(csa2_status_string(CSA2_OK)) > 0);
  CHECK(strlen(csa2_status_string(CSA2_ERR_TIMEOUT)) > 0);

  /* write path: null H / weights */
  CHECK(csa2_kv_write(NULL, NULL, NULL, NULL, NULL, 4, 64, 1, 0, NULL, 4, NULL, NULL) ==
        CSA2_ERR_INVALID_ARGUMENT);
  /* indexer: null argument blocks */
  CHECK(csa2_index(CSA2_FULL, NULL, NULL, NULL, 16, NULL, NULL, NULL, NULL) ==
        CSA2_ERR_INVALID_ARGUMENT);
  /* a page size other than 64 is not implemented */
  pages.page_size = 32;
  ia.num_q = 1;
  ia.q_seq = fi;
  ia.max_q_per_seq = 1;
  CHECK(csa2_index(CSA2_FULL, (const uint16_t*)fake, (const uint16_t*)fake, NULL, 16,
                   (int32_t*)fake, &pages, &ia, NULL) == CSA2_ERR_UNSUPPORTED);
  pages.page_size = 64;
  /* attention: more entries than CSA2_ATTN_MAX_TOPK, and num_q < 1 */
  CHECK(csa2_sparse_attn((const uint16_t*)fake, (const uint8_t*)fake, (const uint8_t*)fake, fi,
                         &pages, (float*)fake, NULL, 1, fi, CSA2_ATTN_MAX_TOPK + 1, 0.04f, NULL, 0,
                         NULL, NULL) == CSA2_ERR_UNSUPPORTED);
  CHECK(csa2_sparse_attn((const uint16_t*)fake, (const uint8_t*)fake, (const uint8_t*)fake, fi,
                         &pages, (float*)fake, NULL, 0, fi, 16, 0.04f, NULL, 0, NULL, NULL) ==
        CSA2_ERR_INVALID_ARGUMENT);
  /* the no-workspace variant refuses what its fixed array cannot hold */
  CHECK(csa2_attn_workspace_size(8, CSA2_ATTN_MAX_TOPK) > CSA2_ATTN_STATIC_SCRATCH_BYTES);
  CHECK(csa2_sparse_attn_static((const uint16_t*)fake, (const uint8_t*)fake,
                                (const uint8_t*)fake, fi, &pages, (float*)fake, NULL, 8, fi,
                                CSA2_ATTN_MAX_TOPK, 0.04f, NULL, NULL) == CSA2_ERR_UNSUPPORTED);
  /* chunked attention: num_q not a multiple of the chunk */
  CHECK(csa2_sparse_attn_chunked((const uint16_t*)fake, (const uint8_t*)fake,
                                 (const uint8_t*)fake, fi, &pages, (float*)fake, NULL, 6, fi, 4,
                                 16, 0.04f, fake, 1u << 30, NULL, NULL) ==
        CSA2_ERR_INVALID_ARGUMENT);
  /* codec geometry */
  CHECK(csa2_quantize(NULL, NULL, NULL, NULL, 4, 24, 4, NULL, NULL) == CSA2_ERR_UNSUPPORTED);
  CHECK(csa2_quantize_mx(NULL, NULL, NULL, NULL, 4, 48, 4, NULL, NULL) == CSA2_ERR_UNSUPPORTED);
  /* persistent tier record sizes */
  CHECK(csa2_page_export_bytes(32) == 34816);
  CHECK(csa2_page_export_bytes(16) == 33792);
  CHECK(csa2_page_export_bytes(8) == 0);
  /* sizes are plain host arithmetic */
  CHECK(csa2_index_workspace_size(CSA2_REINDEX, 64, 2048, 8192) == (size_t)64 * 8192 * 4);
  CHECK(csa2_index_workspace_size(CSA2_REUSE, 64, 2048, 8192) == 0);
  CHECK(csa2_chunk_attn_workspace_size(6, 4, 16) == 0);
  /* status read with a null device word */
  CHECK(csa2_read_status(NULL, NULL, NULL) == CSA2_ERR_INVALID_ARGUMENT);
  /* bounded-wait diagnostic: limit range and null status word */
  CHECK(csa2_check_bounded_wait(0, 1024, NULL, NULL) == CSA2_ERR_INVALID_ARGUMENT);
  CHECK(csa2_check_bounded_wait(0, (1u << 20) + 1, (int32_t*)fake, NULL) ==
        CSA2_ERR_INVALID_ARGUMENT);

  if (failures) return 1;
  printf("ok\n");
  return 0;
}
