/* Plain C99 consumer of include/rvq.h: includes the header and calls every
 * entry point through an early-return path (no GPU needed).  Built with
 * -std=c99 -Wall -Werror -pedantic, as the ABI discipline of omnivoice.cpp
 * ARCHITECTURE.md ("ABI guarantee") asks of its own header. */
#include <stdio.h>
#include <string.h>

#include "rvq.h"

static int failures = 0;
#define EXPECT(cond)                                                   \
  do {                                                                 \
    if (!(cond)) {                                                     \
      fprintf(stderr, "abi_c: line %d: %s\n", __LINE__, #cond);        \
      failures++;                                                      \
    }                                                                  \
  } while (0)

int main(void) {
  rvq_dims ok = {1024, 64, 1024, 8};
  rvq_dims bad_d = {1024, 32, 1024, 8};
  rvq_dims zero = {0, 64, 1024, 8};
  rvq_dims lfq = {768, 8, 1024, 32, RVQ_METRIC_COSINE};
  rvq_dims bad_metric = {1024, 64, 1024, 8, 7};
  rvq_weights w;
  int32_t fake_codes[4];
  memset(&w, 0, sizeof w);

  EXPECT(rvq_dims_supported(ok) == RVQ_OK);
  EXPECT(rvq_dims_supported(bad_d) == RVQ_ERR_UNSUPPORTED);
  EXPECT(rvq_dims_supported(zero) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_dims_supported(lfq) == RVQ_OK);
  EXPECT(rvq_dims_supported(bad_metric) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_tables_bytes(ok) > 0);
  EXPECT(rvq_tables_bytes(bad_d) == 0);
  EXPECT(rvq_encode_scratch_bytes(ok, 1000, 8) >= rvq_encode_min_scratch_bytes(ok, 8));
  EXPECT(rvq_encode_min_scratch_bytes(ok, 9) == 0);
  EXPECT(rvq_prepare(ok, NULL, NULL, 0, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_prepare(ok, &w, NULL, 0, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_encode(ok, NULL, NULL, 10, 8, NULL, NULL, 0, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_encode(ok, NULL, NULL, 0, 8, NULL, NULL, 0, NULL) == RVQ_OK); /* empty batch */
  EXPECT(rvq_encode(ok, NULL, NULL, 10, 0, NULL, NULL, 0, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_encode(ok, NULL, NULL, -1, 8, NULL, NULL, 0, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_decode(ok, NULL, fake_codes, 1, 8, NULL, NULL, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_decode(ok, NULL, NULL, 1, 9, NULL, NULL, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_reconstruct(bad_d, NULL, NULL, 1, 8, NULL, NULL, NULL, 0, NULL) == RVQ_ERR_UNSUPPORTED);
  EXPECT(rvq_pipeline_workspace_bytes(ok, 8, 1024) > 0);
  EXPECT(rvq_pipeline_workspace_bytes(ok, 9, 1024) == 0);
  EXPECT(rvq_pipeline_create(ok, 8, 1024, NULL, 0, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_pipeline_destroy(NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(rvq_pipeline_reconstruct(NULL, NULL, NULL, 1, NULL, NULL) == RVQ_ERR_INVALID_ARG);
  EXPECT(strcmp(rvq_status_string(RVQ_OK), "ok") == 0);
  EXPECT(rvq_status_string(RVQ_ERR_CUDA) != NULL);
  EXPECT(rvq_version() != NULL && strlen(rvq_version()) > 0);
  {
    char want[32];
    snprintf(want, sizeof(want), "%d.%d.%d", RVQ_VERSION_MAJOR, RVQ_VERSION_MINOR, RVQ_VERSION_PATCH);
    EXPECT(strstr(rvq_version(), want) != NULL); /* the string and the header macros agree */
  }
  {
    const int64_t prev = rvq_set_stream_max_frames(-1); /* query only */
    EXPECT(prev >= 0);
    EXPECT(rvq_set_stream_max_frames(5) == prev);
    EXPECT(rvq_set_stream_max_frames(-1) == 5);
    EXPECT(rvq_set_stream_max_frames(prev) == 5);
    EXPECT(rvq_set_stream_max_frames(-7) == prev);
  }
  {
    /* argument checks and the shapes that never take the small-batch kernels
     * answer without the CUDA runtime */
    rvq_dims dm = {256, 64, 1024, 8, RVQ_METRIC_L2, 0, 0};
    int64_t plan[6] = {7, 7, 7, 7, 7, 7};
    EXPECT(rvq_stream_plan(dm, 0, 16, plan) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_stream_plan(dm, 9, 16, plan) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_stream_plan(dm, 8, -1, plan) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_stream_plan(dm, 8, 16, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(plan[0] == 7 && plan[5] == 7);
    const int64_t prev = rvq_set_stream_max_frames(100);
    EXPECT(rvq_stream_plan(dm, 8, 101, plan) == RVQ_OK && plan[0] == 0 && plan[4] == 0);
    EXPECT(rvq_stream_plan(dm, 8, 0, plan) == RVQ_OK && plan[0] == 0);
    rvq_set_stream_max_frames(prev);
    dm.K = 8192; /* d = 64 with K > 4096: tile kernels only */
    EXPECT(rvq_stream_plan(dm, 8, 16, plan) == RVQ_OK && plan[0] == 0);
  }
  {
    /* the no-allocation encode refuses bad calls before any CUDA call */
    rvq_dims dm = {1024, 64, 1024, 8, RVQ_METRIC_L2, 0, 0};
    const void *tab = (const void *)(uintptr_t)0x100000;   /* never dereferenced */
    const float *x = (const float *)(uintptr_t)0x200000;
    int32_t *codes = (int32_t *)(uintptr_t)0x300000;
    EXPECT(rvq_encode_static(dm, NULL, x, 10, 8, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, NULL, 10, 8, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, x, 10, 8, NULL, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, x, 10, 0, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, x, 10, 9, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, x, -1, 8, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, NULL, NULL, 0, 8, NULL, NULL) == RVQ_OK); /* empty batch */
    EXPECT(rvq_encode_static(dm, (const void *)(uintptr_t)0x100010, x, 10, 8, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, (const float *)(uintptr_t)0x200004, 10, 8, codes, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_encode_static(dm, tab, x, 10, 8, (int32_t *)(uintptr_t)0x300008, NULL) == RVQ_ERR_INVALID_ARG);
    /* (16 MiB - 256) / (8 * 64 * 4) = 8191 frames fit; 8192 do not */
    EXPECT(rvq_encode_static(dm, tab, x, 8192, 8, codes, NULL) == RVQ_ERR_WORKSPACE);
    EXPECT(rvq_encode_static(bad_d, tab, x, 10, 8, codes, NULL) == RVQ_ERR_UNSUPPORTED);
  }
  {
    /* the readers and the cancel hook check their pointers first */
    int64_t n = 0;
    EXPECT(rvq_read_error_count(NULL, &n, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_read_error_count((const int64_t *)(uintptr_t)0x100000, NULL, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_read_error_count((const int64_t *)(uintptr_t)0x100004, &n, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_read_status((const void *)(uintptr_t)0x100008, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(rvq_pipeline_set_cancel(NULL, NULL, NULL) == RVQ_ERR_INVALID_ARG);
    EXPECT(strcmp(rvq_status_string(RVQ_ERR_CANCELLED), "cancelled") == 0);
    EXPECT(strcmp(rvq_status_string(RVQ_ERR_TIMEOUT), "device wait timed out") == 0);
    EXPECT(rvq_status_string(RVQ_ERR_INTERNAL) != NULL && strcmp(rvq_status_string(RVQ_ERR_INTERNAL), "unknown status") != 0);
  }
  if (failures == 0) printf("abi_c: ok\n");
  return failures == 0 ? 0 : 1;
}
