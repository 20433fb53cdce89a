/* The C ABI used from plain C (no Python, no GPU): configuration defaults,
 * error strings, the scheduler's plan for an 8-rank allreduce on copy engines
 * and the two-domain stage scheduler.  Prints one line per check and exits 0
 * when every check holds. */
#include <stdio.h>
#include <string.h>

#include "hoc.h"
#include "hoc_sched.h"

#define CHECK(cond)                                         \
  do {                                                      \
    if (!(cond)) {                                          \
      printf("FAIL %s:%d: %s\n", __FILE__, __LINE__, #cond); \
      return 1;                                             \
    }                                                       \
  } while (0)

int main(void) {
  hocConfig_t cfg;
  CHECK(hoc_config_default(&cfg) == HOC_SUCCESS);
  CHECK(cfg.path == HOC_PATH_AUTO);
  CHECK(strcmp(hoc_error_string(HOC_ERR_INVALID_ARG), "invalid argument") == 0);
  printf("config and error strings ok\n");

  /* allreduce of 8 ranks x 1 Mi bf16 on copy engines in 256 KiB chunks: every
   * block's chunks are reduced once (REDUCE items) and copied to the 7 other
   * ranks (COPY items) */
  cfg.path = HOC_PATH_CE;
  cfg.chunk_bytes = 256 * 1024;
  size_t n = 0;
  CHECK(hoc_plan_query(8, &cfg, HOC_OP_ALLREDUCE, 1u << 20, HOC_BFLOAT16, NULL, NULL, 0, &n) == HOC_SUCCESS);
  static hocPlanItem_t items[4096];
  CHECK(n > 0 && n <= 4096);
  CHECK(hoc_plan_query(8, &cfg, HOC_OP_ALLREDUCE, 1u << 20, HOC_BFLOAT16, NULL, items, n, &n) == HOC_SUCCESS);
  size_t reduced = 0, copied = 0;
  for (size_t i = 0; i < n; ++i) {
    if (items[i].kind == HOC_ITEM_REDUCE) reduced += items[i].bytes;
    if (items[i].kind == HOC_ITEM_COPY) copied += items[i].bytes;
  }
  CHECK(reduced == (size_t)(1u << 20) * 2);     /* every element's output written once */
  CHECK(copied == (size_t)(1u << 20) * 2 * 7);  /* and copied to the 7 other ranks */
  printf("allreduce plan ok: %zu items\n", n);

  /* sizes past the library's limits are rejected before any plan: a rank
   * span above 2^40 bytes, a count whose byte size wraps size_t, and more
   * than 2^24 chunks per rank buffer */
  CHECK(hoc_plan_query(8, &cfg, HOC_OP_ALLREDUCE, ((size_t)1 << 39) + 1, HOC_BFLOAT16, NULL, NULL, 0, &n) ==
        HOC_ERR_INVALID_ARG);
  CHECK(hoc_plan_query(8, &cfg, HOC_OP_ALLREDUCE, (size_t)-1, HOC_FLOAT32, NULL, NULL, 0, &n) == HOC_ERR_INVALID_ARG);
  cfg.chunk_bytes = 256;
  CHECK(hoc_plan_query(8, &cfg, HOC_OP_SENDRECV, ((size_t)1 << 32) + 256, HOC_UINT8, NULL, NULL, 0, &n) ==
        HOC_ERR_INVALID_ARG);
  cfg.chunk_bytes = 256 * 1024;
  printf("size limits ok\n");

  /* 4 GPUs in 2 nodes (peers 0-1 and 2-3): GPU 0 sends 100 bytes to GPU 2 and
   * GPU 2 sends 100 to GPU 0.  Each inter-node flow is staged through the
   * sender's peer (Eqs. 2-5), so T carries it on NVLink 0 -> 1 and 2 -> 3 and
   * on RDMA 1 -> 3 and 3 -> 1, and the stages sum to T (Eq. 7). */
  int node_of[4] = {0, 0, 1, 1};
  int sym[4] = {1, 0, 3, 2};
  uint64_t C[16] = {0};
  C[0 * 4 + 2] = 100;
  C[2 * 4 + 0] = 100;
  uint64_t T[16], stages[16 * 8];
  double taus[8], total = 0.0;
  int ns = 0;
  CHECK(hoc_topo_schedule(4, node_of, sym, C, 400, 50, T, stages, taus, 8, &ns, &total) == HOC_SUCCESS);
  CHECK(ns >= 1 && ns <= 8 && total > 0.0);
  for (int c = 0; c < 16; ++c) {
    uint64_t sum = 0;
    for (int s = 0; s < ns; ++s) sum += stages[s * 16 + c];
    CHECK(sum == T[c]);
  }
  printf("topo schedule ok: %d stages, total %.3f\n", ns, total);
  printf("ABI OK\n");
  return 0;
}
