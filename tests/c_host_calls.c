/*
 * A plain C99 host of libdsa.so: includes dsa.h as C, links the library and
 * makes the calls that need no GPU (config checks, workspace layout, score
 * windows, split suggestion, row building), plus device calls with NULL
 * arguments, which must be refused on the host before anything is launched.
 * Prints "ok" and exits 0 when every check holds; tests/test_c_host.py
 * compiles and runs it.
 */
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include "dsa.h"

static int failures = 0;

#define CHECK(cond)                                                    \
  do {                                                                 \
    if (!(cond)) {                                                     \
      fprintf(stderr, "check failed at line %d: %s (last error: %s)\n", \
              __LINE__, #cond, dsa_last_error());                      \
      ++failures;                                                      \
    }                                                                  \
  } while (0)

static dsa_config_t decode_config(void) {
  /* decode, batch 64, 32K context, top-k 2048, 64 query / 8 KV heads */
  dsa_config_t c;
  memset(&c, 0, sizeof(c));
  c.num_q_heads = 64;
  c.num_kv_heads = 8;
  c.head_dim = 128;
  c.idx_heads = 64;
  c.idx_dim = 128;
  c.page_size = 64;
  c.topk = 2048;
  c.num_splits = 19;
  c.max_rows = 64;
  c.max_reqs = 64;
  c.max_pages_per_req = 512;
  c.score_width = 32768;
  c.num_pages = 32768;
  c.block_rows = 1;
  c.idx_key_dtype = DSA_KEY_BF16;
  c.sm_scale = 0.08838834764831845f;
  c.flags = 0;
  c.score_buffer_bytes = 0;
  return c;
}

int main(int argc, char **argv) {
  dsa_config_t cfg = decode_config();
  /* the struct layouts the Python binding mirrors (argv[1..4]: its sizes
   * and the offset of score_buffer_bytes) */
  if (argc == 5) {
    long want[4];
    int i;
    for (i = 0; i < 4; ++i) sscanf(argv[i + 1], "%ld", &want[i]);
    CHECK((long)sizeof(dsa_config_t) == want[0]);
    CHECK((long)offsetof(dsa_config_t, score_buffer_bytes) == want[1]);
    CHECK((long)sizeof(dsa_step_args_t) == want[2]);
    CHECK((long)sizeof(dsa_workspace_layout_t) == want[3]);
  } else {
    CHECK(argc == 1);
  }
  CHECK(strlen(dsa_version()) > 0);
  CHECK(dsa_validate_config(&cfg) == DSA_OK);

  /* an invalid config is refused with its reason */
  {
    dsa_config_t bad = cfg;
    bad.head_dim = 96;
    CHECK(dsa_validate_config(&bad) == DSA_ERR_UNSUPPORTED);
    CHECK(strstr(dsa_last_error(), "head_dim") != NULL);
    CHECK(dsa_validate_config(NULL) == DSA_ERR_INVALID_ARG);
  }

  /* workspace: size = layout total, regions 256-byte aligned and in order */
  {
    size_t bytes = 0;
    dsa_workspace_layout_t lay;
    CHECK(dsa_workspace_size(&cfg, &bytes) == DSA_OK);
    CHECK(dsa_workspace_layout(&cfg, &lay) == DSA_OK);
    CHECK(bytes == lay.total);
    CHECK(lay.scores % 256 == 0 && lay.topk_idx % 256 == 0 && lay.part_acc % 256 == 0);
    CHECK(lay.status < lay.scores && lay.scores < lay.topk_idx && lay.key_hist < lay.total);
    CHECK(lay.topk_idx - lay.scores >= (size_t)64 * 32768 * 4);
  }

  /* score windows under a byte budget */
  {
    int32_t wr = 0, nw = 0;
    CHECK(dsa_score_windows(&cfg, &wr, &nw) == DSA_OK && wr == 64 && nw == 1);
    dsa_config_t win = cfg;
    win.score_buffer_bytes = (int64_t)20 * 32768 * 4;
    CHECK(dsa_score_windows(&win, &wr, &nw) == DSA_OK && wr == 20 && nw == 4);
    win.score_buffer_bytes = 100;  /* below one score row */
    CHECK(dsa_validate_config(&win) == DSA_ERR_INVALID_ARG);
  }

  /* the split count the library suggests for 152 SMs */
  {
    int32_t s = 0;
    CHECK(dsa_suggest_num_splits(&cfg, 152, &s) == DSA_OK && s == 19);
  }

  /* rows of a mixed step: one decode token, one 5-token prefill chunk */
  {
    dsa_config_t mix = cfg;
    int32_t cache_len[2] = {100, 12};
    int32_t new_tokens[2] = {1, 5};
    int32_t row_req[64], row_len[64], row_pos[64], block_first[64], block_nrows[64];
    int32_t nr = -1, nb = -1;
    mix.block_rows = 4;
    CHECK(dsa_build_rows(&mix, 2, cache_len, new_tokens, row_req, row_len, row_pos, block_first,
                         block_nrows, &nr, &nb) == DSA_OK);
    CHECK(nr == 6 && nb == 3);
    CHECK(row_req[0] == 0 && row_len[0] == 100 && row_pos[0] == 99);
    CHECK(row_req[1] == 1 && row_len[1] == 8 && row_len[5] == 12 && row_pos[5] == 11);
    CHECK(block_first[0] == 0 && block_nrows[0] == 1);
    CHECK(block_first[1] == 1 && block_nrows[1] == 4 && block_first[2] == 5 && block_nrows[2] == 1);
    CHECK(row_len[6] == 0 && block_nrows[3] == 0);  /* padding */
    new_tokens[1] = 13;  /* more new tokens than the cache holds */
    CHECK(dsa_build_rows(&mix, 2, cache_len, new_tokens, row_req, row_len, row_pos, block_first,
                         block_nrows, &nr, &nb) == DSA_ERR_INVALID_ARG);
  }

  /* device calls refuse NULL arguments on the host, before any launch */
  {
    dsa_step_args_t args;
    memset(&args, 0, sizeof(args));
    CHECK(dsa_step(&cfg, NULL, NULL, NULL) == DSA_ERR_INVALID_ARG);
    CHECK(dsa_step(&cfg, &args, NULL, NULL) == DSA_ERR_INVALID_ARG);
    CHECK(dsa_topk(&cfg, NULL, NULL, NULL, NULL, NULL) == DSA_ERR_INVALID_ARG);
    CHECK(dsa_merge(&cfg, NULL, NULL, NULL, NULL, NULL, NULL) == DSA_ERR_INVALID_ARG);
    CHECK(dsa_indexer_scores_window(&cfg, 0, 65, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                    NULL, NULL, NULL) == DSA_ERR_INVALID_ARG);
    CHECK(strstr(dsa_last_error(), "row window") != NULL);
  }

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
