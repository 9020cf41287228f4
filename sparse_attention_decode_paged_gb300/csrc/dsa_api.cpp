// C-ABI of libdsa.so: argument checks, the host row builder, workspace
// layout and kernel dispatch.  The declarations and the contract of every
// entry point are in include/dsa.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <initializer_list>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "dsa_internal.h"

namespace {

// Longest row (keys) a config may ask for.  Rows up to 8 x 32K keys are
// selected in one cluster's shared memory; longer ones by the streaming
// top-k, whose passes read the score buffer.
constexpr int32_t kMaxScoreWidth = 1 << 22;

thread_local std::string g_last_error;

dsa_status_t fail(dsa_status_t st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dsa_status_t ok() {
  g_last_error.clear();
  return DSA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

bool is_one_of(int v, std::initializer_list<int> set) {
  for (int x : set)
    if (v == x) return true;
  return false;
}

#define DSA_CHECK_CFG(cfg)                                  \
  do {                                                      \
    const dsa_status_t st_ = dsa_validate_config(cfg);      \
    if (st_ != DSA_OK) return st_;                          \
  } while (0)

#define DSA_CHECK_DEV_PTR(p)                                                          \
  do {                                                                                \
    if ((p) == nullptr) return fail(DSA_ERR_INVALID_ARG, "%s is NULL", #p);           \
    if (!aligned16(p)) return fail(DSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

dsa_status_t cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return ok();
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Rows per score window (commit message 3): all rows without a budget, else
// as many whole score rows as the budget holds.  The config is validated.
int32_t window_rows_of(const dsa_config_t *c) {
  if (c->score_buffer_bytes == 0) return c->max_rows;
  const long long fit = c->score_buffer_bytes / (static_cast<long long>(c->score_width) * 4);
  return static_cast<int32_t>(std::min<long long>(fit, c->max_rows));
}

dsa_status_t layout_of(const dsa_config_t *c, dsa_workspace_layout_t *l) {
  const size_t R = static_cast<size_t>(c->max_rows);
  const size_t HS = static_cast<size_t>(c->num_q_heads) * c->num_splits;
  size_t off = 0;
  l->status = off;
  off += 256;
  l->scores = off;
  off = align256(off + static_cast<size_t>(window_rows_of(c)) * c->score_width * sizeof(float));
  l->topk_idx = off;
  off = align256(off + R * c->topk * sizeof(int32_t));
  l->part_m = off;
  off = align256(off + R * HS * sizeof(float));
  l->part_l = off;
  off = align256(off + R * HS * sizeof(float));
  l->part_acc = off;
  off = align256(off + R * HS * c->head_dim * sizeof(float));
  l->group = off;
  if (dsa::group_path_enabled(*c)) {  // grouped flags, union counts, positions, masks
    const size_t nslots = (R + dsa::kGroupRows - 1) / dsa::kGroupRows;
    const size_t umax = static_cast<size_t>(dsa::group_union_capacity(*c));
    off = align256(off + R * sizeof(int32_t));
    off = align256(off + nslots * sizeof(int32_t));
    off = align256(off + nslots * (umax / 128) * sizeof(int32_t));
    off = align256(off + nslots * umax * sizeof(uint16_t));
  }
  l->key_hist = off;
  off = align256(off + R * 4096 * sizeof(uint32_t));
  l->total = off;
  return DSA_OK;
}

uint32_t *status_word(void *workspace) { return static_cast<uint32_t *>(workspace); }

// Pointers into the prefill-group scratch of a workspace (the config uses
// the group path).
dsa::GroupParams group_params(const dsa_config_t *c, void *workspace) {
  dsa_workspace_layout_t l;
  layout_of(c, &l);
  char *g = static_cast<char *>(workspace) + l.group;
  const size_t R = static_cast<size_t>(c->max_rows);
  dsa::GroupParams gp;
  gp.nslots = static_cast<int32_t>((R + dsa::kGroupRows - 1) / dsa::kGroupRows);
  gp.umax = dsa::group_union_capacity(*c);
  size_t off = 0;
  gp.grouped = reinterpret_cast<int32_t *>(g + off);
  off = align256(off + R * sizeof(int32_t));
  gp.ntiles = reinterpret_cast<int32_t *>(g + off);
  off = align256(off + gp.nslots * sizeof(int32_t));
  gp.tiles = reinterpret_cast<int32_t *>(g + off);
  off = align256(off + static_cast<size_t>(gp.nslots) * (gp.umax / 128) * sizeof(int32_t));
  gp.umask = reinterpret_cast<uint32_t *>(g + off);
  return gp;
}

}  // namespace

namespace dsa {
dsa_status_t set_error(dsa_status_t st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}
}  // namespace dsa

extern "C" {

dsa_status_t dsa_validate_config(const dsa_config_t *c) {
  if (c == nullptr) return fail(DSA_ERR_INVALID_ARG, "config is NULL");
  if (c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->num_q_heads % c->num_kv_heads != 0)
    return fail(DSA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                c->num_q_heads, c->num_kv_heads);
  if (c->num_q_heads / c->num_kv_heads > 8)
    return fail(DSA_ERR_UNSUPPORTED, "more than 8 query heads per KV head (%d)",
                c->num_q_heads / c->num_kv_heads);
  if (c->num_kv_heads > 8) return fail(DSA_ERR_UNSUPPORTED, "num_kv_heads %d > 8", c->num_kv_heads);
  if (!is_one_of(c->head_dim, {64, 128}))
    return fail(DSA_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", c->head_dim);
  if (c->idx_heads < 1 || c->idx_heads > 64)
    return fail(DSA_ERR_UNSUPPORTED, "idx_heads %d not in [1, 64]", c->idx_heads);
  if (!is_one_of(c->idx_dim, {32, 64, 128}))
    return fail(DSA_ERR_UNSUPPORTED, "idx_dim %d not in {32, 64, 128}", c->idx_dim);
  if (!is_one_of(c->page_size, {16, 32, 64, 128}))
    return fail(DSA_ERR_UNSUPPORTED, "page_size %d not in {16, 32, 64, 128}", c->page_size);
  if (c->block_rows < 1 || c->block_rows > 4)
    return fail(DSA_ERR_UNSUPPORTED, "block_rows %d not in [1, 4]", c->block_rows);
  if (c->max_rows < 1 || c->max_reqs < 1 || c->max_pages_per_req < 1 || c->num_pages < 1)
    return fail(DSA_ERR_INVALID_ARG, "max_rows, max_reqs, max_pages_per_req and num_pages must be >= 1");
  if (c->score_width < 1 || static_cast<long long>(c->score_width) >
                                static_cast<long long>(c->max_pages_per_req) * c->page_size)
    return fail(DSA_ERR_INVALID_ARG, "score_width %d must be in [1, max_pages_per_req * page_size]",
                c->score_width);
  if (c->score_width > kMaxScoreWidth)
    return fail(DSA_ERR_UNSUPPORTED, "score_width %d > %d", c->score_width, kMaxScoreWidth);
  if (c->topk < 1 || c->topk > c->score_width)
    return fail(DSA_ERR_INVALID_ARG, "topk %d must be in [1, score_width]", c->topk);
  if (c->num_splits < 1 || c->num_splits > 64)
    return fail(DSA_ERR_UNSUPPORTED, "num_splits %d not in [1, 64]", c->num_splits);
  if (c->idx_key_dtype != DSA_KEY_BF16 && c->idx_key_dtype != DSA_KEY_FP8_E4M3)
    return fail(DSA_ERR_INVALID_ARG, "idx_key_dtype %d unknown", c->idx_key_dtype);
  if (!(c->sm_scale > 0.f) || !std::isfinite(c->sm_scale))
    return fail(DSA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
  if ((c->flags & ~static_cast<int32_t>(DSA_FLAG_TOPK_HISTOGRAM | DSA_FLAG_KV_INTERLEAVED |
                                        DSA_FLAG_TEST_WAIT_TIMEOUT | DSA_FLAG_NO_PREFILL_GROUPS)) != 0)
    return fail(DSA_ERR_INVALID_ARG, "unknown flags 0x%x", c->flags);
  if (static_cast<long long>(c->max_reqs) * c->max_pages_per_req > 0x7FFFFFFFLL)
    return fail(DSA_ERR_INVALID_ARG, "page table larger than 2^31 entries");
  if (c->max_rows > 4096) return fail(DSA_ERR_UNSUPPORTED, "max_rows %d > 4096", c->max_rows);
  if (c->score_buffer_bytes < 0 ||
      (c->score_buffer_bytes > 0 && c->score_buffer_bytes < static_cast<long long>(c->score_width) * 4))
    return fail(DSA_ERR_INVALID_ARG, "score_buffer_bytes %lld must be 0 or hold one score row (%lld bytes)",
                static_cast<long long>(c->score_buffer_bytes), static_cast<long long>(c->score_width) * 4);
  return ok();
}

dsa_status_t dsa_score_windows(const dsa_config_t *cfg, int32_t *window_rows, int32_t *num_windows) {
  DSA_CHECK_CFG(cfg);
  if (window_rows == nullptr || num_windows == nullptr) return fail(DSA_ERR_INVALID_ARG, "output is NULL");
  const int32_t wr = window_rows_of(cfg);
  *window_rows = wr;
  *num_windows = (cfg->max_rows + wr - 1) / wr;
  return ok();
}

dsa_status_t dsa_workspace_layout(const dsa_config_t *cfg, dsa_workspace_layout_t *layout) {
  DSA_CHECK_CFG(cfg);
  if (layout == nullptr) return fail(DSA_ERR_INVALID_ARG, "layout is NULL");
  layout_of(cfg, layout);
  return ok();
}

dsa_status_t dsa_workspace_size(const dsa_config_t *cfg, size_t *bytes) {
  DSA_CHECK_CFG(cfg);
  if (bytes == nullptr) return fail(DSA_ERR_INVALID_ARG, "bytes is NULL");
  dsa_workspace_layout_t l;
  layout_of(cfg, &l);
  *bytes = l.total;
  return ok();
}

dsa_status_t dsa_suggest_num_splits(const dsa_config_t *cfg, int32_t num_sms, int32_t *num_splits) {
  DSA_CHECK_CFG(cfg);
  if (num_splits == nullptr) return fail(DSA_ERR_INVALID_ARG, "num_splits is NULL");
  if (num_sms <= 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e, "SM count");
    num_sms = sms;
  }
  const long long C = 2LL * num_sms, R = cfg->max_rows;
  const long long cap = std::min<long long>(64, std::max(1, cfg->topk / 32));
  const long long s4 = (4 * C + R / 2) / R;
  const long long s1 = std::max<long long>(1, C / R);
  long long S = s4 <= cap ? std::max<long long>(1, s4) : std::min(cap, s1);
  if (dsa::group_path_enabled(*cfg)) {
    // prefill row groups run one program per (slot, KV head, split) on one
    // CTA per SM: about 8 programs per CTA when half the slots form groups
    const long long slots = (R + dsa::kGroupRows - 1) / dsa::kGroupRows;
    const long long sg = (16LL * num_sms) / (slots * cfg->num_kv_heads);
    S = std::max(S, std::min(cap, std::max<long long>(1, sg)));
  }
  *num_splits = static_cast<int32_t>(S);
  return ok();
}

dsa_status_t dsa_reset_device_status(void *workspace, dsa_stream_t stream) {
  DSA_CHECK_DEV_PTR(workspace);
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), stream), "reset status");
}

dsa_status_t dsa_read_device_status(const void *workspace, uint32_t *status, dsa_stream_t stream) {
  DSA_CHECK_DEV_PTR(workspace);
  if (status == nullptr) return fail(DSA_ERR_INVALID_ARG, "status is NULL");
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_status(e, "read status");
  *status = v;
  if (v != 0) return fail(DSA_ERR_DEVICE_BOUNDS, "device status word 0x%x", v);
  return ok();
}

dsa_status_t dsa_build_rows(const dsa_config_t *cfg, int32_t num_reqs, const int32_t *req_cache_len,
                            const int32_t *req_new_tokens, int32_t *row_req, int32_t *row_len,
                            int32_t *row_pos, int32_t *block_first, int32_t *block_nrows,
                            int32_t *num_rows, int32_t *num_blocks) {
  DSA_CHECK_CFG(cfg);
  if (num_reqs < 0) return fail(DSA_ERR_INVALID_ARG, "num_reqs %d < 0", num_reqs);
  if (num_reqs > cfg->max_reqs)
    return fail(DSA_ERR_CAPACITY, "num_reqs %d > max_reqs %d", num_reqs, cfg->max_reqs);
  if (num_reqs > 0 && (req_cache_len == nullptr || req_new_tokens == nullptr))
    return fail(DSA_ERR_INVALID_ARG, "request arrays are NULL");
  if (!row_req || !row_len || !row_pos || !block_first || !block_nrows || !num_rows || !num_blocks)
    return fail(DSA_ERR_INVALID_ARG, "an output array is NULL");
  const long long max_len = std::min<long long>(
      cfg->score_width, static_cast<long long>(cfg->max_pages_per_req) * cfg->page_size);
  long long total = 0;
  for (int32_t b = 0; b < num_reqs; ++b) {
    const int32_t c = req_cache_len[b], n = req_new_tokens[b];
    if (n < 0 || c < n)
      return fail(DSA_ERR_INVALID_ARG, "request %d: new tokens %d, cache length %d", b, n, c);
    if (c > max_len)
      return fail(DSA_ERR_CAPACITY, "request %d: cache length %d > %lld", b, c, max_len);
    total += n;
  }
  if (total > cfg->max_rows)
    return fail(DSA_ERR_CAPACITY, "%lld rows > max_rows %d", total, cfg->max_rows);

  const int32_t R = cfg->max_rows;
  for (int32_t i = 0; i < R; ++i) {
    row_req[i] = 0;
    row_len[i] = 0;
    row_pos[i] = 0;
    block_first[i] = 0;
    block_nrows[i] = 0;
  }
  int32_t r = 0, nb = 0;
  for (int32_t b = 0; b < num_reqs; ++b) {
    const int32_t c = req_cache_len[b], n = req_new_tokens[b];
    const int32_t start = r;
    for (int32_t j = 0; j < n; ++j, ++r) {
      row_req[r] = b;
      row_pos[r] = c - n + j;
      row_len[r] = c - n + j + 1;
    }
    for (int32_t j = 0; j < n; j += cfg->block_rows) {
      block_first[nb] = start + j;
      block_nrows[nb] = std::min(cfg->block_rows, n - j);
      ++nb;
    }
  }
  *num_rows = r;
  *num_blocks = nb;
  return ok();
}

}  // extern "C"

namespace {
uint32_t *key_hist_of(const dsa_config_t *cfg, void *workspace) {
  dsa_workspace_layout_t l;
  layout_of(cfg, &l);
  return reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + l.key_hist);
}

dsa_status_t check_window(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end) {
  if (row_begin < 0 || row_end > cfg->max_rows || row_begin >= row_end)
    return fail(DSA_ERR_INVALID_ARG, "row window [%d, %d) not inside [0, %d)", row_begin, row_end,
                cfg->max_rows);
  return DSA_OK;
}

dsa_status_t indexer_impl(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end,
                          const void *q_idx, const float *w,
                          const void *idx_cache, const float *idx_scale, const int32_t *page_table,
                          const int32_t *row_req, const int32_t *row_len, const int32_t *block_first,
                          const int32_t *block_nrows, float *scores, void *workspace, bool hist,
                          dsa_stream_t stream) {
  DSA_CHECK_CFG(cfg);
  if (check_window(cfg, row_begin, row_end) != DSA_OK) return DSA_ERR_INVALID_ARG;
  DSA_CHECK_DEV_PTR(q_idx);
  DSA_CHECK_DEV_PTR(w);
  DSA_CHECK_DEV_PTR(idx_cache);
  DSA_CHECK_DEV_PTR(page_table);
  DSA_CHECK_DEV_PTR(row_req);
  DSA_CHECK_DEV_PTR(row_len);
  DSA_CHECK_DEV_PTR(block_first);
  DSA_CHECK_DEV_PTR(block_nrows);
  DSA_CHECK_DEV_PTR(scores);
  DSA_CHECK_DEV_PTR(workspace);
  if (cfg->idx_key_dtype == DSA_KEY_FP8_E4M3) DSA_CHECK_DEV_PTR(idx_scale);
  dsa::IndexerParams p;
  p.q_idx = static_cast<const uint8_t *>(q_idx);
  p.w = w;
  p.idx_cache = static_cast<const uint8_t *>(idx_cache);
  p.idx_scale = cfg->idx_key_dtype == DSA_KEY_FP8_E4M3 ? idx_scale : nullptr;
  p.page_table = page_table;
  p.row_req = row_req;
  p.row_len = row_len;
  p.block_first = block_first;
  p.block_nrows = block_nrows;
  p.scores = scores;
  p.status = status_word(workspace);
  p.idx_heads = cfg->idx_heads;
  p.idx_dim = cfg->idx_dim;
  p.max_rows = cfg->max_rows;
  p.max_reqs = cfg->max_reqs;
  p.max_pages_per_req = cfg->max_pages_per_req;
  p.score_width = cfg->score_width;
  p.num_pages = cfg->num_pages;
  p.page_size = cfg->page_size;
  p.block_rows = cfg->block_rows;
  p.row_hist = hist ? key_hist_of(cfg, workspace) : nullptr;
  p.row_lo = row_begin;
  p.row_hi = row_end;
  p.test_timeout = (cfg->flags & DSA_FLAG_TEST_WAIT_TIMEOUT) != 0 ? 1 : 0;
  return cuda_status(dsa::launch_indexer_tc(*cfg, p, stream), "indexer launch");
}

dsa_status_t topk_impl(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end, const float *scores,
                       const int32_t *row_len, int32_t *topk_idx, void *workspace, bool hist,
                       dsa_stream_t stream) {
  DSA_CHECK_CFG(cfg);
  if (check_window(cfg, row_begin, row_end) != DSA_OK) return DSA_ERR_INVALID_ARG;
  DSA_CHECK_DEV_PTR(scores);
  DSA_CHECK_DEV_PTR(row_len);
  DSA_CHECK_DEV_PTR(topk_idx);
  DSA_CHECK_DEV_PTR(workspace);
  dsa::TopkParams p;
  p.scores = scores;
  p.row_len = row_len;
  p.topk_idx = topk_idx;
  p.status = status_word(workspace);
  p.row_hist = hist ? key_hist_of(cfg, workspace) : nullptr;
  p.topk = cfg->topk;
  p.score_width = cfg->score_width;
  p.row_lo = row_begin;
  return cuda_status(dsa::launch_topk(*cfg, p, row_end - row_begin, stream), "top-k launch");
}
}  // namespace

namespace {
dsa_status_t merge_impl(const dsa_config_t *cfg, const float *part_m, const float *part_l, const float *part_acc,
                        void *out, float *lse, const int32_t *row_len, dsa_stream_t stream) {
  DSA_CHECK_CFG(cfg);
  DSA_CHECK_DEV_PTR(part_m);
  DSA_CHECK_DEV_PTR(part_l);
  DSA_CHECK_DEV_PTR(part_acc);
  DSA_CHECK_DEV_PTR(out);
  if (lse != nullptr && !aligned16(lse)) return fail(DSA_ERR_INVALID_ARG, "lse is not 16-byte aligned");
  dsa::MergeParams p;
  p.part_m = part_m;
  p.part_l = part_l;
  p.part_acc = part_acc;
  p.out = static_cast<uint8_t *>(out);
  p.lse = lse;
  p.row_len = row_len;
  p.max_rows = cfg->max_rows;
  p.num_q_heads = cfg->num_q_heads;
  p.num_splits = cfg->num_splits;
  return cuda_status(dsa::launch_merge(*cfg, p, stream), "merge launch");
}
}  // namespace

extern "C" {

dsa_status_t dsa_indexer_scores(const dsa_config_t *cfg, const void *q_idx, const float *w,
                                const void *idx_cache, const float *idx_scale,
                                const int32_t *page_table, const int32_t *row_req,
                                const int32_t *row_len, const int32_t *block_first,
                                const int32_t *block_nrows, float *scores, void *workspace,
                                dsa_stream_t stream) {
  const bool hist = cfg != nullptr && (cfg->flags & DSA_FLAG_TOPK_HISTOGRAM) != 0;
  return indexer_impl(cfg, 0, cfg != nullptr ? cfg->max_rows : 0, q_idx, w, idx_cache, idx_scale, page_table,
                      row_req, row_len, block_first, block_nrows, scores, workspace, hist, stream);
}

dsa_status_t dsa_indexer_scores_window(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end,
                                       const void *q_idx, const float *w, const void *idx_cache,
                                       const float *idx_scale, const int32_t *page_table,
                                       const int32_t *row_req, const int32_t *row_len,
                                       const int32_t *block_first, const int32_t *block_nrows,
                                       float *scores, void *workspace, dsa_stream_t stream) {
  const bool hist = cfg != nullptr && (cfg->flags & DSA_FLAG_TOPK_HISTOGRAM) != 0;
  return indexer_impl(cfg, row_begin, row_end, q_idx, w, idx_cache, idx_scale, page_table, row_req, row_len,
                      block_first, block_nrows, scores, workspace, hist, stream);
}

dsa_status_t dsa_topk(const dsa_config_t *cfg, const float *scores, const int32_t *row_len,
                      int32_t *topk_idx, void *workspace, dsa_stream_t stream) {
  const bool hist = cfg != nullptr && (cfg->flags & DSA_FLAG_TOPK_HISTOGRAM) != 0;
  return topk_impl(cfg, 0, cfg != nullptr ? cfg->max_rows : 0, scores, row_len, topk_idx, workspace, hist,
                   stream);
}

dsa_status_t dsa_topk_window(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end,
                             const float *scores, const int32_t *row_len, int32_t *topk_idx,
                             void *workspace, dsa_stream_t stream) {
  const bool hist = cfg != nullptr && (cfg->flags & DSA_FLAG_TOPK_HISTOGRAM) != 0;
  return topk_impl(cfg, row_begin, row_end, scores, row_len, topk_idx, workspace, hist, stream);
}

}  // extern "C"

namespace {
// The attention calls; inside dsa_step (skip_empty_rows) the rows of length
// 0 get no split partials, since the step's merge writes their outputs
// without reading them.
dsa_status_t attn_impl(const dsa_config_t *cfg, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *page_table, const int32_t *row_req, const int32_t *row_len,
                       const int32_t *topk_idx, float *part_m, float *part_l, float *part_acc, void *workspace,
                       bool skip_empty_rows, dsa_stream_t stream) {
  DSA_CHECK_CFG(cfg);
  DSA_CHECK_DEV_PTR(q);
  DSA_CHECK_DEV_PTR(k_cache);
  DSA_CHECK_DEV_PTR(v_cache);
  DSA_CHECK_DEV_PTR(page_table);
  DSA_CHECK_DEV_PTR(row_req);
  DSA_CHECK_DEV_PTR(row_len);
  DSA_CHECK_DEV_PTR(topk_idx);
  DSA_CHECK_DEV_PTR(part_m);
  DSA_CHECK_DEV_PTR(part_l);
  const bool kv_interleaved = (cfg->flags & DSA_FLAG_KV_INTERLEAVED) != 0;
  if (kv_interleaved &&
      static_cast<const char *>(v_cache) !=
          static_cast<const char *>(k_cache) + static_cast<size_t>(cfg->num_kv_heads) * cfg->head_dim * 2)
    return fail(DSA_ERR_INVALID_ARG, "DSA_FLAG_KV_INTERLEAVED: v_cache must be k_cache + num_kv_heads*head_dim*2 bytes");
  DSA_CHECK_DEV_PTR(part_acc);
  DSA_CHECK_DEV_PTR(workspace);
  dsa::AttnParams p;
  p.q = static_cast<const uint8_t *>(q);
  p.k_cache = static_cast<const uint8_t *>(k_cache);
  p.v_cache = static_cast<const uint8_t *>(v_cache);
  p.page_table = page_table;
  p.row_req = row_req;
  p.row_len = row_len;
  p.topk_idx = topk_idx;
  p.part_m = part_m;
  p.part_l = part_l;
  p.part_acc = part_acc;
  p.status = status_word(workspace);
  p.num_q_heads = cfg->num_q_heads;
  p.num_kv_heads = cfg->num_kv_heads;
  p.topk = cfg->topk;
  p.num_splits = cfg->num_splits;
  p.max_rows_attn = cfg->max_rows;
  p.max_reqs = cfg->max_reqs;
  p.max_pages_per_req = cfg->max_pages_per_req;
  p.score_width = cfg->score_width;
  p.num_pages = cfg->num_pages;
  p.page_size = cfg->page_size;
  p.sm_scale_log2 = cfg->sm_scale * 1.4426950408889634f;
  p.kv_interleaved = kv_interleaved ? 1 : 0;
  p.page_shift = 0;
  while ((1 << p.page_shift) < cfg->page_size) ++p.page_shift;  // page_size is a validated power of two
  p.grouped = nullptr;
  p.skip_empty_rows = skip_empty_rows ? 1 : 0;
  if (dsa::group_path_enabled(*cfg)) {
    // prefill row groups: the union, the other rows (the decode kernel leaves
    // the grouped rows alone), then the groups' tensor-core attention, whose
    // split partials — most of the step's — are then the last written before
    // the merge reads them
    const dsa::GroupParams gp = group_params(cfg, workspace);
    p.grouped = gp.grouped;
    cudaError_t e = dsa::launch_group_union(*cfg, p, gp, stream);
    if (e == cudaSuccess) e = dsa::launch_sparse_attn(*cfg, p, stream);
    if (e == cudaSuccess) e = dsa::launch_group_attn(*cfg, p, gp, stream);
    return cuda_status(e, "prefill-group attention launch");
  }
  return cuda_status(dsa::launch_sparse_attn(*cfg, p, stream), "sparse attention launch");
}
}  // namespace

extern "C" {

dsa_status_t dsa_sparse_attn(const dsa_config_t *cfg, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *page_table,
                             const int32_t *row_req, const int32_t *row_len,
                             const int32_t *topk_idx, float *part_m, float *part_l,
                             float *part_acc, void *workspace, dsa_stream_t stream) {
  return attn_impl(cfg, q, k_cache, v_cache, page_table, row_req, row_len, topk_idx, part_m, part_l, part_acc,
                   workspace, false, stream);
}


dsa_status_t dsa_merge(const dsa_config_t *cfg, const float *part_m, const float *part_l,
                       const float *part_acc, void *out, float *lse, dsa_stream_t stream) {
  return merge_impl(cfg, part_m, part_l, part_acc, out, lse, nullptr, stream);
}

dsa_status_t dsa_step(const dsa_config_t *cfg, const dsa_step_args_t *a, void *workspace,
                      dsa_stream_t stream) {
  DSA_CHECK_CFG(cfg);
  if (a == nullptr) return fail(DSA_ERR_INVALID_ARG, "args is NULL");
  DSA_CHECK_DEV_PTR(workspace);
  dsa_workspace_layout_t l;
  layout_of(cfg, &l);
  char *ws = static_cast<char *>(workspace);
  float *scores = reinterpret_cast<float *>(ws + l.scores);
  int32_t *topk_idx = reinterpret_cast<int32_t *>(ws + l.topk_idx);
  float *part_m = reinterpret_cast<float *>(ws + l.part_m);
  float *part_l = reinterpret_cast<float *>(ws + l.part_l);
  float *part_acc = reinterpret_cast<float *>(ws + l.part_acc);
  // per row window (one window without a score budget): the indexer counts
  // the first-level key histogram the top-k then uses; the next window's
  // indexer is an ordinary launch, so it starts once this top-k is done
  // reading the shared score buffer
  const int32_t wr = window_rows_of(cfg);
  dsa_status_t st = DSA_OK;
  for (int32_t lo = 0; lo < cfg->max_rows; lo += wr) {
    const int32_t hi = std::min(lo + wr, cfg->max_rows);
    st = indexer_impl(cfg, lo, hi, a->q_idx, a->w, a->idx_cache, a->idx_scale, a->page_table, a->row_req,
                      a->row_len, a->block_first, a->block_nrows, scores, workspace, true, stream);
    if (st != DSA_OK) return st;
    st = topk_impl(cfg, lo, hi, scores, a->row_len, topk_idx, workspace, true, stream);
    if (st != DSA_OK) return st;
  }
  st = attn_impl(cfg, a->q, a->k_cache, a->v_cache, a->page_table, a->row_req, a->row_len, topk_idx, part_m,
                 part_l, part_acc, workspace, true, stream);
  if (st != DSA_OK) return st;
  // the step knows its rows: pad rows are written empty without their partials
  return merge_impl(cfg, part_m, part_l, part_acc, a->out, a->lse, a->row_len, stream);
}

const char *dsa_last_error(void) { return g_last_error.c_str(); }

const char *dsa_version(void) { return "dsa-gb300 0.3 (sm_103a)"; }

}  // extern "C"
