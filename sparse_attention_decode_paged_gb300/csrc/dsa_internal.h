// Internal interface between the C-ABI layer (dsa_api.cpp) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

struct IndexerParams {
  const uint8_t *q_idx;     // bf16 [R, H_I, D_I]
  const float *w;           // [R, H_I]
  const uint8_t *idx_cache; // bf16 / e4m3 [NP, P, D_I]
  const float *idx_scale;   // [NP, P] or null
  const int32_t *page_table;
  const int32_t *row_req;
  const int32_t *row_len;
  const int32_t *block_first;
  const int32_t *block_nrows;
  float *scores;            // [row_hi - row_lo, W]: row r at (r - row_lo) * W
  uint32_t *status;
  uint32_t *row_hist;       // [R, 4096] key-bin counts for the top-k, or null
  int32_t idx_heads, idx_dim, max_rows, max_reqs, max_pages_per_req, score_width, num_pages;
  int32_t page_size, block_rows;
  int32_t row_lo, row_hi;   // the row window scored (0, max_rows for all rows)
  int32_t test_timeout;     // DSA_FLAG_TEST_WAIT_TIMEOUT: one wait that nothing completes
};

struct TopkParams {
  const float *scores;     // [rows of the window, W]
  const int32_t *row_len;
  int32_t *topk_idx;
  uint32_t *status;
  uint32_t *row_hist;  // [R, 4096] filled by the indexer (used, then zeroed), or null
  int32_t topk, score_width;
  int32_t row_lo;          // first row of the window; one cluster per row of it
};

struct AttnParams {
  const uint8_t *q;        // bf16 [R, Hq, D]
  const uint8_t *k_cache;  // bf16 [NP, P, Hkv, D], or [NP, P, 2, Hkv, D] with V interleaved
  const uint8_t *v_cache;  // k_cache + Hkv * D * 2 when interleaved
  const int32_t *page_table;
  const int32_t *row_req;
  const int32_t *row_len;
  const int32_t *topk_idx; // [R, K]
  float *part_m;           // [R, Hq, S]
  float *part_l;
  float *part_acc;         // [R, Hq, S, D]
  uint32_t *status;
  int32_t num_q_heads, num_kv_heads, topk, num_splits;
  int32_t max_rows_attn, max_reqs, max_pages_per_req, score_width, num_pages, page_size;
  float sm_scale_log2;     // sm_scale * log2(e)
  int32_t kv_interleaved;  // 1: one copy moves a token's K and V rows
  int32_t page_shift;      // log2(page_size)
  const int32_t *grouped;  // [R] 1: the row is attended by the prefill-group kernel (null: no groups)
  int32_t skip_empty_rows; // 1: rows of length 0 get no partials (the step's merge never reads them)
};

// Prefill row groups: the rows of one request in a slot of kGroupRows
// consecutive rows (at least kGroupMin of them) attend to the union of their
// selections on the tensor cores (group_attn.cu).
constexpr int kGroupRows = 16;
constexpr int kGroupMin = 8;

struct GroupParams {
  int32_t *grouped;  // [R] 1: the row is a group member
  int32_t *ntiles;   // [nslots] 128-position tiles holding a selected position (0: the slot is no group)
  int32_t *tiles;    // [nslots, umax / 128] those tiles' indices, ascending
  uint32_t *umask;   // [nslots, umax / 128, 16, 4] per tile and slot row j: bit b of word w set if
                     // row j selected position 128 * tile + 32 * w + b
  int32_t umax, nslots;  // umax: positions a group may span (a multiple of 128)
};

struct MergeParams {
  const float *part_m, *part_l, *part_acc;
  uint8_t *out;  // bf16 [R, Hq, D]
  float *lse;    // [R, Hq] or null
  const int32_t *row_len;  // [R] or null: a row of length 0 is written empty without reading its partials
  int32_t max_rows, num_q_heads, num_splits;
};

// Launches `kernel` on `st` with programmatic stream serialization, so it may
// start while the previous kernel on the stream drains (the kernel itself
// waits with griddepcontrol.wait before reading that kernel's output).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  lc.attrs = attr;
  lc.numAttrs = n;
  return cudaLaunchKernelEx(&lc, kernel, args...);
}

// Records the thread's last-error text (see dsa_last_error) and returns st.
dsa_status_t set_error(dsa_status_t st, const char *fmt, ...);

// Each launcher returns the launch error (cudaSuccess when queued).
cudaError_t launch_indexer_tc(const dsa_config_t &cfg, const IndexerParams &p, cudaStream_t st);
cudaError_t launch_topk(const dsa_config_t &cfg, const TopkParams &p, int rows, cudaStream_t st);
cudaError_t launch_sparse_attn(const dsa_config_t &cfg, const AttnParams &p, cudaStream_t st);
cudaError_t launch_merge(const dsa_config_t &cfg, const MergeParams &p, cudaStream_t st);
// The prefill-group path: whether a config uses it, the union capacity per
// slot (positions, a multiple of 128), and its two kernels.
bool group_path_enabled(const dsa_config_t &cfg);
int32_t group_union_capacity(const dsa_config_t &cfg);
cudaError_t launch_group_union(const dsa_config_t &cfg, const AttnParams &p, const GroupParams &gp, cudaStream_t st);
cudaError_t launch_group_attn(const dsa_config_t &cfg, const AttnParams &p, const GroupParams &gp, cudaStream_t st);

}  // namespace dsa
