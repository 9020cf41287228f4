/*
 * dsa.h -- C-ABI of libdsa.so: the per-step hot path of DeepSeek-style
 * sparse attention (DSA) over paged GQA caches, for decode, chunked prefill
 * and mixed steps, on one NVIDIA GB300 (sm_103a).
 *
 * Source: Megatron-LM PR #7211 (dynamic-inference DSA over GQA with paged
 * caches).  Its commit messages define the method; they are cited below as
 * "commit message N" in the order the PR page lists them:
 *   1  length-aware indexer over page-contiguous key tiles; sparse attention
 *      with all heads of a KV group together, top-k slots split across
 *      programs and merged flash-decoding style;
 *   2  every query token is a row (request, causal length); score blocks;
 *      static padded buffers, no host syncs, CUDA-graph capture;
 *   3  scores and selection in row windows under a score-buffer byte budget;
 *   6  exact chunk merging for long contexts;
 *   8  probabilities enter the value reduction in fp32;
 *  10  a position inside the row's length outranks padding even when its
 *      score is -inf.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - The caller owns every buffer.  No call allocates or frees memory.
 *  - "device" pointers are CUDA global-memory pointers on the current
 *    device and must be 16-byte aligned; "host" pointers are ordinary
 *    process memory.  A NULL or misaligned pointer is DSA_ERR_INVALID_ARG.
 *  - bf16 tensors are passed as raw 16-bit storage (const void*); fp8 index
 *    keys as raw OCP E4M3 bytes.  All tensors are dense, row-major, with the
 *    shapes given per argument.
 *  - The workspace (dsa_workspace_size bytes) must be zero-filled once after
 *    allocation; the calls keep the parts that must start at zero at zero.
 *  - Every launch size depends only on dsa_config_t.  Lengths, page tables,
 *    row maps and row counts are device data, so changing them between CUDA
 *    graph replays needs no re-capture (commit message 2).  The device calls
 *    never synchronize, never read device memory on the host and never
 *    allocate, so they may be captured into a CUDA graph once the library
 *    has been called once on the device outside capture.
 *  - Errors the host can see (bad config, NULL or misaligned pointers)
 *    return a status before anything is launched; the text of the last
 *    error is available from dsa_last_error().  Errors only the device can
 *    see (a page id outside the pool, a row longer than score_width, a
 *    selected position at or past the row's length...) set a bit in a
 *    sticky status word inside the workspace and the offending unit is
 *    skipped (its outputs are written as empty); the kernels never trap.
 *    Read the word with dsa_read_device_status().
 *  - Pad rows (row_len == 0) read nothing: their scores are not written,
 *    their top-k slots are -1, their partials are empty and their output is
 *    zero with lse = -inf.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *dsa_stream_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* bad pointer, size or config field          */
  DSA_ERR_UNSUPPORTED = 2,   /* valid shape this library has no kernel for */
  DSA_ERR_CAPACITY = 3,      /* inputs exceed the config's static capacity */
  DSA_ERR_CUDA = 4,          /* a CUDA runtime call failed                 */
  DSA_ERR_DEVICE_BOUNDS = 5  /* the device status word is non-zero         */
} dsa_status_t;

/* Bits of the device status word. */
enum {
  DSA_DEV_BAD_ROW = 1u << 0,   /* row_req >= max_reqs, row_len < 0 or > score_width */
  DSA_DEV_BAD_PAGE = 1u << 1,  /* page-table entry outside [0, num_pages)           */
  DSA_DEV_BAD_INDEX = 1u << 2, /* top-k position outside [0, row_len)               */
  DSA_DEV_BAD_BLOCK = 1u << 3, /* score block outside max_rows or mixing requests   */
  DSA_DEV_TIMEOUT = 1u << 4,   /* a bounded device-side wait ran out                */
  DSA_DEV_BAD_HIST = 1u << 5   /* a handed-over key histogram disagrees with scores */
};

typedef enum { DSA_KEY_BF16 = 0, DSA_KEY_FP8_E4M3 = 1 } dsa_key_dtype_t;

/*
 * Model shape and static capacity; fixed for the lifetime of a captured
 * graph.  Supported by this library:
 *   num_q_heads % num_kv_heads == 0, num_q_heads / num_kv_heads <= 8,
 *   num_kv_heads <= 8, head_dim in {64, 128}, max_rows <= 4096;
 *   1 <= idx_heads <= 64, idx_dim in {32, 64, 128};
 *   page_size in {16, 32, 64, 128}; 1 <= block_rows <= 4;
 *   1 <= topk <= score_width <= min(4194304, max_pages_per_req * page_size);
 *   1 <= num_splits <= 64; sm_scale > 0 and finite;
 *   score_buffer_bytes == 0 or >= score_width * 4 (one score row).
 */
typedef struct {
  int32_t num_q_heads;       /* Hq: attention query heads                        */
  int32_t num_kv_heads;      /* Hkv: KV heads; query head h reads KV head h/(Hq/Hkv) */
  int32_t head_dim;          /* D                                                 */
  int32_t idx_heads;         /* H_I: indexer heads                                */
  int32_t idx_dim;           /* D_I: indexer query / key dim (one key per token)   */
  int32_t page_size;         /* P: tokens per cache page                          */
  int32_t topk;              /* K: keys selected per row                          */
  int32_t num_splits;        /* S: top-k slot splits per row (flash decoding)      */
  int32_t max_rows;          /* R: static row slots (query tokens) per step        */
  int32_t max_reqs;          /* page-table rows                                   */
  int32_t max_pages_per_req; /* page-table row stride                              */
  int32_t score_width;       /* W: longest causal length; score row stride         */
  int32_t num_pages;         /* pool size of every cache                          */
  int32_t block_rows;        /* G: most rows in one score block                    */
  int32_t idx_key_dtype;     /* dsa_key_dtype_t                                    */
  float sm_scale;            /* softmax scale on q.k                              */
  int32_t flags;             /* DSA_FLAG_* bits, 0 for none                       */
  int64_t score_buffer_bytes;/* byte budget of dsa_step's score buffer: the step
                              * scores and selects its rows in windows of
                              * floor(budget / (score_width * 4)) rows (commit
                              * message 3); 0 = all max_rows rows at once   */
} dsa_config_t;

/* Bits of dsa_config_t.flags. */
enum {
  /* dsa_indexer_scores also counts, per row, the top 12 bits of each score's
   * order-preserving key into the workspace histogram, and dsa_topk uses
   * (then zeroes) those counts instead of recounting.  With this bit set,
   * every dsa_indexer_scores call must be followed by dsa_topk on the same
   * scores and workspace before the next dsa_indexer_scores call (for the
   * _window calls: the top-k of the same window before an indexer call
   * that covers any of its rows again).  dsa_step always works this way.  dsa_topk checks the hand-over: a row whose
   * histogram does not count exactly row_len scores (the indexer ran without
   * the bit, or twice) is recounted from its scores, with the same result; a
   * histogram with the right total that does not match the scores (the scores
   * changed in between) sets DSA_DEV_BAD_HIST and that row's selection is
   * unspecified.  No case reads or writes outside the buffers. */
  DSA_FLAG_TOPK_HISTOGRAM = 1 << 0,
  /* K and V of a token are adjacent in one cache: k_cache is
   * [num_pages, page_size, 2, num_kv_heads, head_dim] bf16 (the token's K row
   * for all KV heads, then its V row) and v_cache must equal
   * k_cache + num_kv_heads * head_dim * 2 bytes (else DSA_ERR_INVALID_ARG).
   * The sparse attention then moves each selected token with one copy
   * instead of two; results are identical to the separate layout.  A layout
   * of this library's own (the pages keep K and V apart). */
  DSA_FLAG_KV_INTERLEAVED = 1 << 1,
  /* Test only: exercises the bounded-wait failure path without a fault.  The
   * lightning indexer's MMA thread first waits on a barrier that nothing
   * completes, with a budget of about 1 ms instead of the usual ~1 s; the wait
   * runs out, the kernel sets DSA_DEV_TIMEOUT and its abort flag, every role
   * leaves its loop (the producer still waits for its copies in flight), the
   * launch returns and the scores are incomplete.  The next call without the
   * bit runs normally once the status word is reset.  Never set it outside a
   * test. */
  DSA_FLAG_TEST_WAIT_TIMEOUT = 1 << 2,
  /* Every row takes the per-row sparse attention (top-k slot splits): no
   * prefill row groups are formed (see dsa_sparse_attn), the workspace has no
   * group region, and dsa_suggest_num_splits leaves out the group term. */
  DSA_FLAG_NO_PREFILL_GROUPS = 1 << 3
};

/* Every pointer one fused step needs (all device pointers). */
typedef struct {
  const int32_t *page_table;  /* [max_reqs, max_pages_per_req] physical page ids   */
  const int32_t *row_req;     /* [max_rows] request of each row                    */
  const int32_t *row_len;     /* [max_rows] causal length of each row (0 = pad)    */
  const int32_t *block_first; /* [max_rows] first row of each score block          */
  const int32_t *block_nrows; /* [max_rows] rows in each block (0 = unused block)  */
  const void *q_idx;          /* bf16 [max_rows, idx_heads, idx_dim]               */
  const float *w;             /* fp32 [max_rows, idx_heads] indexer head weights   */
  const void *idx_cache;      /* bf16 or e4m3 [num_pages, page_size, idx_dim]      */
  const float *idx_scale;     /* fp32 [num_pages, page_size], NULL for bf16 keys   */
  const void *q;              /* bf16 [max_rows, num_q_heads, head_dim]            */
  const void *k_cache;        /* bf16 [num_pages, page_size, num_kv_heads, head_dim]
                               * ([num_pages, page_size, 2, ...] with
                               * DSA_FLAG_KV_INTERLEAVED)                          */
  const void *v_cache;        /* bf16, same shape as k_cache (k_cache + one K row
                               * with DSA_FLAG_KV_INTERLEAVED)                     */
  void *out;                  /* bf16 [max_rows, num_q_heads, head_dim] (output)   */
  float *lse;                 /* fp32 [max_rows, num_q_heads] (output), nullable   */
} dsa_step_args_t;

/* Byte offsets of the intermediates inside a step workspace. */
typedef struct {
  size_t status;    /* uint32 sticky device status word                   */
  size_t scores;    /* fp32 [window_rows, score_width] (dsa_score_windows) */
  size_t topk_idx;  /* int32 [max_rows, topk]                             */
  size_t part_m;    /* fp32 [max_rows, num_q_heads, num_splits]           */
  size_t part_l;    /* fp32 [max_rows, num_q_heads, num_splits]           */
  size_t part_acc;  /* fp32 [max_rows, num_q_heads, num_splits, head_dim] */
  size_t group;     /* prefill-group scratch (see dsa_sparse_attn); empty
                     * (= key_hist) when the config has no prefill groups  */
  size_t key_hist;  /* uint32 [max_rows, 4096]: score-key histograms (zero between steps) */
  size_t total;     /* bytes to allocate (256-byte aligned regions)       */
} dsa_workspace_layout_t;

/* Checks a config against the supported set above.  Host only. */
dsa_status_t dsa_validate_config(const dsa_config_t *cfg);

/* Size and layout of the workspace dsa_step needs.  Host only.
 * The individual kernel calls use its status word, and with
 * DSA_FLAG_TOPK_HISTOGRAM dsa_indexer_scores / dsa_topk its key histogram. */
dsa_status_t dsa_workspace_size(const dsa_config_t *cfg, size_t *bytes);
dsa_status_t dsa_workspace_layout(const dsa_config_t *cfg, dsa_workspace_layout_t *layout);

/*
 * dsa_score_windows -- the row windows dsa_step scores and selects in
 * (commit message 3: a score buffer under a byte budget; the window count
 * depends only on the padded rows and the width, so a captured graph
 * replays it).  Host only.
 * *window_rows = max_rows if score_buffer_bytes == 0, else
 * min(max_rows, floor(score_buffer_bytes / (score_width * 4)));
 * *num_windows = ceil(max_rows / *window_rows).  Window i covers rows
 * [i * window_rows, min((i + 1) * window_rows, max_rows)).
 */
dsa_status_t dsa_score_windows(const dsa_config_t *cfg, int32_t *window_rows, int32_t *num_windows);

/*
 * dsa_suggest_num_splits -- a num_splits for this config's row count and
 * top-k on a GPU with num_sms SMs (num_sms <= 0: the current device's).
 * Host only; no launch.  A tuning aid measured on GB300, not part of the
 * method: the sparse attention runs one program per (row, split) on two
 * resident CTAs per SM (C = 2 * num_sms).  It suggests
 *   cap = min(64, max(1, topk / 32))        (>= 32 selected keys per split)
 *   S4  = round(4 * C / max_rows)           (about four programs per CTA)
 *   S1  = max(1, floor(C / max_rows))       (one wave of programs)
 *   S   = S4 <= cap ? max(1, S4) : min(cap, S1)
 * and, when the config has prefill row groups (see dsa_sparse_attn), whose
 * programs are (16-row slot, KV head, split) on one CTA per SM,
 *   S   = max(S, min(cap, max(1, floor(16 * num_sms / (slots * num_kv_heads)))))
 * with slots = ceil(max_rows / 16) (about 8 programs per CTA when half the
 * slots form groups).
 * e.g. on 152 SMs: 64 rows, top-k 2048 -> 19; 8 rows, top-k 512 -> 16;
 * 16 rows -> 19; 1024 rows -> 1, or 4 with prefill groups and 8 KV heads.
 * Errors: DSA_ERR_INVALID_ARG (bad config, NULL), DSA_ERR_CUDA (num_sms <= 0
 * and no device to query).
 */
dsa_status_t dsa_suggest_num_splits(const dsa_config_t *cfg, int32_t num_sms, int32_t *num_splits);

/* Clears the device status word (an async 4-byte memset on `stream`).
 * Call once after allocating a workspace and after reading a failure. */
dsa_status_t dsa_reset_device_status(void *workspace, dsa_stream_t stream);

/* Copies the status word to *status (host) and synchronizes `stream`.
 * Not for use inside stream capture.  Returns DSA_ERR_DEVICE_BOUNDS if the
 * word is non-zero, DSA_OK otherwise. */
dsa_status_t dsa_read_device_status(const void *workspace, uint32_t *status,
                                    dsa_stream_t stream);

/*
 * dsa_build_rows -- rows and score blocks of one step (host only).
 * Commit message 2: every query token, decode or prefill, is a row
 * (request, causal length); a score block is a run of consecutive rows of
 * one request scored against shared key tiles.
 *
 * Request b has cache length req_cache_len[b] after this step's
 * req_new_tokens[b] tokens were appended (the caches already hold them).
 * Its j-th new token becomes a row with row_req = b, row_pos =
 * cache_len - new + j and row_len = row_pos + 1 (the prefix includes the
 * token itself).  Rows are packed request by request from slot 0; slots
 * from *num_rows to max_rows-1 are padding (req 0, len 0, pos 0).  Each
 * request's rows are cut into blocks of at most block_rows rows; unused
 * block slots have block_first = block_nrows = 0.
 *
 * In:  req_cache_len, req_new_tokens  host int32 [num_reqs]
 * Out: row_req, row_len, row_pos, block_first, block_nrows  host int32 [max_rows]
 *      *num_rows, *num_blocks
 * Errors: DSA_ERR_INVALID_ARG (NULL, negative counts, new > cache length),
 *         DSA_ERR_CAPACITY (num_reqs > max_reqs, rows > max_rows, a cache
 *         length > score_width or > max_pages_per_req * page_size).
 */
dsa_status_t dsa_build_rows(const dsa_config_t *cfg, int32_t num_reqs,
                            const int32_t *req_cache_len, const int32_t *req_new_tokens,
                            int32_t *row_req, int32_t *row_len, int32_t *row_pos,
                            int32_t *block_first, int32_t *block_nrows,
                            int32_t *num_rows, int32_t *num_blocks);

/*
 * dsa_indexer_scores -- lightning-indexer scores (commit message 1).
 *   scores[r, t] = s_t * sum_h w[r, h] * max(0, q_idx[r, h, :] . k_t)
 * for every row r and every t < row_len[r], where k_t is the index key of
 * the row's request at logical position t: idx_cache[page_table[req][t / P],
 * t % P, :], and s_t = idx_scale[same page, same slot] for fp8 keys (1 for
 * bf16).  Products are exact, sums are fp32.  Rows are processed per score
 * block (block_first / block_nrows): all rows of a block share each key
 * tile.  scores[r, t] for t >= row_len[r] is neither read nor written.
 * scores: device fp32 [max_rows, score_width].  workspace: status word, and
 * with DSA_FLAG_TOPK_HISTOGRAM the per-row key histogram it adds to.
 */
dsa_status_t dsa_indexer_scores(const dsa_config_t *cfg, const void *q_idx, const float *w,
                                const void *idx_cache, const float *idx_scale,
                                const int32_t *page_table, const int32_t *row_req,
                                const int32_t *row_len, const int32_t *block_first,
                                const int32_t *block_nrows, float *scores, void *workspace,
                                dsa_stream_t stream);

/*
 * dsa_indexer_scores_window -- dsa_indexer_scores for the rows in
 * [row_begin, row_end) only (commit message 3).  A score block that
 * straddles a window edge contributes its rows inside the window; the
 * block's validity is still checked over all its rows.  Row r's scores go
 * to scores[(r - row_begin) * score_width + t]: scores is device fp32
 * [row_end - row_begin, score_width].  Same arithmetic, so every row's
 * scores equal those of the whole-batch call.
 * 0 <= row_begin < row_end <= max_rows, else DSA_ERR_INVALID_ARG.
 */
dsa_status_t dsa_indexer_scores_window(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end,
                                       const void *q_idx, const float *w, const void *idx_cache,
                                       const float *idx_scale, const int32_t *page_table,
                                       const int32_t *row_req, const int32_t *row_len,
                                       const int32_t *block_first, const int32_t *block_nrows,
                                       float *scores, void *workspace, dsa_stream_t stream);

/*
 * dsa_topk -- length-aware exact top-k per row (commit messages 1, 10).
 * For each row, the positions of the topk largest scores[r, t] among
 * t < row_len[r]: higher score first, equal scores to the lower position,
 * NaN below every number (-inf included).  If topk >= row_len every
 * position is selected.  Output is ascending, padded with -1.
 * scores: device fp32 [max_rows, score_width]; topk_idx: device int32
 * [max_rows, topk].  Bit-exact and deterministic.  With
 * DSA_FLAG_TOPK_HISTOGRAM it starts from the workspace histogram the
 * indexer counted (checked against the row, see the flag) and zeroes it.
 * Rows of up to 262144 keys are selected inside one thread-block cluster's
 * shared memory; with a longer score_width every pass streams the row from
 * `scores` instead, keeping on chip only the keys of the k-th key's
 * first-level bin (commit message 4: past 64K keys, selection works on the
 * candidates of a threshold); the result is the same.
 */
dsa_status_t dsa_topk(const dsa_config_t *cfg, const float *scores, const int32_t *row_len,
                      int32_t *topk_idx, void *workspace, dsa_stream_t stream);

/*
 * dsa_topk_window -- dsa_topk for the rows in [row_begin, row_end) only
 * (commit message 3), reading the window's scores as
 * dsa_indexer_scores_window wrote them (scores: device fp32
 * [row_end - row_begin, score_width]).  topk_idx is the whole device int32
 * [max_rows, topk] array; only the window's rows are written.
 * 0 <= row_begin < row_end <= max_rows, else DSA_ERR_INVALID_ARG.
 */
dsa_status_t dsa_topk_window(const dsa_config_t *cfg, int32_t row_begin, int32_t row_end,
                             const float *scores, const int32_t *row_len, int32_t *topk_idx,
                             void *workspace, dsa_stream_t stream);

/*
 * dsa_sparse_attn -- sparse GQA attention over the selected keys, split
 * (commit messages 1, 8).  For row r, KV head g and split s, the query
 * heads of group g share the split's selected positions: with
 * n = min(topk, row_len[r]), split s covers top-k slots [s*n/S, (s+1)*n/S)
 * (integer division).  A slot holding -1 is skipped; a slot holding a
 * position outside [0, row_len) sets DSA_DEV_BAD_INDEX and is skipped.  Each
 * selected K and V row is read once for the whole group.  With
 * x = sm_scale * q[r,h] . K[t,g], the split's partial state is m = max x,
 * l = sum e^(x-m), acc = sum e^(x-m) V[t,g], probabilities in fp32.  An
 * empty split writes m = -inf, l = 0, acc = 0.  With DSA_FLAG_KV_INTERLEAVED
 * k_cache is the one interleaved cache and v_cache = k_cache + one K row.
 * part_m, part_l: device fp32 [max_rows, num_q_heads, num_splits];
 * part_acc: device fp32 [max_rows, num_q_heads, num_splits, head_dim].
 */
/*
 * Prefill row groups (commit message 5: a group of consecutive prefill
 * tokens attends to the union of the group's selected keys with a per-token
 * mask).  When block_rows > 1, num_q_heads == 8 * num_kv_heads and head_dim
 * == 128, each slot of 16 consecutive rows [16i, 16i + 16) whose most common
 * request has at least 8 rows there is considered: if their longest row is
 * at most min(score_width, 64 * topk) rounded up to 128 positions long and
 * the union of their selections fills at least a quarter of it, those rows
 * form a group and their attention runs on the tensor cores over the union,
 * each row masked to its own selection, computing the same partial state as
 * the per-row path: probabilities in fp32, carried into the value product as
 * two bf16 terms whose sum is the fp32 value to about 2^-17 relative, and m
 * the exact maximum.  For a group row, split s covers the positions in the tiles
 * [s*T/S, (s+1)*T/S) of the T tiles of 128 positions ([128i, 128i + 128))
 * that hold a position some group row selected, in ascending order; the
 * row's partial state for split s is over its own selected positions in
 * those tiles (an empty share gives the empty state).  Every other row
 * splits its top-k slots as above.  The union lives in the workspace's
 * `group` region.
 */
dsa_status_t dsa_sparse_attn(const dsa_config_t *cfg, const void *q, const void *k_cache,
                             const void *v_cache, const int32_t *page_table,
                             const int32_t *row_req, const int32_t *row_len,
                             const int32_t *topk_idx, float *part_m, float *part_l,
                             float *part_acc, void *workspace, dsa_stream_t stream);

/*
 * dsa_merge -- flash-decoding merge of the split partials (commit messages
 * 1, 6).  m* = max_s m_s, l* = sum_s l_s e^(m_s - m*),
 * out = sum_s acc_s e^(m_s - m*) / l* (rounded to bf16), lse = m* + ln l*.
 * Rows whose splits are all empty get out = 0 and lse = -inf.
 * out: device bf16 [max_rows, num_q_heads, head_dim]; lse: device fp32
 * [max_rows, num_q_heads] or NULL.
 */
dsa_status_t dsa_merge(const dsa_config_t *cfg, const float *part_m, const float *part_l,
                       const float *part_acc, void *out, float *lse, dsa_stream_t stream);

/*
 * dsa_step -- indexer -> top-k -> sparse attention -> merge on `stream`,
 * with the intermediates in `workspace` (see dsa_workspace_layout); the
 * indexer always hands its key histogram to the top-k (as with
 * DSA_FLAG_TOPK_HISTOGRAM).  With a score_buffer_bytes budget the indexer
 * and the top-k run once per row window (dsa_score_windows) on one score
 * buffer of window_rows rows, each window's indexer starting after the
 * previous window's top-k has finished; the results equal those of one
 * window.  Rows of length 0 (pad rows) get out = 0 and lse = -inf without
 * split partials: the step writes none for them (dsa_sparse_attn called on
 * its own writes empty ones, which dsa_merge reads).  The top-k, attention
 * and merge launch with programmatic dependent launch, so each one's start
 * overlaps its predecessor's tail.
 * The whole step is capturable into one CUDA graph: no host sync,
 * allocation or host read, static grids.
 */
dsa_status_t dsa_step(const dsa_config_t *cfg, const dsa_step_args_t *args, void *workspace,
                      dsa_stream_t stream);

/*
 * dsa_step_noalloc -- dsa_step for callers that cannot allocate device
 * memory: code running inside CUDA-graph stream capture (cudaMalloc cannot
 * be captured), runtimes whose device memory is owned by another allocator,
 * and C hosts without a device allocator.  The page has no counterpart for
 * this entry point; it exists for those callers.
 *
 * The step's intermediates (status word, scores, top-k, split partials,
 * prefill-group region, key histogram) go
 * to a 32 MiB array inside the library's device image instead of a caller
 * workspace; every GPU that loads the library holds those 32 MiB until the
 * process exits.  Configs whose dsa_workspace_size exceeds 32 MiB are
 * rejected with DSA_ERR_CAPACITY before anything is launched (a
 * score_buffer_bytes budget shrinks the score part of that size).  The call
 * itself allocates nothing: the first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current, so make
 * that first call outside stream capture.  All calls on a device share the
 * array and it keeps the last call's contents; the status word is cleared at
 * the start of every call, and a call whose config lays the array out
 * differently from the previous call's on that device first clears its key
 * histogram region (an async memset on `stream`).  Calls whose executions
 * overlap on the GPU (other streams, concurrent graph replays) race on the
 * array.
 *
 * args: as dsa_step.  status_out: device uint32 (nullable, 4-byte aligned);
 * when given, the step's device status word is copied there at the end of
 * the step, on `stream`.
 */
dsa_status_t dsa_step_noalloc(const dsa_config_t *cfg, const dsa_step_args_t *args,
                              uint32_t *status_out, dsa_stream_t stream);

/* Text of the last error on the calling thread ("" if none). */
const char *dsa_last_error(void);

/* Library version string.  0.2: dsa_config_t gained score_buffer_bytes
 * (its size changed; rebuild callers), and the _window calls,
 * dsa_score_windows and dsa_suggest_num_splits were added.  0.3:
 * dsa_workspace_layout_t gained `group` (its size changed), prefill row
 * groups attend on the tensor cores (DSA_FLAG_NO_PREFILL_GROUPS turns them
 * off), score_width may reach 4194304. */
const char *dsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
