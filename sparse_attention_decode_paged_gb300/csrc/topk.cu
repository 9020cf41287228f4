// Length-aware exact top-k per row: radix select on order-preserving keys.
//
// Megatron-LM PR #7211, commit message 1: the selection reads each row only
// up to its length; commit message 10: a position inside the length outranks
// every padded position, even at score -inf.  Ranking: higher score first,
// equal scores to the lower position, NaN below every number.
//
// One CTA (1024 threads) per row.  Each fp32 score maps to a 32-bit key whose
// unsigned order is the ranking (NaN -> 0, -0 -> +0).  Four 8-bit radix passes
// find the key tau of the k-th best position and how many positions with key
// == tau still fit ("need"); a warp-ordered compaction then writes every
// position with key > tau and the first `need` positions with key == tau, in
// ascending position order.  Integer work only, so the result is bit-exact
// and deterministic.  Rows up to 48K wide are cached in shared memory as keys
// for the passes; wider rows re-read the score row (from L2).
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemMaxKeys = 48 * 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: below every number
  if (b == 0x80000000u) b = 0u;                     // -0 ties with +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

template <bool CACHE>
__global__ void __launch_bounds__(kThreads, 1) topk_radix_kernel(const TopkParams p) {
  extern __shared__ uint32_t keys_s[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_cnt[2][kWarps];
  __shared__ uint32_t sel_digit, sel_above;
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.topk;
  int32_t *out = p.topk_idx + static_cast<size_t>(r) * K;
  int L = p.row_len[r];
  if (L < 0 || L > p.score_width) {
    if (tid == 0) flag_status(p.status, DSA_DEV_BAD_ROW);
    L = 0;
  }
  if (L <= K) {  // every position is selected
    for (int i = tid; i < K; i += kThreads) out[i] = i < L ? i : -1;
    return;
  }
  const float *srow = p.scores + static_cast<size_t>(r) * p.score_width;
  if constexpr (CACHE) {
    for (int t = tid; t < L; t += kThreads) keys_s[t] = order_key(srow[t]);
    __syncthreads();
  }
  auto key_at = [&](int t) -> uint32_t {
    if constexpr (CACHE) return keys_s[t];
    else return order_key(__ldg(srow + t));
  };

  uint32_t prefix = 0u, mask = 0u, need = static_cast<uint32_t>(K);
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
    for (int t = tid; t < L; t += kThreads) {
      const uint32_t k = key_at(t);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane j owns bins 255-8j .. 248-8j, scanned from the top
      uint32_t c[8], tot = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        tot += c[i];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - tot;
      if (excl < need && need <= incl) {
        uint32_t above = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (need <= above + c[i]) {
            sel_digit = static_cast<uint32_t>(255 - 8 * lane - i);
            sel_above = above;
            break;
          }
          above += c[i];
        }
      }
    }
    __syncthreads();
    need -= sel_above;
    prefix |= sel_digit << shift;
    mask |= 0xFFu << shift;
  }
  const uint32_t thr = prefix;

  // ordered compaction: warp w scans a contiguous run of 32-wide chunks
  const int nchunks = (L + 31) / 32;
  const int per = (nchunks + kWarps - 1) / kWarps;
  const int c_beg = warp * per, c_end = min(nchunks, c_beg + per);
  uint32_t gt = 0u, eq = 0u;
  for (int c = c_beg; c < c_end; ++c) {
    const int t = c * 32 + lane;
    const bool valid = t < L;
    const uint32_t k = valid ? key_at(t) : 0u;
    gt += __popc(__ballot_sync(0xFFFFFFFFu, valid && k > thr));
    eq += __popc(__ballot_sync(0xFFFFFFFFu, valid && k == thr));
  }
  if (lane == 0) {
    warp_cnt[0][warp] = gt;
    warp_cnt[1][warp] = eq;
  }
  __syncthreads();
  uint32_t gt_before = 0u, eq_before = 0u;
  for (int w2 = 0; w2 < warp; ++w2) {
    gt_before += warp_cnt[0][w2];
    eq_before += warp_cnt[1][w2];
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int c = c_beg; c < c_end; ++c) {
    const int t = c * 32 + lane;
    const bool valid = t < L;
    const uint32_t k = valid ? key_at(t) : 0u;
    const bool is_gt = valid && k > thr, is_eq = valid && k == thr;
    const uint32_t mg = __ballot_sync(0xFFFFFFFFu, is_gt);
    const uint32_t me = __ballot_sync(0xFFFFFFFFu, is_eq);
    const uint32_t g_rank = gt_before + __popc(mg & lt_mask);
    const uint32_t e_rank = eq_before + __popc(me & lt_mask);
    if (is_gt) out[g_rank + min(e_rank, need)] = t;
    else if (is_eq && e_rank < need) out[g_rank + e_rank] = t;
    gt_before += __popc(mg);
    eq_before += __popc(me);
  }
}

}  // namespace

cudaError_t launch_topk(const dsa_config_t &cfg, const TopkParams &p, cudaStream_t st) {
  if (cfg.score_width <= kSmemMaxKeys) {
    const size_t smem = static_cast<size_t>(cfg.score_width) * 4;
    cudaError_t e = cudaFuncSetAttribute(topk_radix_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    topk_radix_kernel<true><<<cfg.max_rows, kThreads, smem, st>>>(p);
  } else {
    topk_radix_kernel<false><<<cfg.max_rows, kThreads, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace dsa
