// Length-aware exact top-k per row: radix select on order-preserving keys.
//
// Megatron-LM PR #7211, commit message 1: the selection reads each row only
// up to its length; commit message 10: a position inside the length outranks
// every padded position, even at score -inf.  Ranking: higher score first,
// equal scores to the lower position, NaN below every number.
//
// One CTA (1024 threads) per row.  Each fp32 score maps to a 32-bit key whose
// unsigned order is the ranking (NaN -> 0, -0 -> +0).
//  1. Load the row with wide loads (16 bytes, all loads of a thread in
//     flight together), caching the keys in shared memory when the row fits
//     (<= 48K), and histogram the top 12 key bits.
//  2. Scan the 4096 bins from the top: the bin holding the k-th best key and
//     how many keys rank above it.
//  3. If that bin holds <= 4096 keys, copy them out (warp-aggregated) and
//     finish the select on the candidates alone with two 10-bit passes;
//     otherwise (heavy ties) run the two 10-bit passes over the whole row.
//  4. Knowing the k-th key tau and how many keys equal to tau still fit
//     ("need"), a warp-ordered compaction (ballots + popc) writes every
//     position with key > tau and the first `need` positions with key == tau,
//     in ascending position order.
// Integer work only, so the result is bit-exact and deterministic.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmemMaxKeys = 48 * 1024;
constexpr int kBins1 = 4096;   // key bits 31..20
constexpr int kBins2 = 1024;   // key bits 19..10, then 9..0
constexpr int kCandMax = 4096;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: below every number
  if (b == 0x80000000u) b = 0u;                     // -0 ties with +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkShared {
  uint32_t hist[kBins1];
  uint32_t cand[kCandMax];
  uint32_t scan[kWarps];
  uint32_t warp_cnt[2][kWarps];
  uint32_t digit, above, count;
};

// Finds, scanning bins from the top, the bin d with above(d) < need <=
// above(d) + hist[d]; writes d and above(d) to sh.digit / sh.above.
__device__ __forceinline__ void select_bin(TopkShared &sh, int nbins, uint32_t need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins / kThreads;  // 1 or 4 bins per thread, descending
  uint32_t c[4] = {0u, 0u, 0u, 0u}, tot = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < per) {
      c[j] = sh.hist[nbins - 1 - tid * per - j];
      tot += c[j];
    }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sh.scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t v = sh.scan[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, v, o);
      if (lane >= o) v += u;
    }
    sh.scan[lane] = v;
  }
  __syncthreads();
  const uint32_t excl = incl - tot + (warp > 0 ? sh.scan[warp - 1] : 0u);
  if (excl < need && need <= excl + tot) {
    uint32_t above = excl;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j < per) {
        if (need <= above + c[j]) {
          sh.digit = static_cast<uint32_t>(nbins - 1 - tid * per - j);
          sh.above = above;
          break;
        }
        above += c[j];
      }
    }
  }
  __syncthreads();
}

template <bool CACHE>
__global__ void __launch_bounds__(kThreads, 1) topk_radix_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint32_t keys_s[];
  __shared__ TopkShared sh;
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
  auto key_at = [&](int t) -> uint32_t {
    if constexpr (CACHE) return keys_s[t];
    else return order_key(__ldg(srow + t));
  };

  for (int i = tid; i < kBins1; i += kThreads) sh.hist[i] = 0u;
  if (tid == 0) sh.count = 0u;
  __syncthreads();

  // ---- 1. load (+ cache) and histogram of the top 12 bits
  const bool vec = (p.score_width & 3) == 0;
  const int L4 = vec ? (L >> 2) : 0;
  for (int base = 0; base < L4; base += kThreads * 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = base + u * kThreads + tid;
      v[u] = i4 < L4 ? __ldg(reinterpret_cast<const float4 *>(srow) + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = base + u * kThreads + tid;
      if (i4 < L4) {
        const uint32_t k0 = order_key(v[u].x), k1 = order_key(v[u].y);
        const uint32_t k2 = order_key(v[u].z), k3 = order_key(v[u].w);
        if constexpr (CACHE) {
          reinterpret_cast<uint4 *>(keys_s)[i4] = make_uint4(k0, k1, k2, k3);
        }
        atomicAdd(&sh.hist[k0 >> 20], 1u);
        atomicAdd(&sh.hist[k1 >> 20], 1u);
        atomicAdd(&sh.hist[k2 >> 20], 1u);
        atomicAdd(&sh.hist[k3 >> 20], 1u);
      }
    }
  }
  for (int t = L4 * 4 + tid; t < L; t += kThreads) {
    const uint32_t k = order_key(srow[t]);
    if constexpr (CACHE) keys_s[t] = k;
    atomicAdd(&sh.hist[k >> 20], 1u);
  }
  __syncthreads();

  // ---- 2. the bin of the k-th key
  uint32_t need = static_cast<uint32_t>(K);
  select_bin(sh, kBins1, need);
  uint32_t prefix = sh.digit << 20, mask = 0xFFF00000u;
  need -= sh.above;
  const uint32_t in_bin = sh.hist[sh.digit];
  __syncthreads();

  // ---- 3. finish the select on the candidates (or on the whole row)
  if (in_bin <= static_cast<uint32_t>(kCandMax)) {
    for (int base = 0; base < L; base += kThreads) {
      const int t = base + tid;
      const uint32_t k = t < L ? key_at(t) : 0u;
      const bool hit = t < L && (k & mask) == prefix;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, hit);
      uint32_t slot0 = 0u;
      if (lane == 0 && m) slot0 = atomicAdd(&sh.count, static_cast<uint32_t>(__popc(m)));
      slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
      if (hit) sh.cand[slot0 + __popc(m & ((1u << lane) - 1u))] = k;
    }
    __syncthreads();
    const int nc = static_cast<int>(sh.count);
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      for (int i = tid; i < kBins2; i += kThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < nc; i += kThreads) {
        const uint32_t k = sh.cand[i];
        if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 0x3FFu], 1u);
      }
      __syncthreads();
      select_bin(sh, kBins2, need);
      need -= sh.above;
      prefix |= sh.digit << shift;
      mask |= 0x3FFu << shift;
      __syncthreads();
    }
  } else {
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      for (int i = tid; i < kBins2; i += kThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (int t = tid; t < L; t += kThreads) {
        const uint32_t k = key_at(t);
        if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 0x3FFu], 1u);
      }
      __syncthreads();
      select_bin(sh, kBins2, need);
      need -= sh.above;
      prefix |= sh.digit << shift;
      mask |= 0x3FFu << shift;
      __syncthreads();
    }
  }
  const uint32_t thr = prefix;

  // ---- 4. ordered compaction: warp w scans a contiguous run of 32-wide chunks
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
    sh.warp_cnt[0][warp] = gt;
    sh.warp_cnt[1][warp] = eq;
  }
  __syncthreads();
  uint32_t gt_before = 0u, eq_before = 0u;
  for (int w2 = 0; w2 < warp; ++w2) {
    gt_before += sh.warp_cnt[0][w2];
    eq_before += sh.warp_cnt[1][w2];
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
