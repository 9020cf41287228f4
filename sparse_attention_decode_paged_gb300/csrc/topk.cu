// Length-aware exact top-k per row: radix select on order-preserving keys,
// one thread-block cluster per row.
//
// Megatron-LM PR #7211, commit message 1: the selection reads each row only
// up to its length; commit message 10: a position inside the length outranks
// every padded position, even at score -inf.  Ranking: higher score first,
// equal scores to the lower position, NaN below every number.
//
// Each fp32 score maps to a 32-bit key whose unsigned order is the ranking
// (NaN -> 0, -0 -> +0).  A row is split across a cluster of C CTAs (1024
// threads each, C = ceil(W / 16K) up to 8), each holding its contiguous
// segment of the row as keys in shared memory; the CTAs exchange histograms,
// candidates and counts through distributed shared memory:
//  A. each CTA loads its segment with 16-byte loads and histograms the top
//     12 key bits; the cluster sums the histograms and every CTA finds the
//     bin of the k-th key and how many keys rank above it (in the fused step
//     the indexer has already counted the row's bins in the workspace, so
//     the CTAs read that histogram instead, and zero it for the next step);
//  B. each CTA counts, per warp, its keys above that bin and copies out the
//     keys inside it (the candidates, with their positions);
//  C. every CTA runs the same two 10-bit radix passes over the cluster's
//     candidates and obtains the k-th key tau and how many keys equal to tau
//     still fit ("need"); heavy ties (more than 4096 candidates) instead run
//     the two passes over the whole row;
//  D. per-CTA and per-warp prefix counts place every key > tau and the first
//     `need` keys == tau in ascending position order.
// Integer work only, so the result is bit-exact and deterministic.
#include <cooperative_groups.h>

#include "dsa_common.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = kKeyBins;  // key bits 31..20
constexpr int kBins2 = 1024;  // key bits 19..10, then 9..0
constexpr int kCandMax = 4096;
constexpr int kMaxCluster = 8;
constexpr int kSegPerCta = 16384;  // target keys per CTA
constexpr int kSegMax = 32768;     // shared-memory capacity per CTA

struct TopkShared {
  uint32_t hist[kBins1];      // this CTA's histogram (read by the whole cluster)
  uint32_t hist_tot[kBins1];  // the cluster's histogram
  uint32_t cand_key[kCandMax];
  int32_t cand_pos[kCandMax];  // local position in this CTA's segment
  uint32_t scan[kWarps];
  uint32_t warp_gt[kWarps], warp_eq[kWarps];
  uint32_t cta_gt, cta_eq;  // this CTA's totals (read by later ranks)
  uint32_t digit, above, count;
};

// Finds, scanning bins from the top, the bin d with above(d) < need <=
// above(d) + hist[d]; writes d and above(d) to sh.digit / sh.above, or nbins
// and 0 when the histogram holds fewer than `need` keys.
__device__ __forceinline__ void select_bin(TopkShared &sh, const uint32_t *hist, int nbins, uint32_t need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins / kThreads;  // 1 or 4 bins per thread, descending
  uint32_t c[4] = {0u, 0u, 0u, 0u}, tot = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < per) {
      c[j] = hist[nbins - 1 - tid * per - j];
      tot += c[j];
    }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sh.scan[warp] = incl;
  if (tid == 0) {  // no bin: the histogram holds fewer than `need` keys
    sh.digit = static_cast<uint32_t>(nbins);
    sh.above = 0u;
  }
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

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) topk_cluster_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkShared &sh = *reinterpret_cast<TopkShared *>(smem_raw);
  uint32_t *keys_s = reinterpret_cast<uint32_t *>(smem_raw + ((sizeof(TopkShared) + 15) & ~size_t(15)));
  cg::cluster_group cl = cg::this_cluster();
  pdl_launch_dependents();
  pdl_wait();  // the scores come from the indexer kernel
  const int C = static_cast<int>(cl.num_blocks());
  const int q = static_cast<int>(cl.block_rank());
  const int r = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.topk;
  int32_t *out = p.topk_idx + static_cast<size_t>(r) * K;
  int L = p.row_len[r];
  if (L < 0 || L > p.score_width) {
    if (tid == 0 && q == 0) flag_status(p.status, DSA_DEV_BAD_ROW);
    L = 0;
  }
  uint32_t *ghist = p.row_hist != nullptr ? p.row_hist + static_cast<size_t>(r) * kBins1 : nullptr;
  if (L <= K) {  // every position is selected (same branch in every CTA of the cluster)
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;  // ready for the next step
    const int per = (K + C - 1) / C;
    for (int i = q * per + tid; i < min(K, (q + 1) * per); i += kThreads) out[i] = i < L ? i : -1;
    return;
  }
  // this CTA's segment [lo, lo + n) of the row, a multiple of 128 long
  const int seg = (((L + C - 1) / C) + 127) & ~127;
  const int lo = min(L, q * seg);
  const int n = min(L, lo + seg) - lo;
  const float *srow = p.scores + static_cast<size_t>(r) * p.score_width + lo;

  for (int i = tid; i < kBins1; i += kThreads) sh.hist[i] = 0u;
  if (tid < kWarps) {
    sh.warp_gt[tid] = 0u;
    sh.warp_eq[tid] = 0u;
  }
  if (tid == 0) sh.count = 0u;
  __syncthreads();

  // ---- A. load the segment and histogram the top 12 bits
  const bool vec = (p.score_width & 3) == 0;
  const int n4 = vec ? (n >> 2) : 0;
  for (int base = 0; base < n4; base += kThreads * 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = base + u * kThreads + tid;
      v[u] = i4 < n4 ? __ldg(reinterpret_cast<const float4 *>(srow) + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = base + u * kThreads + tid;
      if (i4 < n4) {
        const uint4 k = make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
        reinterpret_cast<uint4 *>(keys_s)[i4] = k;
        if (ghist == nullptr) {
          atomicAdd(&sh.hist[k.x >> 20], 1u);
          atomicAdd(&sh.hist[k.y >> 20], 1u);
          atomicAdd(&sh.hist[k.z >> 20], 1u);
          atomicAdd(&sh.hist[k.w >> 20], 1u);
        }
      }
    }
  }
  for (int i = n4 * 4 + tid; i < n; i += kThreads) {
    const uint32_t k = order_key(srow[i]);
    keys_s[i] = k;
    if (ghist == nullptr) atomicAdd(&sh.hist[k >> 20], 1u);
  }
  // pad the segment to whole 128-key chunks with key 0 (NaN's key): unless the
  // k-th key lies in bin 0, a 0 is never above, at or inside the threshold bin,
  // so the hot loops below need no per-key bounds check
  const int n_pad = (n + 127) & ~127;
  for (int i = n + tid; i < n_pad; i += kThreads) keys_s[i] = 0u;
  __syncthreads();
  bool recount = ghist == nullptr;
  if (!recount) {
    // the indexer already counted the row's key bins; use them only if they
    // count exactly the row's L scores (every CTA of the cluster reads the
    // same counts, so all take the same branch)
    uint32_t part = 0u;
    for (int b = tid; b < kBins1; b += kThreads) {
      const uint32_t v = __ldcg(ghist + b);
      sh.hist_tot[b] = v;
      part += v;
    }
    part = warp_sum(part);
    if (lane == 0) sh.scan[warp] = part;
    __syncthreads();
    uint32_t total = 0u;
#pragma unroll 8
    for (int w = 0; w < kWarps; ++w) total += sh.scan[w];
    if (total != static_cast<uint32_t>(L)) {
      recount = true;
      for (int i = tid; i < n; i += kThreads) atomicAdd(&sh.hist[keys_s[i] >> 20], 1u);
    }
  }
  if (recount) {
    __syncthreads();
    cl.sync();
    for (int b = tid; b < kBins1; b += kThreads) {
      uint32_t s = 0u;
      for (int rr = 0; rr < C; ++rr) s += cl.map_shared_rank(sh.hist, rr)[b];
      sh.hist_tot[b] = s;
    }
  }
  __syncthreads();
  uint32_t need = static_cast<uint32_t>(K);
  select_bin(sh, sh.hist_tot, kBins1, need);
  const uint32_t d1 = min(sh.digit, static_cast<uint32_t>(kBins1 - 1));  // found whenever L > K
  need -= sh.above;
  const uint32_t in_bin = sh.hist_tot[d1];
  uint32_t prefix = d1 << 20, mask = 0xFFF00000u;

  // warp w owns the contiguous 128-key chunks [c_beg, c_end) of the segment
  const int nchunks = n_pad / 128;
  const int per = (nchunks + kWarps - 1) / kWarps;
  const int c_beg = warp * per, c_end = min(nchunks, c_beg + per);
  const bool checked = d1 == 0;  // the NaN bin is in play: check bounds per key

  if (in_bin <= static_cast<uint32_t>(kCandMax)) {
    // ---- B. per-warp count above the bin, candidates inside it
    uint32_t gtw = 0u;
    for (int c = c_beg; c < c_end; ++c) {
      const int i0 = c * 128 + lane * 4;
      const uint4 kk = reinterpret_cast<const uint4 *>(keys_s)[i0 >> 2];
      const uint32_t ks[4] = {kk.x, kk.y, kk.z, kk.w};
      uint32_t hits = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool valid = !checked || i0 + j < n;
        const uint32_t top = ks[j] >> 20;
        gtw += (valid && top > d1) ? 1u : 0u;
        hits |= (valid && top == d1) ? (1u << j) : 0u;
      }
      const uint32_t nh = __popc(hits);
      uint32_t incl = nh;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
      uint32_t base = 0u;
      if (lane == 0 && tot) base = atomicAdd(&sh.count, tot);
      base = __shfl_sync(0xFFFFFFFFu, base, 0) + incl - nh;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (hits & (1u << j)) {
          if (base < static_cast<uint32_t>(kCandMax)) {  // holds whenever the histogram is exact
            sh.cand_key[base] = ks[j];
            sh.cand_pos[base] = i0 + j;
          }
          ++base;
        }
    }
    gtw = warp_sum(gtw);
    if (lane == 0) sh.warp_gt[warp] = gtw;
    __syncthreads();
    cl.sync();  // every CTA's candidates are complete (and the row histogram was read)
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;  // ready for the next step
    if (tid == 0 && sh.count > static_cast<uint32_t>(kCandMax)) {
      flag_status(p.status, DSA_DEV_BAD_ROW);  // histogram and scores disagree
      sh.count = kCandMax;
    }
    // ---- C. the same radix select over the cluster's candidates, in every CTA
    uint32_t cluster_cands = 0u;
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      for (int i = tid; i < kBins2; i += kThreads) sh.hist_tot[i] = 0u;
      __syncthreads();
      cluster_cands = 0u;
      for (int rr = 0; rr < C; ++rr) {
        const uint32_t *ck = cl.map_shared_rank(sh.cand_key, rr);
        const uint32_t cnt = min(*cl.map_shared_rank(&sh.count, rr), static_cast<uint32_t>(kCandMax));
        cluster_cands += cnt;
        for (uint32_t i = tid; i < cnt; i += kThreads) {
          const uint32_t k = ck[i];
          if ((k & mask) == prefix) atomicAdd(&sh.hist_tot[(k >> shift) & 0x3FFu], 1u);
        }
      }
      __syncthreads();
      select_bin(sh, sh.hist_tot, kBins2, need);
      const uint32_t dg = min(sh.digit, static_cast<uint32_t>(kBins2 - 1));  // found if the counts agree
      need -= sh.above;
      prefix |= dg << shift;
      mask |= 0x3FFu << shift;
    }
    // the candidates the cluster found must be the keys the histogram put in
    // the k-th key's bin
    if (tid == 0 && q == 0 && cluster_cands != in_bin) flag_status(p.status, DSA_DEV_BAD_HIST);
    // own candidates above / at the k-th key, credited to the warp that owns them
    const uint32_t thr = prefix;
    const uint32_t cnt = sh.count;
    for (uint32_t i = tid; i < cnt; i += kThreads) {
      const uint32_t k = sh.cand_key[i];
      const int w = (sh.cand_pos[i] / 128) / max(per, 1);
      if (k > thr) atomicAdd(&sh.warp_gt[w], 1u);
      else if (k == thr) atomicAdd(&sh.warp_eq[w], 1u);
    }
  } else {
    // heavy ties: two more 10-bit passes over the whole row
    if (ghist != nullptr) {
      cl.sync();  // every CTA has read the row histogram
      if (q == 0)
        for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;
    }
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      cl.sync();  // nobody still reads this CTA's previous histogram
      for (int i = tid; i < kBins2; i += kThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t k = keys_s[i];
        if ((k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 0x3FFu], 1u);
      }
      __syncthreads();
      cl.sync();
      for (int b = tid; b < kBins2; b += kThreads) {
        uint32_t s = 0u;
        for (int rr = 0; rr < C; ++rr) s += cl.map_shared_rank(sh.hist, rr)[b];
        sh.hist_tot[b] = s;
      }
      __syncthreads();
      select_bin(sh, sh.hist_tot, kBins2, need);
      const uint32_t dg = min(sh.digit, static_cast<uint32_t>(kBins2 - 1));  // found if the counts agree
      if (tid == 0 && q == 0 && sh.digit >= static_cast<uint32_t>(kBins2)) flag_status(p.status, DSA_DEV_BAD_HIST);
      need -= sh.above;
      prefix |= dg << shift;
      mask |= 0x3FFu << shift;
    }
    const uint32_t thr = prefix;
    uint32_t gtw = 0u, eqw = 0u;
    for (int c = c_beg; c < c_end; ++c) {
      const int i0 = c * 128 + lane * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool valid = i0 + j < n;
        const uint32_t k = valid ? keys_s[i0 + j] : 0u;
        gtw += (valid && k > thr) ? 1u : 0u;
        eqw += (valid && k == thr) ? 1u : 0u;
      }
    }
    gtw = warp_sum(gtw);
    eqw = warp_sum(eqw);
    if (lane == 0) {
      sh.warp_gt[warp] = gtw;
      sh.warp_eq[warp] = eqw;
    }
  }
  const uint32_t thr = prefix;
  __syncthreads();
  if (tid == 0) {
    uint32_t g = 0u, e = 0u;
    for (int w = 0; w < kWarps; ++w) {
      g += sh.warp_gt[w];
      e += sh.warp_eq[w];
    }
    sh.cta_gt = g;
    sh.cta_eq = e;
  }
  __syncthreads();
  cl.sync();  // every CTA's totals are visible

  // ---- D. ordered write
  uint32_t g_before = 0u, e_before = 0u;
  for (int rr = 0; rr < q; ++rr) {
    g_before += *cl.map_shared_rank(&sh.cta_gt, rr);
    e_before += *cl.map_shared_rank(&sh.cta_eq, rr);
  }
  for (int w = 0; w < warp; ++w) {
    g_before += sh.warp_gt[w];
    e_before += sh.warp_eq[w];
  }
  for (int c = c_beg; c < c_end; ++c) {
    const int i0 = c * 128 + lane * 4;
    const uint4 kk = reinterpret_cast<const uint4 *>(keys_s)[i0 >> 2];
    const uint32_t ks[4] = {kk.x, kk.y, kk.z, kk.w};
    uint32_t ng = 0u, ne = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = !checked || i0 + j < n;
      ng += (valid && ks[j] > thr) ? 1u : 0u;
      ne += (valid && ks[j] == thr) ? 1u : 0u;
    }
    const uint32_t packed = (ng << 16) | ne;
    uint32_t incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - packed;
    uint32_t g = g_before + (excl >> 16), e = e_before + (excl & 0xFFFFu);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const bool valid = !checked || i0 + j < n;
      const int t = lo + i0 + j;
      if (valid && ks[j] > thr) {
        const uint32_t pos = g + min(e, need);
        if (pos < static_cast<uint32_t>(K)) out[pos] = t;
        ++g;
      } else if (valid && ks[j] == thr) {
        if (e < need && g + e < static_cast<uint32_t>(K)) out[g + e] = t;
        ++e;
      }
    }
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    g_before += tot >> 16;
    e_before += tot & 0xFFFFu;
  }
  cl.sync();  // keep this CTA's shared memory alive until the cluster is done with it
}

}  // namespace

int topk_cluster_size(int score_width) {
  int c = (score_width + kSegPerCta - 1) / kSegPerCta;
  return c < 1 ? 1 : (c > kMaxCluster ? kMaxCluster : c);
}

cudaError_t launch_topk(const dsa_config_t &cfg, const TopkParams &p, cudaStream_t st) {
  const int C = topk_cluster_size(cfg.score_width);
  const int seg_w = (((cfg.score_width + C - 1) / C) + 127) & ~127;
  if (seg_w > kSegMax) return cudaErrorInvalidValue;
  const size_t smem = ((sizeof(TopkShared) + 15) & ~size_t(15)) + static_cast<size_t>(seg_w) * 4;
  cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(topk_cluster_kernel, dim3(static_cast<unsigned>(cfg.max_rows * C)), dim3(kThreads), smem, st,
                 static_cast<unsigned>(C), p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
