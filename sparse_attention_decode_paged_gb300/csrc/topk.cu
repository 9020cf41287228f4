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
// threads each; a CTA holds at most 32K keys, so C >= ceil(W / 32K), up to
// 8; above that floor C = ceil(W / 16K) capped at 4, or the floor alone
// when the rows outnumber what the GPU holds at once), each holding its
// contiguous segment of the row as keys in shared memory.
// One launch covers one row window (commit message 3): all rows, or those
// of a score window, whose scores start at the window's first row.  Thread t of a CTA owns the
// 4-key groups t, t + 1024, t + 2048, ... of the segment, so every pass over
// the keys is a short fixed loop of 16-byte shared-memory reads, and a
// position-ordered result takes one block-wide scan (per-group counts packed
// in 8-bit fields), not one scan per chunk:
//  A. the segment is loaded with 16-byte loads while the row's first-level
//     histogram (top 12 key bits) is read: the indexer's counts when it made
//     them and they total the row length, else counted here and summed
//     across the cluster through distributed shared memory;
//  B. every CTA finds the bin of the k-th key and how many keys rank above
//     it, and copies out the keys inside that bin (the candidates);
//  C. each CTA gathers the cluster's candidates and runs two 10-bit radix
//     passes over them for the k-th key tau and how many keys equal to tau
//     still fit ("need"); heavy ties (more than 4096 candidates) run the two
//     passes over the whole row instead;
//  D. one pass counts each thread's keys above tau and equal to it per
//     group; the block scan of those counts and the cluster's per-CTA totals
//     give every key > tau and the first `need` keys == tau its rank in
//     ascending position order.
// Integer work only, so the result is bit-exact and deterministic.
#include <cooperative_groups.h>

#include <algorithm>

#include "dsa_common.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = kKeyBins;  // key bits 31..20
constexpr int kBins2 = 1024;      // key bits 19..10, then 9..0
constexpr int kCandMax = 4096;
constexpr int kMaxCluster = 8;
constexpr int kSegPerCta = 16384;                       // target keys per CTA
constexpr int kSegMax = 32768;                          // shared-memory capacity per CTA
constexpr int kGroupsMax = kSegMax / (4 * kThreads);    // 4-key groups per thread

struct TopkShared {
  uint32_t hist[kBins1];       // this CTA's histogram (read by the whole cluster)
  uint32_t hist_tot[kBins1];   // the row's histogram
  uint32_t cand[kCandMax];     // this CTA's candidates (read by the whole cluster)
  uint32_t all_cand[kCandMax];  // the cluster's candidates
  uint32_t wtot[kGroupsMax][kWarps];  // per group and warp: (keys > tau) << 16 | (keys == tau)
  uint32_t gbase[kGroupsMax];         // the same, per group: its total over the CTA's warps
  uint32_t scan[kWarps];
  uint32_t count;           // this CTA's candidates
  uint32_t cta_gt, cta_eq;  // this CTA's totals (read by later ranks)
  uint32_t digit, above;
};

// Finds, scanning bins from the top, the bin d with above(d) < need <=
// above(d) + hist[d]; writes d and above(d) to sh.digit / sh.above, or nbins
// and 0 when the histogram holds fewer than `need` keys.
template <class SH>
__device__ __forceinline__ void select_bin(SH &sh, const uint32_t *hist, int nbins, uint32_t need) {
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

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// One radix pass over `cnt` keys: histogram of bits [shift, shift+10) of the
// keys matching prefix/mask, then the bin of the need-th key.  Returns the
// bin (clamped; sh.digit == kBins2 flags a histogram that came up short).
template <class SH>
__device__ __forceinline__ uint32_t radix_pass(SH &sh, const uint32_t *keys, uint32_t cnt, int shift,
                                               uint32_t prefix, uint32_t mask, uint32_t &need) {
  const int tid = threadIdx.x;
  for (int i = tid; i < kBins2; i += kThreads) sh.hist_tot[i] = 0u;
  __syncthreads();
  for (uint32_t i = tid; i < cnt; i += kThreads) {
    const uint32_t k = keys[i];
    if ((k & mask) == prefix) atomicAdd(&sh.hist_tot[(k >> shift) & 0x3FFu], 1u);
  }
  __syncthreads();
  select_bin(sh, sh.hist_tot, kBins2, need);
  need -= sh.above;
  return min(sh.digit, static_cast<uint32_t>(kBins2 - 1));
}

// NG: 4-key groups per thread the launch provides for (a power of two >= the
// segment's groups), so the unrolled per-group loops hold only the groups a
// segment can have.
template <int NG>
__global__ void __launch_bounds__(kThreads, 1) topk_cluster_kernel(const TopkParams p) {
  constexpr int NW = (NG + 3) / 4;  // 32-bit words of 8-bit per-group fields
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkShared &sh = *reinterpret_cast<TopkShared *>(smem_raw);
  uint32_t *keys_s = reinterpret_cast<uint32_t *>(smem_raw + ((sizeof(TopkShared) + 15) & ~size_t(15)));
  const uint4 *keys4 = reinterpret_cast<const uint4 *>(keys_s);
  cg::cluster_group cl = cg::this_cluster();
  pdl_launch_dependents();
  const int C = static_cast<int>(cl.num_blocks());
  const int q = static_cast<int>(cl.block_rank());
  const int wr = blockIdx.x / C;  // row within the window
  const int r = p.row_lo + wr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.topk;
  int32_t *out = p.topk_idx + static_cast<size_t>(r) * K;
  int L = p.row_len[r];  // row metadata, not the indexer's output: read while it finishes
  pdl_wait();            // the scores come from the indexer kernel
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
  // this CTA's segment [lo, lo + n) of the row, a multiple of 128 long; its
  // keys are padded with key 0 (NaN's key) to ng whole groups per thread
  const int seg = (((L + C - 1) / C) + 127) & ~127;
  const int lo = min(L, q * seg);
  const int n = min(L, lo + seg) - lo;
  const int ng = (n + 4 * kThreads - 1) / (4 * kThreads);  // <= NG
  const float *srow = p.scores + static_cast<size_t>(wr) * p.score_width + lo;

  // ---- A. the row's histogram and this segment's keys
  uint32_t gh[kBins1 / kThreads];
  if (ghist != nullptr) {
#pragma unroll
    for (int j = 0; j < kBins1 / kThreads; ++j) gh[j] = __ldcg(ghist + j * kThreads + tid);
  }
  if ((p.score_width & 3) == 0) {
    const int n4 = n >> 2;
    float4 v[NG];
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      const int i4 = u * kThreads + tid;
      if (u < ng) v[u] = i4 < n4 ? __ldg(reinterpret_cast<const float4 *>(srow) + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      const int i4 = u * kThreads + tid;
      if (u < ng) {
        uint4 k = make_uint4(0u, 0u, 0u, 0u);
        if (i4 < n4) {
          k = make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
        } else if (i4 == n4) {  // the ragged end of the segment (n not a multiple of 4)
          if (4 * i4 + 0 < n) k.x = order_key(srow[4 * i4 + 0]);
          if (4 * i4 + 1 < n) k.y = order_key(srow[4 * i4 + 1]);
          if (4 * i4 + 2 < n) k.z = order_key(srow[4 * i4 + 2]);
        }
        reinterpret_cast<uint4 *>(keys_s)[i4] = k;
      }
    }
  } else {
    for (int i = tid; i < ng * 4 * kThreads; i += kThreads) keys_s[i] = i < n ? order_key(srow[i]) : 0u;
  }
  bool recount = ghist == nullptr;
  if (!recount) {
    // use the indexer's counts only if they total the row length (every CTA
    // of the cluster reads the same counts, so all take the same branch)
    uint32_t part = 0u;
#pragma unroll
    for (int j = 0; j < kBins1 / kThreads; ++j) {
      sh.hist_tot[j * kThreads + tid] = gh[j];
      part += gh[j];
    }
    part = warp_sum(part);
    if (lane == 0) sh.scan[warp] = part;
  }
  if (tid == 0) sh.count = 0u;  // the candidate count (phase B)
  __syncthreads();  // keys, row histogram, scan
  if (!recount) {
    uint32_t total = 0u;
#pragma unroll 8
    for (int w = 0; w < kWarps; ++w) total += sh.scan[w];
    recount = total != static_cast<uint32_t>(L);
  }
  if (recount) {
    for (int i = tid; i < kBins1; i += kThreads) sh.hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) atomicAdd(&sh.hist[keys_s[i] >> 20], 1u);
    __syncthreads();
    cl.sync();
    for (int b = tid; b < kBins1; b += kThreads) {
      uint32_t s = 0u;
      for (int rr = 0; rr < C; ++rr) s += cl.map_shared_rank(sh.hist, rr)[b];
      sh.hist_tot[b] = s;
    }
  }
  __syncthreads();  // every read of sh.scan above precedes the scan below

  // ---- B. the bin of the k-th key; candidates inside it
  uint32_t need = static_cast<uint32_t>(K);
  select_bin(sh, sh.hist_tot, kBins1, need);
  const uint32_t d1 = min(sh.digit, static_cast<uint32_t>(kBins1 - 1));  // found whenever L > K
  need -= sh.above;
  const uint32_t in_bin = sh.hist_tot[d1];
  uint32_t prefix = d1 << 20, mask = 0xFFF00000u;
  const bool checked = d1 == 0;  // the NaN bin is in play: the padding must not count

  if (in_bin <= static_cast<uint32_t>(kCandMax)) {
    uint32_t hits[NG];
    uint32_t nh = 0u;
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      hits[u] = 0u;
      if (u < ng) {
        const uint4 kk = keys4[u * kThreads + tid];
        const uint32_t ks[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool valid = !checked || (u * kThreads + tid) * 4 + j < n;
          if (valid && (ks[j] >> 20) == d1) hits[u] |= 1u << j;
        }
        nh += __popc(hits[u]);
      }
    }
    // offsets: a warp scan of the per-thread counts and one shared atomic
    // per warp (the candidates' order is irrelevant: only counts follow)
    const uint32_t incl = warp_incl_scan(nh, lane);
    uint32_t wbase = 0u;
    if (lane == 31 && incl != 0u) wbase = atomicAdd(&sh.count, incl);
    uint32_t base = __shfl_sync(0xFFFFFFFFu, wbase, 31) + incl - nh;
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      if (u < ng && hits[u]) {
        const uint4 kk = keys4[u * kThreads + tid];
        const uint32_t ks[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (hits[u] & (1u << j)) {
            if (base < static_cast<uint32_t>(kCandMax)) sh.cand[base] = ks[j];  // holds whenever the histogram is exact
            ++base;
          }
      }
    }
    __syncthreads();
    cl.sync();  // every CTA's candidates are complete (and the row histogram was read)
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;  // ready for the next step
    // ---- C. gather the cluster's candidates, then two radix passes over them
    uint32_t total = 0u;
    for (int rr = 0; rr < C; ++rr) {
      const uint32_t cnt = min(*cl.map_shared_rank(&sh.count, rr), static_cast<uint32_t>(kCandMax));
      const uint32_t *src = cl.map_shared_rank(sh.cand, rr);
      for (uint32_t i = tid; i < cnt && total + i < static_cast<uint32_t>(kCandMax); i += kThreads)
        sh.all_cand[total + i] = src[i];
      total += cnt;
    }
    if (tid == 0 && q == 0) {
      if (total > static_cast<uint32_t>(kCandMax)) flag_status(p.status, DSA_DEV_BAD_ROW);  // scores vs histogram
      // the candidates the cluster found must be the keys the histogram put in
      // the k-th key's bin
      if (total != in_bin) flag_status(p.status, DSA_DEV_BAD_HIST);
    }
    total = min(total, static_cast<uint32_t>(kCandMax));
    __syncthreads();
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      const uint32_t dg = radix_pass(sh, sh.all_cand, total, shift, prefix, mask, need);
      prefix |= dg << shift;
      mask |= 0x3FFu << shift;
    }
  } else {
    // heavy ties: two more 10-bit passes over the whole row
    cl.sync();  // every CTA has read the row histogram
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;
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
  }
  const uint32_t thr = prefix;  // tau

  // ---- D. ranks of the selected keys in position order
  // per group: this thread's (keys > tau) << 16 | (keys == tau), and the
  // exclusive prefix of those counts over the warp's lanes (8-bit fields:
  // a warp holds at most 128 keys of a group)
  uint32_t sel_gt[NW] = {}, sel_eq[NW] = {};
#pragma unroll
  for (int u = 0; u < NG; ++u) {
    if (u < ng) {
      const uint4 kk = keys4[u * kThreads + tid];
      const uint32_t ks[4] = {kk.x, kk.y, kk.z, kk.w};
      uint32_t g = 0u, e = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool valid = !checked || (u * kThreads + tid) * 4 + j < n;
        g += (valid && ks[j] > thr) ? 1u : 0u;
        e += (valid && ks[j] == thr) ? 1u : 0u;
      }
      sel_gt[u >> 2] |= g << (8 * (u & 3));
      sel_eq[u >> 2] |= e << (8 * (u & 3));
    }
  }
  uint32_t ex_gt[NW], ex_eq[NW];
#pragma unroll
  for (int w4 = 0; w4 < NW; ++w4) {
    if (w4 * 4 < ng) {
      const uint32_t ig = warp_incl_scan(sel_gt[w4], lane), ie = warp_incl_scan(sel_eq[w4], lane);
      ex_gt[w4] = ig - sel_gt[w4];
      ex_eq[w4] = ie - sel_eq[w4];
      if (lane == 31) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (w4 * 4 + j < ng)
            sh.wtot[w4 * 4 + j][warp] = (((ig >> (8 * j)) & 0xFFu) << 16) | ((ie >> (8 * j)) & 0xFFu);
      }
    }
  }
  __syncthreads();
  // warp u: exclusive prefix over the warps of group u, and the group's total
  if (warp < ng) {
    const uint32_t v = sh.wtot[warp][lane];
    const uint32_t iv = warp_incl_scan(v, lane);
    sh.wtot[warp][lane] = iv - v;
    if (lane == 31) sh.gbase[warp] = iv;  // the group's total for now
  }
  __syncthreads();
  if (tid == 0) {  // this CTA's totals, for the later ranks of the cluster
    uint32_t run = 0u;
    for (int u = 0; u < ng; ++u) run += sh.gbase[u];
    sh.cta_gt = run >> 16;
    sh.cta_eq = run & 0xFFFFu;
  }
  cl.sync();  // every CTA's totals are visible (and a barrier of this CTA)
  uint32_t g_cta = 0u, e_cta = 0u;
  for (int rr = 0; rr < q; ++rr) {
    g_cta += *cl.map_shared_rank(&sh.cta_gt, rr);
    e_cta += *cl.map_shared_rank(&sh.cta_eq, rr);
  }
  uint32_t grun = 0u;  // the CTA's earlier groups' totals
#pragma unroll
  for (int u = 0; u < NG; ++u) {
    if (u < ng) {
      const uint32_t before = grun + sh.wtot[u][warp];
      grun += sh.gbase[u];
      uint32_t g = g_cta + (before >> 16) + ((ex_gt[u >> 2] >> (8 * (u & 3))) & 0xFFu);
      uint32_t e = e_cta + (before & 0xFFFFu) + ((ex_eq[u >> 2] >> (8 * (u & 3))) & 0xFFu);
      const uint4 kk = keys4[u * kThreads + tid];
      const uint32_t ks[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = (u * kThreads + tid) * 4 + j;
        const bool valid = !checked || pos < n;
        if (valid && ks[j] > thr) {
          const uint32_t o = g + min(e, need);
          if (o < static_cast<uint32_t>(K)) out[o] = lo + pos;
          ++g;
        } else if (valid && ks[j] == thr) {
          if (e < need && g + e < static_cast<uint32_t>(K)) out[g + e] = lo + pos;
          ++e;
        }
      }
    }
  }
  cl.sync();  // keep this CTA's shared memory alive until the cluster is done with it
}

// ---------------------------------------------------------------------------
// Rows longer than a cluster's shared memory holds (score_width > 8 x 32K):
// the same selection, with every pass streaming the row's scores from the
// score buffer instead of shared memory (commit message 4: past 64K keys the
// selection should touch only the candidates of the threshold; here the
// indexer's exact first-level histogram names the k-th key's bin before any
// score is read, so a pass keeps only that bin's keys on chip).
//
// One cluster of 2, 4 or 8 CTAs per row; CTA q owns a contiguous segment of
// the row (at most 512K keys) and warp w of the CTA a contiguous range of
// that segment, read in steps of kStreamU float4 loads per lane:
//  A. the row's histogram: the indexer's counts if they total the row
//     length, else counted in one pass and summed over the cluster;
//  B. the bin of the k-th key; C. one pass copies out the keys inside it
//     (at most kCandMax for the row, then two radix passes over them in
//     shared memory) or, for heavier bins, two passes refine the threshold
//     10 bits at a time;
//  D. one pass counts, per warp, the keys above the threshold key tau and
//     equal to it; warp and cluster prefixes of those counts then give, in a
//     second pass, every selected key its rank in ascending position order.
// Integer work on the same keys as the in-shared-memory kernel, so the
// result is the same, bit for bit.
// ---------------------------------------------------------------------------
constexpr int kStreamCluster = 8;
constexpr int kMaxStreamWidth = 1 << 22;                  // the longest row (score_width) supported
constexpr int kStreamU = 4;                               // float4 loads per lane and step
constexpr int kStreamStep = 4 * 32 * kStreamU;            // keys per warp step
constexpr int kStreamSegAlign = kStreamStep * kWarps;     // a CTA segment is a multiple of this

constexpr int kSelMax = 4096;                             // top-k sizes the one-pass path takes
constexpr int kStreamSegMax = kMaxStreamWidth / kStreamCluster;  // the longest CTA segment (512K keys)
constexpr int kStreamWordsMax = kStreamSegMax / 32;               // its bitmap words

struct StreamShared {
  uint32_t hist[kBins1];        // this CTA's counts (read by the whole cluster)
  uint32_t hist_tot[kBins1];    // the row's counts
  uint32_t cand[kCandMax];      // this CTA's candidates (read by the whole cluster)
  uint32_t all_cand[kCandMax];  // the cluster's candidates
  uint32_t cand_pos[kCandMax];  // one-pass path: the positions of this CTA's candidates
  uint32_t sel_pos[kSelMax];    // one-pass path: positions of this CTA's keys above the threshold bin
  uint32_t bits[kStreamWordsMax];  // one-pass path: one bit per position of this CTA's segment
  uint32_t nsel, cta_n, tie_cut;
  uint32_t scan[kWarps];
  uint32_t wgt[kWarps], weq[kWarps];  // per warp: keys > tau and == tau in its range, then their prefixes
  uint32_t count;                     // this CTA's candidates
  uint32_t cta_gt, cta_eq;            // this CTA's totals (read by later ranks)
  uint32_t digit, above;
};

// Keys of row positions i .. i+3 (i a multiple of 4) that lie before `end`;
// nv = how many do.  vec: the row is 16-byte aligned, so whole groups load
// as one float4.
__device__ __forceinline__ void load_keys4(const float *srow, int i, int end, bool vec, uint32_t (&k)[4],
                                           int &nv) {
  nv = min(max(end - i, 0), 4);
  if (vec && nv == 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(srow + i));
    k[0] = order_key(v.x);
    k[1] = order_key(v.y);
    k[2] = order_key(v.z);
    k[3] = order_key(v.w);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) k[j] = j < nv ? order_key(__ldcg(srow + i + j)) : 0u;
  }
}

// The block's set bits of sh.bits[0, nwords) in ascending order: returns
// each thread's first rank (exclusive prefix of the counts of the threads
// before it; thread t holds words [t*per, (t+1)*per)) and the block's total.
__device__ __forceinline__ uint32_t bits_prefix(StreamShared &sh, int nwords, int per, uint32_t &total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t cnt = 0u;
  for (int w = tid * per; w < min(nwords, (tid + 1) * per); ++w) cnt += __popc(sh.bits[w]);
  const uint32_t incl = warp_incl_scan(cnt, lane);
  if (lane == 31) sh.scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = warp_incl_scan(sh.scan[lane], lane);
    sh.scan[lane] = v;
  }
  __syncthreads();
  total = sh.scan[kWarps - 1];
  return incl - cnt + (warp > 0 ? sh.scan[warp - 1] : 0u);
}

__global__ void __launch_bounds__(kThreads, 1) topk_stream_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  StreamShared &sh = *reinterpret_cast<StreamShared *>(smem_raw);
  cg::cluster_group cl = cg::this_cluster();
  pdl_launch_dependents();
  const int C = static_cast<int>(cl.num_blocks());
  const int q = static_cast<int>(cl.block_rank());
  const int wr = blockIdx.x / C;  // row within the window
  const int r = p.row_lo + wr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.topk;
  int32_t *out = p.topk_idx + static_cast<size_t>(r) * K;
  int L = p.row_len[r];  // row metadata, not the indexer's output: read while it finishes
  pdl_wait();            // the scores come from the indexer kernel
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
  // this CTA's segment [lo, hi) and this warp's range [wlo, whi) of it
  const int seg = (((L + C - 1) / C) + kStreamSegAlign - 1) / kStreamSegAlign * kStreamSegAlign;
  const int lo = min(L, q * seg), hi = min(L, lo + seg);
  const int ws = seg / kWarps;  // a multiple of kStreamStep
  const int wlo = min(hi, lo + warp * ws), whi = min(hi, wlo + ws);
  const float *srow = p.scores + static_cast<size_t>(wr) * p.score_width;
  const bool vec = (p.score_width & 3) == 0;

  // ---- A. the row's histogram
  bool recount = ghist == nullptr;
  if (!recount) {
    uint32_t part = 0u;
#pragma unroll
    for (int j = 0; j < kBins1 / kThreads; ++j) {
      const uint32_t v = __ldcg(ghist + j * kThreads + tid);
      sh.hist_tot[j * kThreads + tid] = v;
      part += v;
    }
    part = warp_sum(part);
    if (lane == 0) sh.scan[warp] = part;
  }
  __syncthreads();
  if (!recount) {
    uint32_t total = 0u;
#pragma unroll 8
    for (int w = 0; w < kWarps; ++w) total += sh.scan[w];
    recount = total != static_cast<uint32_t>(L);  // same verdict in every CTA
  }
  if (recount) {
    for (int i = tid; i < kBins1; i += kThreads) sh.hist[i] = 0u;
    __syncthreads();
    for (int base = wlo; base < whi; base += kStreamStep) {
      uint32_t k[kStreamU][4];
      int nv[kStreamU];
#pragma unroll
      for (int u = 0; u < kStreamU; ++u) load_keys4(srow, base + u * 128 + 4 * lane, whi, vec, k[u], nv[u]);
#pragma unroll
      for (int u = 0; u < kStreamU; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nv[u]) atomicAdd(&sh.hist[k[u][j] >> 20], 1u);
    }
    __syncthreads();
    cl.sync();
    for (int b = tid; b < kBins1; b += kThreads) {
      uint32_t s = 0u;
      for (int rr = 0; rr < C; ++rr) s += cl.map_shared_rank(sh.hist, rr)[b];
      sh.hist_tot[b] = s;
    }
  }
  __syncthreads();

  // ---- B. the bin of the k-th key
  uint32_t need = static_cast<uint32_t>(K);
  select_bin(sh, sh.hist_tot, kBins1, need);
  const uint32_t d1 = min(sh.digit, static_cast<uint32_t>(kBins1 - 1));  // found whenever L > K
  need -= sh.above;
  const uint32_t in_bin = sh.hist_tot[d1];
  uint32_t prefix = d1 << 20, mask = 0xFFF00000u;

  if (in_bin <= static_cast<uint32_t>(kCandMax) && K <= kSelMax) {
    // ---- one pass over the row: a key above the threshold bin is selected
    // (its position kept), a key inside it is a candidate (key and position
    // kept); everything after this runs on chip
    if (tid == 0) {
      sh.count = 0u;
      sh.nsel = 0u;
    }
    __syncthreads();
    for (int base = wlo; base < whi; base += kStreamStep) {
      uint32_t k[kStreamU][4];
      int nv[kStreamU];
#pragma unroll
      for (int u = 0; u < kStreamU; ++u) load_keys4(srow, base + u * 128 + 4 * lane, whi, vec, k[u], nv[u]);
#pragma unroll
      for (int u = 0; u < kStreamU; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nv[u]) {
            const uint32_t kb = k[u][j] & mask;
            const uint32_t pos = static_cast<uint32_t>(base + u * 128 + 4 * lane + j);
            if (kb > prefix) {
              const uint32_t at = atomicAdd(&sh.nsel, 1u);
              if (at < static_cast<uint32_t>(kSelMax)) sh.sel_pos[at] = pos;
            } else if (kb == prefix) {
              const uint32_t at = atomicAdd(&sh.count, 1u);
              if (at < static_cast<uint32_t>(kCandMax)) {
                sh.cand[at] = k[u][j];
                sh.cand_pos[at] = pos;
              }
            }
          }
    }
    __syncthreads();
    cl.sync();  // every CTA's candidates are complete (and the row histogram was read)
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;  // ready for the next step
    uint32_t total = 0u;
    for (int rr = 0; rr < C; ++rr) {
      const uint32_t cnt = min(*cl.map_shared_rank(&sh.count, rr), static_cast<uint32_t>(kCandMax));
      const uint32_t *src = cl.map_shared_rank(sh.cand, rr);
      for (uint32_t i = tid; i < cnt && total + i < static_cast<uint32_t>(kCandMax); i += kThreads)
        sh.all_cand[total + i] = src[i];
      total += cnt;
    }
    if (tid == 0 && q == 0) {
      if (total > static_cast<uint32_t>(kCandMax)) flag_status(p.status, DSA_DEV_BAD_ROW);  // scores vs histogram
      if (total != in_bin) flag_status(p.status, DSA_DEV_BAD_HIST);
    }
    total = min(total, static_cast<uint32_t>(kCandMax));
    __syncthreads();
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      const uint32_t dg = radix_pass(sh, sh.all_cand, total, shift, prefix, mask, need);
      prefix |= dg << shift;
      mask |= 0x3FFu << shift;
    }
    const uint32_t tau = prefix;  // `need` keys equal to tau still fit
    // this CTA's candidates above tau (all selected) and equal to it
    const uint32_t own = min(sh.count, static_cast<uint32_t>(kCandMax));
    uint32_t gt = 0u, eq = 0u;
    for (uint32_t i = tid; i < own; i += kThreads) {
      gt += sh.cand[i] > tau ? 1u : 0u;
      eq += sh.cand[i] == tau ? 1u : 0u;
    }
    gt = warp_sum(gt);
    eq = warp_sum(eq);
    if (lane == 0) {
      sh.wgt[warp] = gt;
      sh.weq[warp] = eq;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t tg = 0u, te = 0u;
      for (int w = 0; w < kWarps; ++w) {
        tg += sh.wgt[w];
        te += sh.weq[w];
      }
      sh.cta_gt = tg;
      sh.cta_eq = te;
    }
    __syncthreads();
    cl.sync();  // every CTA's tie count is visible
    // ties are taken in position order: the CTAs before this one come first
    uint32_t e_before = 0u;
    for (int rr = 0; rr < q; ++rr) e_before += *cl.map_shared_rank(&sh.cta_eq, rr);
    const uint32_t eq_cta = sh.cta_eq;
    const uint32_t allowed = need > e_before ? min(need - e_before, eq_cta) : 0u;
    const int nwords = (hi - lo + 31) / 32;
    const int per = (nwords + kThreads - 1) / kThreads;
    // the position of this CTA's allowed-th tie (when only some of them fit)
    if (tid == 0) sh.tie_cut = allowed == eq_cta ? 0xFFFFFFFFu : 0u;
    if (allowed > 0u && allowed < eq_cta) {
      for (int w = tid; w < nwords; w += kThreads) sh.bits[w] = 0u;
      __syncthreads();
      for (uint32_t i = tid; i < own; i += kThreads)
        if (sh.cand[i] == tau) {
          const uint32_t b = sh.cand_pos[i] - static_cast<uint32_t>(lo);
          atomicOr(&sh.bits[b >> 5], 1u << (b & 31));
        }
      __syncthreads();
      uint32_t tot;
      uint32_t rank = bits_prefix(sh, nwords, per, tot);
      for (int w = tid * per; w < min(nwords, (tid + 1) * per); ++w) {
        uint32_t bw = sh.bits[w];
        while (bw != 0u) {
          const int b = __ffs(static_cast<int>(bw)) - 1;
          if (rank == allowed - 1u) sh.tie_cut = static_cast<uint32_t>(lo + w * 32 + b);
          ++rank;
          bw &= bw - 1u;
        }
      }
    }
    __syncthreads();
    const uint32_t tie_cut = sh.tie_cut;
    // this CTA's selection, marked in its segment's bitmap
    for (int w = tid; w < nwords; w += kThreads) sh.bits[w] = 0u;
    __syncthreads();
    const uint32_t nsel = min(sh.nsel, static_cast<uint32_t>(kSelMax));
    for (uint32_t i = tid; i < nsel; i += kThreads) {
      const uint32_t b = sh.sel_pos[i] - static_cast<uint32_t>(lo);
      atomicOr(&sh.bits[b >> 5], 1u << (b & 31));
    }
    for (uint32_t i = tid; i < own; i += kThreads) {
      const uint32_t key = sh.cand[i], pos = sh.cand_pos[i];
      if (key > tau || (key == tau && allowed > 0u && pos <= tie_cut)) {
        const uint32_t b = pos - static_cast<uint32_t>(lo);
        atomicOr(&sh.bits[b >> 5], 1u << (b & 31));
      }
    }
    if (tid == 0) sh.cta_n = nsel + sh.cta_gt + allowed;
    __syncthreads();
    cl.sync();  // every CTA's count is visible
    uint32_t offset = 0u;
    for (int rr = 0; rr < q; ++rr) offset += *cl.map_shared_rank(&sh.cta_n, rr);
    uint32_t tot;
    uint32_t rank = offset + bits_prefix(sh, nwords, per, tot);
    for (int w = tid * per; w < min(nwords, (tid + 1) * per); ++w) {
      uint32_t bw = sh.bits[w];
      while (bw != 0u) {
        const int b = __ffs(static_cast<int>(bw)) - 1;
        if (rank < static_cast<uint32_t>(K)) out[rank] = lo + w * 32 + b;
        ++rank;
        bw &= bw - 1u;
      }
    }
    if (tid == 0 && q == C - 1 && offset + tot != static_cast<uint32_t>(K))
      flag_status(p.status, DSA_DEV_BAD_HIST);  // the counts do not add up to k
    cl.sync();  // keep this CTA's shared memory alive until the cluster is done with it
    return;
  }

  // ---- C. the threshold key tau and how many keys equal to it still fit
  if (in_bin <= static_cast<uint32_t>(kCandMax)) {
    if (tid == 0) sh.count = 0u;
    __syncthreads();
    for (int base = wlo; base < whi; base += kStreamStep) {
      uint32_t k[kStreamU][4];
      int nv[kStreamU];
#pragma unroll
      for (int u = 0; u < kStreamU; ++u) load_keys4(srow, base + u * 128 + 4 * lane, whi, vec, k[u], nv[u]);
#pragma unroll
      for (int u = 0; u < kStreamU; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nv[u] && (k[u][j] & mask) == prefix) {
            const uint32_t at = atomicAdd(&sh.count, 1u);  // order is irrelevant: only counts follow
            if (at < static_cast<uint32_t>(kCandMax)) sh.cand[at] = k[u][j];
          }
    }
    __syncthreads();
    cl.sync();  // every CTA's candidates are complete (and the row histogram was read)
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;  // ready for the next step
    uint32_t total = 0u;
    for (int rr = 0; rr < C; ++rr) {
      const uint32_t cnt = min(*cl.map_shared_rank(&sh.count, rr), static_cast<uint32_t>(kCandMax));
      const uint32_t *src = cl.map_shared_rank(sh.cand, rr);
      for (uint32_t i = tid; i < cnt && total + i < static_cast<uint32_t>(kCandMax); i += kThreads)
        sh.all_cand[total + i] = src[i];
      total += cnt;
    }
    if (tid == 0 && q == 0) {
      if (total > static_cast<uint32_t>(kCandMax)) flag_status(p.status, DSA_DEV_BAD_ROW);  // scores vs histogram
      if (total != in_bin) flag_status(p.status, DSA_DEV_BAD_HIST);
    }
    total = min(total, static_cast<uint32_t>(kCandMax));
    __syncthreads();
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      const uint32_t dg = radix_pass(sh, sh.all_cand, total, shift, prefix, mask, need);
      prefix |= dg << shift;
      mask |= 0x3FFu << shift;
    }
  } else {
    cl.sync();  // every CTA has read the row histogram
    if (ghist != nullptr && q == 0)
      for (int i = tid; i < kBins1; i += kThreads) ghist[i] = 0u;
#pragma unroll 1
    for (int shift = 10; shift >= 0; shift -= 10) {
      cl.sync();  // nobody still reads this CTA's previous counts
      for (int i = tid; i < kBins2; i += kThreads) sh.hist[i] = 0u;
      __syncthreads();
      for (int base = wlo; base < whi; base += kStreamStep) {
        uint32_t k[kStreamU][4];
        int nv[kStreamU];
#pragma unroll
        for (int u = 0; u < kStreamU; ++u) load_keys4(srow, base + u * 128 + 4 * lane, whi, vec, k[u], nv[u]);
#pragma unroll
        for (int u = 0; u < kStreamU; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < nv[u] && (k[u][j] & mask) == prefix) atomicAdd(&sh.hist[(k[u][j] >> shift) & 0x3FFu], 1u);
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
  }
  const uint32_t thr = prefix;  // tau

  // ---- D. ranks of the selected keys in position order
  {
    uint32_t g = 0u, e = 0u;
    for (int base = wlo; base < whi; base += kStreamStep) {
      uint32_t k[kStreamU][4];
      int nv[kStreamU];
#pragma unroll
      for (int u = 0; u < kStreamU; ++u) load_keys4(srow, base + u * 128 + 4 * lane, whi, vec, k[u], nv[u]);
#pragma unroll
      for (int u = 0; u < kStreamU; ++u)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nv[u]) {
            g += k[u][j] > thr ? 1u : 0u;
            e += k[u][j] == thr ? 1u : 0u;
          }
    }
    g = warp_sum(g);
    e = warp_sum(e);
    if (lane == 0) {
      sh.wgt[warp] = g;
      sh.weq[warp] = e;
    }
  }
  __syncthreads();
  if (tid == 0) {  // exclusive prefixes over the warps, and the CTA's totals
    uint32_t rg = 0u, re = 0u;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t tg = sh.wgt[w], te = sh.weq[w];
      sh.wgt[w] = rg;
      sh.weq[w] = re;
      rg += tg;
      re += te;
    }
    sh.cta_gt = rg;
    sh.cta_eq = re;
  }
  __syncthreads();
  cl.sync();  // every CTA's totals are visible
  uint32_t g = sh.wgt[warp], e = sh.weq[warp];
  for (int rr = 0; rr < q; ++rr) {
    g += *cl.map_shared_rank(&sh.cta_gt, rr);
    e += *cl.map_shared_rank(&sh.cta_eq, rr);
  }
  for (int base = wlo; base < whi; base += kStreamStep) {
    uint32_t k[kStreamU][4];
    int nv[kStreamU];
#pragma unroll
    for (int u = 0; u < kStreamU; ++u) load_keys4(srow, base + u * 128 + 4 * lane, whi, vec, k[u], nv[u]);
#pragma unroll
    for (int u = 0; u < kStreamU; ++u) {
      // this lane's four positions follow those of the lanes below it
      uint32_t cg4 = 0u, ce4 = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < nv[u]) {
          cg4 += k[u][j] > thr ? 1u : 0u;
          ce4 += k[u][j] == thr ? 1u : 0u;
        }
      const uint32_t packed = (cg4 << 16) | ce4;
      if (__any_sync(0xFFFFFFFFu, packed != 0u)) {  // most steps select nothing
        const uint32_t incl = warp_incl_scan(packed, lane);
        const uint32_t ex = incl - packed;
        uint32_t gl = g + (ex >> 16), el = e + (ex & 0xFFFFu);
        const int i0 = base + u * 128 + 4 * lane;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j >= nv[u]) continue;
          if (k[u][j] > thr) {
            const uint32_t o = gl + min(el, need);
            if (o < static_cast<uint32_t>(K)) out[o] = i0 + j;
            ++gl;
          } else if (k[u][j] == thr) {
            if (el < need && gl + el < static_cast<uint32_t>(K)) out[gl + el] = i0 + j;
            ++el;
          }
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        g += tot >> 16;
        e += tot & 0xFFFFu;
      }
    }
  }
  cl.sync();  // keep this CTA's shared memory alive until the cluster is done with it
}

}  // namespace

// CTAs per row: ceil(W / 16K), at most 4, keeps one row's chain short when
// the rows' clusters fit on the GPU at once (an 8-CTA cluster waits for 8
// free SMs of one GPC as the indexer drains: at W = 128K keys, 4 CTAs of 32K
// keys finish in 22.7 us against 28.7 us for 8 of 16K); with more rows than
// that, the fewest CTAs the shared memory allows (ceil(W / 32K), which is
// 8 only for rows longer than 128K keys) finish the batch in fewer waves.
constexpr int kPreferredCluster = 4;
int topk_cluster_size(int score_width, int max_rows) {
  const int c_min = std::max(1, (score_width + kSegMax - 1) / kSegMax);
  int c = std::max(c_min, std::min(kPreferredCluster, (score_width + kSegPerCta - 1) / kSegPerCta));
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      static_cast<long long>(max_rows) * c > sms)
    c = c_min;
  return c;
}

cudaError_t launch_topk(const dsa_config_t &cfg, const TopkParams &p, int rows, cudaStream_t st) {
  if (cfg.score_width > kSegMax * kMaxCluster) {  // rows past what a cluster's shared memory holds
    const size_t smem = sizeof(StreamShared);
    cudaError_t e = cudaFuncSetAttribute(topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // CTAs per row: at least what keeps a CTA's segment within its bitmap
    // (512K keys), more (up to 8) while the rows' clusters still fit on the
    // GPU at once; an 8-CTA cluster needs 8 free SMs of one GPC, and only
    // 15 of them fit at a time (1M prefill: 66 rows, 195 us with 8 CTAs per
    // row)
    int sms = 0, dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int c_min = (cfg.score_width + kStreamSegMax - 1) / kStreamSegMax;
    int c = 2;
    while (c < kStreamCluster && static_cast<long long>(rows) * c * 2 <= sms) c *= 2;
    c = std::max(c, c_min);
    c = c <= 2 ? 2 : c <= 4 ? 4 : 8;
    e = launch_pdl(topk_stream_kernel, dim3(static_cast<unsigned>(rows * c)), dim3(kThreads), smem, st,
                   static_cast<unsigned>(c), p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  const int C = topk_cluster_size(cfg.score_width, rows);
  if (C > kMaxCluster) return cudaErrorInvalidValue;
  const int seg_w = (((cfg.score_width + C - 1) / C) + 127) & ~127;
  if (seg_w > kSegMax) return cudaErrorInvalidValue;
  const int groups = (seg_w + 4 * kThreads - 1) / (4 * kThreads);
  const int ng = groups <= 1 ? 1 : groups <= 2 ? 2 : groups <= 4 ? 4 : 8;
  const size_t smem = ((sizeof(TopkShared) + 15) & ~size_t(15)) + static_cast<size_t>(ng) * 4 * kThreads * 4;
  auto k = ng == 1 ? topk_cluster_kernel<1> : ng == 2 ? topk_cluster_kernel<2>
           : ng == 4 ? topk_cluster_kernel<4> : topk_cluster_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_pdl(k, dim3(static_cast<unsigned>(rows * C)), dim3(kThreads), smem, st,
                 static_cast<unsigned>(C), p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
