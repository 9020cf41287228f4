// Sparse GQA attention over the selected keys (split) and the split merge.
//
// Megatron-LM PR #7211, commit message 1: all query heads of a KV group are
// handled together so each selected key and value row is read once, and the
// top-k slots are split across programs whose slices are merged flash-decoding
// style; commit message 8: probabilities enter the value reduction in fp32.
//
// sparse_attn_kernel: persistent CTAs walk the (row, split) work items.  Warp
// 0 is the gather producer: its lanes resolve 32 selected slots at a time
// (slot -> position -> page -> row offset, bounds-checked), two rounds ahead
// of the copies so the dependent loads never stall the ring, and issue one
// cp.async.bulk per token for its K row and one for its V row (all KV heads
// of a token are contiguous, Hkv*D*2 bytes) — or, with the interleaved cache
// layout, one copy for both (the producer's copy-issue rate, not the bytes,
// bounds an L2-resident gather) — into a ring of shared-memory stages that
// complete on mbarriers.  Warps 1..Hkv are consumers, one per KV
// head g: scores on the tensor cores (mma.sync m16n8k16 with the group's <= 8
// query heads as the A rows and 8 keys as N; key fragments by ldmatrix from
// rows padded by 16 bytes so the 8 rows hit distinct banks), an online
// softmax in the log2 domain in fp32, and the value reduction O^T += V^T P^T
// on the tensor cores too (mma.sync m16n8k8, V^T by ldmatrix.trans): the
// score accumulator fragment is already P^T's B fragment, and each fp32
// probability enters as three bf16 terms hi + mid + lo that sum to it, so
// the probabilities are not rounded before the value reduction.
// Bytes in flight are set by the ring depth, not by registers.  Every wait is
// bounded by an SM-clock budget; a wait that runs out sets DSA_DEV_TIMEOUT.
//
// merge_kernel: one warp per (row, head), or per 2-8 of them when S is
// small; combines the S partial states.
#include <math.h>

#include <algorithm>
#include <type_traits>

#include "dsa_common.cuh"
#include "tc_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTokA = 8;         // selected keys per stage
constexpr int kMaxKvHeads = 8;  // consumer warps per CTA
constexpr int kMaxStagesA = 6;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr long long kWaitBudgetA = 2000000000LL;  // SM cycles (about 1 s)

// Flash-decoding merge of one (row, head): S partial states -> bf16 output
// and lse.  Lane j holds dims [j*VN, j*VN + VN) and the states of splits j
// and j + 32.  The m, l and the first kRound accumulator loads are issued
// together, so a merge of up to kRound splits costs one memory round trip.
constexpr int kMergeRound = 24;

template <int D>
__device__ __forceinline__ void merge_one(const float *part_m, const float *part_l, const float *part_acc,
                                          long long rh, int S, uint8_t *out, float *lse, int lane) {
  constexpr int VN = D / 32;
  using VecT = typename std::conditional<VN == 4, float4, float2>::type;
  const float *pm = part_m + rh * S, *pl = part_l + rh * S;
  const float *src0 = part_acc + rh * S * D + lane * VN;
  float ls0 = 0.f, ls1 = 0.f, mr0 = -INFINITY, mr1 = -INFINITY;
  if (lane < S) { ls0 = __ldcg(pl + lane); mr0 = __ldcg(pm + lane); }
  if (lane + 32 < S) { ls1 = __ldcg(pl + lane + 32); mr1 = __ldcg(pm + lane + 32); }
  float v[kMergeRound][VN];
#pragma unroll
  for (int u = 0; u < kMergeRound; ++u) {
    if (u < S) {
      const VecT t = __ldcg(reinterpret_cast<const VecT *>(src0 + static_cast<size_t>(u) * D));
      v[u][0] = t.x;
      v[u][1] = t.y;
      if constexpr (VN == 4) { v[u][2] = t.z; v[u][3] = t.w; }
    }
  }
  // an empty split (l = 0) carries no weight whatever its m
  const float ms0 = ls0 > 0.f ? mr0 : -INFINITY, ms1 = ls1 > 0.f ? mr1 : -INFINITY;
  float mx = fmaxf(ms0, ms1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  const float f0 = ms0 == -INFINITY ? 0.f : __expf(ms0 - mx);
  const float f1 = ms1 == -INFINITY ? 0.f : __expf(ms1 - mx);
  float lsum = ls0 * f0 + ls1 * f1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);

  float o[VN];
#pragma unroll
  for (int d = 0; d < VN; ++d) o[d] = 0.f;
#pragma unroll
  for (int u = 0; u < kMergeRound; ++u) {
    const float fs = __shfl_sync(0xFFFFFFFFu, f0, u & 31);
    if (u < S) {
#pragma unroll
      for (int d = 0; d < VN; ++d) o[d] = fmaf(fs, v[u][d], o[d]);
    }
  }
  for (int s2 = kMergeRound; s2 < S; ++s2) {  // more splits than one round holds
    const VecT t = __ldcg(reinterpret_cast<const VecT *>(src0 + static_cast<size_t>(s2) * D));
    const float fs = __shfl_sync(0xFFFFFFFFu, (s2 & 32) ? f1 : f0, s2 & 31);
    o[0] = fmaf(fs, t.x, o[0]);
    o[1] = fmaf(fs, t.y, o[1]);
    if constexpr (VN == 4) { o[2] = fmaf(fs, t.z, o[2]); o[3] = fmaf(fs, t.w, o[3]); }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(out) + rh * D + lane * VN;
#pragma unroll
  for (int d = 0; d < VN; d += 2)
    *reinterpret_cast<__nv_bfloat162 *>(dst + d) = __floats2bfloat162_rn(o[d] * inv, o[d + 1] * inv);
  if (lse && lane == 0) lse[rh] = lsum > 0.f ? mx + logf(lsum) : -INFINITY;
}

// PPW (row, head) merges per warp when S <= SMAX: the warp's PPW * S
// partial slices are contiguous (layout [R*Hq, S, D]) and all issued in one
// round, so a small S does not leave the warp one short round trip.  Lane
// j * SMAX + s holds m and l of split s of the warp's pair j.  SMAX is S
// rounded up to the kernels built (the registers holding the slices, and
// with them the warps an SM keeps, follow PPW * SMAX).
template <int D, int PPW, int SMAX>
__device__ __forceinline__ void merge_multi(const MergeParams &p, long long rh0, long long total, int lane) {
  static_assert(PPW * SMAX <= 32, "one lane per (pair, split)");
  constexpr int VN = D / 32;
  using VecT = typename std::conditional<VN == 4, float4, float2>::type;
  const int S = p.num_splits;
  const int mj = lane / SMAX, msl = lane - mj * SMAX;  // this lane's (pair, split) for m and l
  float lsv = 0.f, mrv = -INFINITY;
  if (mj < PPW && msl < S && rh0 + mj < total) {
    lsv = __ldcg(p.part_l + (rh0 + mj) * S + msl);
    mrv = __ldcg(p.part_m + (rh0 + mj) * S + msl);
  }
  float v[PPW][SMAX][VN];
#pragma unroll
  for (int j = 0; j < PPW; ++j)
#pragma unroll
    for (int s = 0; s < SMAX; ++s)
      if (s < S && rh0 + j < total) {
        const VecT t = __ldcg(reinterpret_cast<const VecT *>(p.part_acc + ((rh0 + j) * S + s) * D + lane * VN));
        v[j][s][0] = t.x;
        v[j][s][1] = t.y;
        if constexpr (VN == 4) { v[j][s][2] = t.z; v[j][s][3] = t.w; }
      }
  const float msv = lsv > 0.f ? mrv : -INFINITY;  // an empty split carries no weight
#pragma unroll
  for (int j = 0; j < PPW; ++j) {
    const long long rh = rh0 + j;
    if (rh >= total) break;  // warp-uniform
    float mx = mj == j ? msv : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    const float f = (mj != j || msv == -INFINITY) ? 0.f : __expf(msv - mx);
    float lsum = lsv * f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
    float o[VN];
#pragma unroll
    for (int d = 0; d < VN; ++d) o[d] = 0.f;
#pragma unroll
    for (int s = 0; s < SMAX; ++s) {
      const float fs = __shfl_sync(0xFFFFFFFFu, f, j * SMAX + s);
      if (s < S) {
#pragma unroll
        for (int d = 0; d < VN; ++d) o[d] = fmaf(fs, v[j][s][d], o[d]);
      }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + rh * D + lane * VN;
#pragma unroll
    for (int d = 0; d < VN; d += 2)
      *reinterpret_cast<__nv_bfloat162 *>(dst + d) = __floats2bfloat162_rn(o[d] * inv, o[d + 1] * inv);
    if (p.lse && lane == 0) p.lse[rh] = lsum > 0.f ? mx + logf(lsum) : -INFINITY;
  }
}

// Merges per warp for S splits and the splits' lanes per pair (few kernels).
inline int merge_pairs_per_warp(int S) { return S <= 3 ? 8 : S <= 6 ? 4 : S <= 12 ? 2 : 1; }
inline int merge_split_lanes(int S) {
  return S <= 3 ? S : S == 4 ? 4 : S <= 6 ? 6 : S <= 8 ? 8 : S <= 12 ? 12 : 32;
}

template <int D, int PPW, int SMAX>
__global__ void __launch_bounds__(256, (PPW * SMAX * D <= 16 * 128 ? 3 : 2)) merge_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total = static_cast<long long>(p.max_rows) * p.num_q_heads;
  const long long rh0 = (static_cast<long long>(blockIdx.x) * 8 + warp) * PPW;  // first (row, head)
  // rows of length 0 (pad rows) hold only empty partials: their outputs are
  // written as such without reading them (row lengths are step inputs, read
  // before the wait for the attention kernel)
  bool empty = false;
  if (p.row_len != nullptr && rh0 < total) {
    const long long last = std::min(rh0 + PPW, total) - 1;
    empty = true;
    for (long long r = rh0 / p.num_q_heads; r <= last / p.num_q_heads; ++r) empty = empty && p.row_len[r] == 0;
  }
  pdl_wait();  // the partials come from the attention kernel
  if (rh0 >= total) return;
  if (empty) {
    for (long long rh = rh0; rh < std::min(rh0 + PPW, total); ++rh) {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + rh * D;
      for (int d = lane * 2; d < D; d += 64)
        *reinterpret_cast<__nv_bfloat162 *>(dst + d) = __floats2bfloat162_rn(0.f, 0.f);
      if (p.lse && lane == 0) p.lse[rh] = -INFINITY;
    }
    return;
  }
  if constexpr (PPW == 1)
    merge_one<D>(p.part_m, p.part_l, p.part_acc, rh0, p.num_splits, p.out, p.lse, lane);
  else
    merge_multi<D, PPW, SMAX>(p, rh0, total, lane);
}

struct AttnLayout {
  int stages;
  int row_bytes;  // Hkv * D * 2: one token's K (or V) row, all KV heads
  int tok_pitch;  // shared-memory stride between a stage's tokens (16 B of padding per row)
  int v_off;      // offset of a token's V row from its K row in a stage
  int stage_bytes;
  uint32_t off_ok, off_items, off_bar, off_misc;
};

struct RowSplit {
  int r, s, L, req, a, b;
};

__device__ __forceinline__ RowSplit row_split(const AttnParams &p, int item, bool flag) {
  RowSplit x;
  x.r = item / p.num_splits;
  x.s = item % p.num_splits;
  if (p.grouped != nullptr && p.grouped[x.r] != 0) {  // the prefill-group kernel has this row
    x.L = -1;
    x.req = 0;
    x.a = x.b = 0;
    return x;
  }
  int L = p.row_len[x.r];
  const int req = p.row_req[x.r];
  const bool ok = L >= 0 && L <= p.score_width && (L == 0 || (req >= 0 && req < p.max_reqs));
  if (!ok) {
    if (flag) flag_status(p.status, DSA_DEV_BAD_ROW);
    L = 0;
  }
  x.L = L;
  x.req = L > 0 ? req : 0;
  const int n = min(p.topk, L);
  x.a = static_cast<int>((static_cast<long long>(x.s) * n) / p.num_splits);
  x.b = static_cast<int>((static_cast<long long>(x.s + 1) * n) / p.num_splits);
  return x;
}

// The CTA's items (item k = blockIdx.x + k * gridDim.x), resolved once into
// shared memory before the kernel waits for the top-k, so neither the
// producer's look-ahead nor a consumer starting an item waits on the row
// metadata loads: [kItemCache][8] = a, b, L, req, r, s.  Items past the
// cache are resolved on the spot.
constexpr int kItemCache = 64;

__device__ __forceinline__ RowSplit item_split(const AttnParams &p, const int *tab, int ncache, int k, bool flag) {
  if (k < ncache) {
    const int4 e0 = *reinterpret_cast<const int4 *>(tab + 8 * k);
    const int2 e1 = *reinterpret_cast<const int2 *>(tab + 8 * k + 4);
    RowSplit x;
    x.a = e0.x;
    x.b = e0.y;
    x.L = e0.z;
    x.req = e0.w;
    x.r = e1.x;
    x.s = e1.y;
    return x;
  }
  return row_split(p, blockIdx.x + k * gridDim.x, flag);
}

// One round of the gather: up to 32 consecutive selected slots [base,
// min(base + 32, b)) of one item (row split), lane j holding slot base + j.
struct GatherRound {
  bool valid;
  int k, base, b, L;  // k: the item's index among this CTA's items
  const int32_t *sel, *pt;
};

__device__ __forceinline__ GatherRound round_at(const AttnParams &p, const int *tab, int ncache, int k, int nmine,
                                                int lane) {
  GatherRound d;
  d.valid = false;
  d.base = d.b = d.L = 0;
  d.sel = d.pt = nullptr;
  for (d.k = k; d.k < nmine; ++d.k) {  // the next item with slots
    const RowSplit x = item_split(p, tab, ncache, d.k, lane == 0);
    if (x.a < x.b) {
      d.valid = true;
      d.base = x.a;
      d.b = x.b;
      d.L = x.L;
      d.sel = p.topk_idx + static_cast<size_t>(x.r) * p.topk;
      d.pt = p.page_table + static_cast<size_t>(x.req) * p.max_pages_per_req;
      break;
    }
  }
  return d;
}
__device__ __forceinline__ GatherRound next_round(const AttnParams &p, const int *tab, int ncache, GatherRound d,
                                                  int nmine, int lane) {
  if (!d.valid) return d;
  if (d.base + 4 * kTokA < d.b) {
    d.base += 4 * kTokA;
    return d;
  }
  return round_at(p, tab, ncache, d.k + 1, nmine, lane);
}
// The selected position of this lane's slot (-1: none).
__device__ __forceinline__ int load_slot(const GatherRound &d, int lane) {
  const int i = d.base + lane;
  return d.valid && i < d.b ? d.sel[i] : -1;
}
// The page id holding position t, loaded only for a position inside the row.
__device__ __forceinline__ int load_page(const AttnParams &p, const GatherRound &d, int t) {
  return t >= 0 && t < d.L ? d.pt[t >> p.page_shift] : -1;
}
// Element offset of the token row of position t on page pg, or -1 (slot
// unused or out of bounds; the bounds cases are flagged).
__device__ __forceinline__ long long resolve_slot(const AttnParams &p, const GatherRound &d, int t, int pg,
                                                  long long tok_stride) {
  if (t == -1) return -1;
  if (t < 0 || t >= d.L) {
    flag_status(p.status, DSA_DEV_BAD_INDEX);
    return -1;
  }
  if (pg < 0 || pg >= p.num_pages) {
    flag_status(p.status, DSA_DEV_BAD_PAGE);
    return -1;
  }
  return (static_cast<long long>(pg) * p.page_size + (t & (p.page_size - 1))) * tok_stride;
}

__device__ __forceinline__ bool warp_wait_a(uint32_t bar, uint32_t parity, const volatile int *abort_flag) {
  const bool ok = tc::mbar_wait(bar, parity, abort_flag, kWaitBudgetA);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <int D>
__global__ void __launch_bounds__(32 * (1 + kMaxKvHeads), 2) sparse_attn_kernel(const AttnParams p,
                                                                              const AttnLayout lay) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, G = Hq / Hkv, S = p.num_splits;
  const int NST = lay.stages, pitch = lay.tok_pitch;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t stageB = static_cast<uint32_t>(lay.stage_bytes);  // K block then V block, or [K|V] per token
  int *tok_ok = reinterpret_cast<int *>(smem + lay.off_ok);        // [NST][kTokA]
  const uint32_t bar0 = sbase + lay.off_bar;
  auto FULL = [&](int st) { return bar0 + 8u * st; };
  auto EMPTY = [&](int st) { return bar0 + 8u * (NST + st); };
  volatile int *abort_flag = reinterpret_cast<int *>(smem + lay.off_misc);

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      tc::mbar_init(FULL(st), 1);
      tc::mbar_init(EMPTY(st), Hkv);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  pdl_launch_dependents();
  // this CTA's items from the row metadata (not produced by the top-k, so
  // read while the top-k still runs; with prefill groups the rows the group
  // kernel takes are known only after the kernels before)
  if (p.grouped != nullptr) pdl_wait();
  const int items = p.max_rows_attn * S;
  const int nmine = static_cast<int>(blockIdx.x) < items ? (items - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  const int ncache = min(nmine, kItemCache);
  int *item_tab = reinterpret_cast<int *>(smem + lay.off_items);
  for (int k = threadIdx.x; k < ncache; k += blockDim.x) {
    const RowSplit x = row_split(p, blockIdx.x + k * gridDim.x, true);
    *reinterpret_cast<int4 *>(item_tab + 8 * k) = make_int4(x.a, x.b, x.L, x.req);
    *reinterpret_cast<int2 *>(item_tab + 8 * k + 4) = make_int2(x.r, x.s);
  }
  if (p.grouped == nullptr) pdl_wait();  // the selection comes from the top-k kernel
  __syncthreads();

  const long long tok_stride = static_cast<long long>(Hkv) * D * (p.kv_interleaved ? 2 : 1);  // elements per token

  if (warp == 0) {
    // ====================================================== gather producer
    // Rounds of up to 32 selected slots (one item = one row split) are
    // resolved ahead of their copies: while round A's stages are issued, the
    // page ids of round B and the top-k slots of round C are in flight, so
    // the two dependent loads per slot (slot -> position -> page) never stall
    // the ring.
    const uint64_t policy = tc::l2_evict_first_policy();
    int chunk = 0;  // global chunk counter (ring position)
    int pst = 0, pph = 0;  // its ring stage and phase
    bool stop = false;
    GatherRound dA = round_at(p, item_tab, ncache, 0, nmine, lane);
    GatherRound dB = next_round(p, item_tab, ncache, dA, nmine, lane);
    GatherRound dC = next_round(p, item_tab, ncache, dB, nmine, lane);
    int tA = load_slot(dA, lane);
    int tB = load_slot(dB, lane);
    int tC = load_slot(dC, lane);
    int pgA = load_page(p, dA, tA);
    long long offA = resolve_slot(p, dA, tA, pgA, tok_stride);
    while (dA.valid && !stop) {
      const int pgB = load_page(p, dB, tB);  // lands while round A is issued
      for (int sub = 0; sub < 4 && dA.base + sub * kTokA < dA.b; ++sub, ++chunk) {
        const int st = pst;
        if (!warp_wait_a(EMPTY(st), pph ^ 1, abort_flag)) {
          if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
          stop = true;
          break;
        }
        const bool mine = (lane >> 3) == sub;
        if (mine) tok_ok[st * kTokA + (lane & 7)] = offA >= 0 ? 1 : 0;
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, mine && offA >= 0);
        __syncwarp();
        if (lane == 0)
          tc::mbar_arrive_expect_tx(FULL(st), static_cast<uint32_t>(__popc(valid)) * 2u * lay.row_bytes);
        __syncwarp();
        if (mine && offA >= 0) {
          const uint32_t dk = sbase + st * stageB + (lane & 7) * pitch;
          if (p.kv_interleaved) {  // the token's K and V rows in one copy
            tc::bulk_load(dk, p.k_cache + offA * 2, 2u * lay.row_bytes, FULL(st), policy);
          } else {
            tc::bulk_load(dk, p.k_cache + offA * 2, lay.row_bytes, FULL(st), policy);
            tc::bulk_load(dk + lay.v_off, p.v_cache + offA * 2, lay.row_bytes, FULL(st), policy);
          }
        }
        if (++pst == NST) { pst = 0; pph ^= 1; }
      }
      offA = resolve_slot(p, dB, tB, pgB, tok_stride);
      dA = dB;
      dB = dC;
      tB = tC;
      dC = next_round(p, item_tab, ncache, dC, nmine, lane);
      tC = load_slot(dC, lane);
    }
    // drain: no copy may land after the CTA exits
    if (lane == 0)
      for (int c = max(0, chunk - NST); c < chunk; ++c)
        tc::mbar_wait(FULL(c % NST), (c / NST) & 1, nullptr, kWaitBudgetA);
    __syncwarp();
  } else if (warp <= Hkv) {
    // ============================================ consumers: one per KV head
    const int g = warp - 1;
    const int c4 = lane & 3, g4 = lane >> 2;  // g4: query head of the group (A row)
    int cst = 0, cph = 0;  // ring stage and phase of the next chunk
    for (int k = 0; k < nmine; ++k) {
      const RowSplit x = item_split(p, item_tab, ncache, k, false);
      if (x.L < 0) continue;  // a prefill-group row: its partials come from the group kernel
      if (x.L == 0 && p.skip_empty_rows) continue;  // a pad row inside dsa_step: nothing reads its partials
      // A operand: this group's query heads (rows 8..15 are zero padding)
      uint32_t qa[D / 16][2];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = qa[ks][1] = 0u;
        if (g4 < G) {
          const uint8_t *qrow = p.q + ((static_cast<size_t>(x.r) * Hq + g * G + g4) * D + ks * 16 + 2 * c4) * 2;
          qa[ks][0] = *reinterpret_cast<const uint32_t *>(qrow);
          qa[ks][1] = *reinterpret_cast<const uint32_t *>(qrow + 16);
        }
      }
      float m = -INFINITY, l = 0.f;  // head g4, log2 domain
      // O^T[dim][head] accumulators: o[mt] = dims 16mt + g4 (+8), heads 2c4, 2c4+1
      float o[D / 16][4];
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      bool aborted = false;
      for (int base = x.a; base < x.b; base += kTokA) {
        const int st = cst;
        if (!warp_wait_a(FULL(st), cph, abort_flag)) {
          if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
          aborted = true;
          break;
        }
        const uint32_t kst = sbase + st * stageB;
        const int *ok = tok_ok + st * kTokA;
        const int tok = lane & 7, mat = lane >> 3;
        // S[head][token] = Q . K^T over D (mma m16n8k16: A = query heads, B = keys)
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const uint32_t kaddr = kst + tok * pitch + (g * D + (mat >> 1) * 16 + (mat & 1) * 8) * 2;
#pragma unroll
          for (int ks = 0; ks < D / 16; ks += 2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kaddr + ks * 32, b0, b1, b2, b3);
            mma_bf16_16816(c, qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
            mma_bf16_16816(c, qa[ks + 1][0], 0u, qa[ks + 1][1], 0u, b2, b3);
          }
        }
        const bool v0 = ok[2 * c4] != 0, v1 = ok[2 * c4 + 1] != 0;
        const float x0 = v0 ? c[0] * p.sm_scale_log2 : -INFINITY;
        const float x1 = v1 ? c[1] * p.sm_scale_log2 : -INFINITY;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float mn = fmaxf(m, mx);
        const float al = mn == -INFINITY ? 1.f : exp2f(m - mn);
        const float p0 = x0 == -INFINITY ? 0.f : exp2f(x0 - mn);
        const float p1 = x1 == -INFINITY ? 0.f : exp2f(x1 - mn);
        float ps = p0 + p1;
        ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 1);
        ps += __shfl_xor_sync(0xFFFFFFFFu, ps, 2);
        l = l * al + ps;
        m = mn;
        // rescale the columns of heads 2c4, 2c4+1 (their factors live in lanes 8c4, 8c4+4)
        const float al_a = __shfl_sync(0xFFFFFFFFu, al, 8 * c4);
        const float al_b = __shfl_sync(0xFFFFFFFFu, al, 8 * c4 + 4);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          o[mt][0] *= al_a;
          o[mt][1] *= al_b;
          o[mt][2] *= al_a;
          o[mt][3] *= al_b;
        }
        // O^T += V^T . P^T on the tensor cores with the fp32 probabilities kept
        // exact: p = hi + mid + lo (three bf16 terms), and this lane's (p0, p1)
        // is already the B fragment (P^T[token 2c4, 2c4+1][head g4]).
        uint32_t ph, pm, pl;
        split3_bf16x2(p0, p1, ph, pm, pl);
        const uint32_t vmask = (v0 ? 0x0000FFFFu : 0u) | (v1 ? 0xFFFF0000u : 0u);
        const uint32_t vaddr = kst + lay.v_off + tok * pitch + (g * D + (mat & 1) * 8 + (mat >> 1) * 16) * 2;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt += 2) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(vaddr + mt * 32, a0, a1, a2, a3);
          a0 &= vmask;
          a1 &= vmask;
          a2 &= vmask;
          a3 &= vmask;
          // hi and mid in one k16 MMA: its K runs over (token, term) pairs,
          // so the V^T fragment appears twice and P_hi, P_mid are the two
          // halves of the B fragment; lo in a k8 MMA
          mma_bf16_16816(o[mt], a0, a1, a0, a1, ph, pm);
          mma_bf16_1688(o[mt], a0, a1, pl);
          mma_bf16_16816(o[mt + 1], a2, a3, a2, a3, ph, pm);
          mma_bf16_1688(o[mt + 1], a2, a3, pl);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(EMPTY(st));
        if (++cst == NST) { cst = 0; cph ^= 1; }
      }
      if (aborted) break;
      // partial state of heads g*G .. g*G+G-1 for this split
      const size_t rh0 = static_cast<size_t>(x.r) * Hq + static_cast<size_t>(g) * G;
      // the merge reads them right after this kernel: keep them in L2 while
      // the K/V stream (evict-first) passes through
      const uint64_t keep = tc::l2_evict_last_policy();
      if (c4 == 0 && g4 < G) {
        tc::st_global_hint(p.part_m + (rh0 + g4) * S + x.s, m == -INFINITY ? -INFINITY : m * kLn2, keep);
        tc::st_global_hint(p.part_l + (rh0 + g4) * S + x.s, l, keep);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * c4 + e;
        if (h < G) {
          float *dst = p.part_acc + ((rh0 + h) * S + x.s) * D + g4;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            tc::st_global_hint(dst + 16 * mt, o[mt][e], keep);
            tc::st_global_hint(dst + 16 * mt + 8, o[mt][2 + e], keep);
          }
        }
      }
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_sparse_attn(const dsa_config_t &cfg, const AttnParams &p, cudaStream_t st) {
  AttnLayout lay;
  lay.row_bytes = cfg.num_kv_heads * cfg.head_dim * 2;
  if (p.kv_interleaved) {  // [K|V] per token
    lay.tok_pitch = 2 * lay.row_bytes + 16;
    lay.v_off = lay.row_bytes;
    lay.stage_bytes = kTokA * lay.tok_pitch;
  } else {  // the stage's K rows, then its V rows
    lay.tok_pitch = lay.row_bytes + 16;
    lay.v_off = kTokA * lay.tok_pitch;
    lay.stage_bytes = 2 * kTokA * lay.tok_pitch;
  }
  const int stage_bytes = lay.stage_bytes;
  int stages = (100 * 1024) / stage_bytes;  // about 100 KB of ring: two CTAs per SM
  stages = stages < 2 ? 2 : (stages > kMaxStagesA ? kMaxStagesA : stages);
  lay.stages = stages;
  uint32_t off = static_cast<uint32_t>(stages) * stage_bytes;
  lay.off_ok = off;
  off += stages * kTokA * 4;
  off = (off + 15u) & ~15u;
  lay.off_items = off;
  off += kItemCache * 8 * 4;
  lay.off_bar = off;
  off += 2 * stages * 8;
  lay.off_misc = off;
  off += 16;
  const size_t smem = off;
  const int threads = 32 * (1 + cfg.num_kv_heads);
  cudaError_t e;
  int per_sm = 0, dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int items = cfg.max_rows * cfg.num_splits;
  if (cfg.head_dim == 128) {
    auto k = sparse_attn_kernel<128>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem)) != cudaSuccess) return e;
    const int grid = std::max(1, std::min(items, std::max(1, per_sm) * sms));
    if ((e = launch_pdl(k, dim3(grid), dim3(threads), smem, st, 1u, p, lay)) != cudaSuccess) return e;
  } else if (cfg.head_dim == 64) {
    auto k = sparse_attn_kernel<64>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem)) != cudaSuccess) return e;
    const int grid = std::max(1, std::min(items, std::max(1, per_sm) * sms));
    if ((e = launch_pdl(k, dim3(grid), dim3(threads), smem, st, 1u, p, lay)) != cudaSuccess) return e;
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const dsa_config_t &cfg, const MergeParams &p, cudaStream_t st) {
  const long long pairs = static_cast<long long>(cfg.max_rows) * cfg.num_q_heads;
  const int ppw = merge_pairs_per_warp(cfg.num_splits), sl = merge_split_lanes(cfg.num_splits);
  const unsigned blocks = static_cast<unsigned>((pairs + 8LL * ppw - 1) / (8LL * ppw));
  void (*k)(const MergeParams) = nullptr;
  auto pick = [&](auto d) -> void (*)(const MergeParams) {
    constexpr int D = decltype(d)::value;
    switch (sl) {
      case 1: return merge_kernel<D, 8, 1>;
      case 2: return merge_kernel<D, 8, 2>;
      case 3: return merge_kernel<D, 8, 3>;
      case 4: return merge_kernel<D, 4, 4>;
      case 6: return merge_kernel<D, 4, 6>;
      case 8: return merge_kernel<D, 2, 8>;
      case 12: return merge_kernel<D, 2, 12>;
      default: return merge_kernel<D, 1, 32>;
    }
  };
  if (cfg.head_dim == 128)
    k = pick(std::integral_constant<int, 128>());
  else if (cfg.head_dim == 64)
    k = pick(std::integral_constant<int, 64>());
  else
    return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(k, dim3(blocks), dim3(256), 0, st, 1u, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
