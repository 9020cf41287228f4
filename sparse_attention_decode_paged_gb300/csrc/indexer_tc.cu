// Lightning-indexer scores on the 5th-generation tensor cores (tcgen05 + TMA).
//
//   scores[r, t] = s_t * sum_h w[r, h] * max(0, q_idx[r, h, :] . k_t),  t < row_len[r]
//
// Megatron-LM PR #7211, commit message 1: the indexer streams page-contiguous
// key tiles through tensor cores and each request's programs stride over its
// row only up to its length; commit message 2: the rows of one score block are
// scored against shared key tiles.
//
// Design (one persistent CTA per SM, 10 warps):
//  * Work is the flat list of 128-token key tiles of all score blocks
//    (block b contributes ceil(L_max(b) / 128) tiles).  Every CTA scans the
//    block table, prefix-sums the tile counts and takes an equal contiguous
//    range of tiles, so the launch depends only on the static config while
//    the work follows the real lengths.
//  * Warp 0 (producer): streams each tile's pages with 2-D TMA loads (one box
//    per page and 128-byte K atom, 128-byte swizzle, one lane per box so a
//    tile's boxes issue in parallel) into a ring of shared-memory stages;
//    when the score block changes it stages the block's queries as the
//    MMA's B operand (bf16 by TMA; fp8 swizzled by hand).
//    fp8 keys: each query head x is written as two e4m3 terms with one scale
//    s = amax/448, x/s = hi + lo (lo = the e4m3 rounding of the residual),
//    and both terms are multiplied by the same key tile into the same
//    accumulator (relative error about 2^-8); s is folded into the head
//    weight since ReLU(s y) = s ReLU(y) for s > 0.
//  * Warp 1 (MMA): one thread issues tcgen05.mma, transposed so that the key
//    tile is A (M = 128 tokens) and the block's queries are B (N = 16..256
//    heads x rows), accumulating in fp32 in tensor memory; four accumulator
//    buffers (two when 4 x N columns do not fit in TMEM) let the epilogue of
//    tile i overlap the MMAs of the next tiles, so a slow epilogue does not
//    hold a key stage.
//  * Warps 2..9 (epilogue, two warpgroups taking alternate tiles, so each
//    has two tiles' time): thread i of a warpgroup owns TMEM lane i = token
//    i of the tile, reads its heads with tcgen05.ld, forms
//    sum_h w_h ReLU(acc_h) with no cross-thread reduction, scales by s_t and
//    stores the score.
//  * Every wait is bounded; a wait that runs out sets DSA_DEV_TIMEOUT and an
//    abort flag that releases the other roles, the producer waits for its
//    copies in flight and the MMA warp for its MMAs, and TMEM is freed.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "dsa_common.cuh"
#include "tc_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTok = 128;  // tokens per key tile (MMA M)
constexpr int kWarps = 10;  // 0 producer, 1 MMA, 2..5 and 6..9 two epilogue warpgroups
constexpr int kThreads = kWarps * 32;
constexpr long long kWaitBudget = 2000000000LL;  // SM cycles (about 1 s)
constexpr long long kTestWaitBudget = 2000000LL;  // SM cycles (about 1 ms): the test-only wait
constexpr int kMaxRowsTc = 4096;                  // prefix table capacity
constexpr int kMaxStages = 16;                    // key-tile ring depth at most
constexpr int kTileCost0 = 4;                     // a tile's cost: kTileCost0 + its block's rows

struct TcLayout {
  int hp;         // indexer heads padded to a multiple of 16
  int n_max;      // hp * block_rows: accumulator columns per buffer
  int stages;     // key-tile ring depth
  int nq;         // query buffers (1 or 2)
  int nacc;       // TMEM accumulator buffers (2 or 4)
  int tmem_cols;  // allocated TMEM columns (power of two >= 32)
  uint32_t off_q, off_w, off_prefix, off_blk, off_bar, off_misc;
};

template <int RB>
__device__ __forceinline__ uint32_t swizzle(uint32_t off) {
  constexpr uint32_t mask = RB == 128 ? 7u : (RB == 64 ? 3u : 1u);
  return off ^ (((off >> 7) & mask) << 4);
}

template <int RB>
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr) {
  constexpr uint64_t layout = RB == 128 ? 2u : (RB == 64 ? 4u : 6u);
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1u) << 16) |
         (static_cast<uint64_t>((8u * RB) >> 4) << 32) | (static_cast<uint64_t>(1u) << 46) |
         (layout << 61);
}

// Every lane of the warp waits (each acquires the barrier's phase); the
// verdict is made warp-uniform so no lane continues alone.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag) {
  const bool ok = tc::mbar_wait(bar, parity, abort_flag, kWaitBudget);
  return __all_sync(0xFFFFFFFFu, ok);
}

struct BlockInfo {
  int first, nrows, req, lmax;
  int lens[4];
};

// A block's rows inside the scored window (a block may straddle its edge).
__device__ __forceinline__ BlockInfo load_block(const IndexerParams &p, int b) {
  BlockInfo bi;
  const int first = p.block_first[b];
  bi.first = max(first, p.row_lo);
  bi.nrows = min(first + p.block_nrows[b], p.row_hi) - bi.first;
  bi.req = p.row_req[bi.first];
  bi.lmax = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    bi.lens[i] = i < bi.nrows ? p.row_len[bi.first + i] : 0;
    bi.lmax = max(bi.lmax, bi.lens[i]);
  }
  return bi;
}

// Stages a score block's fp8 queries: each query head x (bf16) becomes two
// e4m3 terms hi + lo with one scale s = amax/448 (x/s = hi + lo, lo the e4m3
// rounding of the residual), written swizzled as the MMA's two B parts, and
// s folds into the head weight.  Threads t of nthr (a multiple of 32) work in
// teams of kMembers per head, each on a share of the head's RB dims (whole
// 16-byte e4m3 chunks); every thread of the participating warps must call it
// (the teams reduce amax by shuffles).
template <int RB>
__device__ __forceinline__ void stage_q_fp8(const IndexerParams &p, const BlockInfo &bi, uint8_t *qdst,
                                            uint32_t qpartB, float *wdst, int NMAX, int HP, int t, int nthr) {
  constexpr int kMembers = RB / 16 < 4 ? RB / 16 : 4;
  constexpr int kPart = RB / kMembers;  // dims (= e4m3 bytes) per team member, a multiple of 16
  const int DIr = p.idx_dim;
  const int team = t / kMembers, part = t % kMembers, nteams = nthr / kMembers;
  for (int base = 0; base < NMAX; base += nteams) {  // same trip count in every lane
    const int n = base + team;
    const int rr = n / HP, h = n % HP;
    const bool live = n < NMAX && rr < bi.nrows && h < p.idx_heads;
    const uint8_t *src = p.q_idx + (static_cast<size_t>(bi.first + rr) * p.idx_heads + h) * DIr * 2;
    uint4 v[kPart / 8];  // this member's kPart bf16 inputs
#pragma unroll
    for (int c = 0; c < kPart / 8; ++c) {
      const int d0 = part * kPart + c * 8;
      v[c] = (live && d0 < DIr) ? *reinterpret_cast<const uint4 *>(src + d0 * 2) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < kPart / 8; ++c) {
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16lo(v[c].x)), fabsf(bf16hi(v[c].x))),
                               fmaxf(fabsf(bf16lo(v[c].y)), fabsf(bf16hi(v[c].y)))));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16lo(v[c].z)), fabsf(bf16hi(v[c].z))),
                               fmaxf(fabsf(bf16lo(v[c].w)), fabsf(bf16hi(v[c].w)))));
    }
#pragma unroll
    for (int o = 1; o < kMembers; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (n >= NMAX) continue;
    const float sigma = amax > 0.f ? amax / 448.f : 1.f;
    const float inv = 1.f / sigma;
#pragma unroll
    for (int c = 0; c < kPart / 16; ++c) {  // 16 e4m3 per 16-byte chunk
      uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
      const uint32_t w8[8] = {v[2 * c].x, v[2 * c].y, v[2 * c].z, v[2 * c].w,
                              v[2 * c + 1].x, v[2 * c + 1].y, v[2 * c + 1].z, v[2 * c + 1].w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float x0 = bf16lo(w8[k]) * inv, x1 = bf16hi(w8[k]) * inv;
        const __nv_fp8x2_storage_t ph = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
        __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(ph, __NV_E4M3);
        const float2 hf = __half22float2(*reinterpret_cast<__half2 *>(&hr));
        const __nv_fp8x2_storage_t pl =
            __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
        hi[k >> 1] |= static_cast<uint32_t>(ph) << (16 * (k & 1));
        lo[k >> 1] |= static_cast<uint32_t>(pl) << (16 * (k & 1));
      }
      const uint32_t o = swizzle<RB>(n * RB + part * kPart + c * 16);
      *reinterpret_cast<uint4 *>(qdst + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4 *>(qdst + qpartB + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (part == 0)
      wdst[n] = live ? p.w[static_cast<size_t>(bi.first + rr) * p.idx_heads + h] * sigma : 0.f;
  }
}

// The score block holding tile `item`: b with pf[b] <= item < pf[b+1].
__device__ __forceinline__ int find_block(const int *pf, int nblocks, int item) {
  int lo = 0, hi = nblocks;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pf[mid] <= item) lo = mid;
    else hi = mid;
  }
  while (item >= pf[lo + 1]) ++lo;  // skip blocks without tiles
  return lo;
}

// Walks this CTA's contiguous range of tiles in order; the current block's
// tile range is kept in registers (the loops that use it are latency-bound).
struct Walker {
  const int *prefix;
  int item, end, block, bstart, bnext;
  __device__ __forceinline__ void start(const int *pf, int nblocks, int beg, int e) {
    prefix = pf;
    item = beg;
    end = e;
    block = find_block(pf, nblocks, beg);
    bstart = pf[block];
    bnext = pf[block + 1];
  }
  __device__ __forceinline__ bool valid() const { return item < end; }
  __device__ __forceinline__ int tile() const { return item - bstart; }
  __device__ __forceinline__ bool last_of_block() const { return item + 1 >= bnext || item + 1 >= end; }
  __device__ __forceinline__ void next() {
    ++item;
    if (item < end && item >= bnext) {
      do {
        ++block;
      } while (item >= prefix[block + 1]);
      bstart = prefix[block];
      bnext = prefix[block + 1];
    }
  }
};

// The CTA's score blocks, read once into shared memory so that a block change
// costs no dependent global loads: [kBlkCache][8] = first, nrows, req, lmax,
// lens[4].  Blocks past the first kBlkCache of the CTA are read from global
// memory (16 entries cost 512 bytes; more would take a key stage away).
constexpr int kBlkCache = 16;
struct BlockCache {
  const int *tab;
  int b_lo, n;
  __device__ __forceinline__ BlockInfo get(const IndexerParams &p, int b) const {
    const int i = b - b_lo;
    if (i >= 0 && i < n) {
      const int4 e0 = *reinterpret_cast<const int4 *>(tab + i * 8);
      const int4 e1 = *reinterpret_cast<const int4 *>(tab + i * 8 + 4);
      BlockInfo bi;
      bi.first = e0.x;
      bi.nrows = e0.y;
      bi.req = e0.z;
      bi.lmax = e0.w;
      bi.lens[0] = e1.x;
      bi.lens[1] = e1.y;
      bi.lens[2] = e1.z;
      bi.lens[3] = e1.w;
      return bi;
    }
    return load_block(p, b);
  }
};

template <int RB, int ATOMS, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_tc_kernel(const IndexerParams p, const TcLayout lay, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap qmap) {
  constexpr int kElem = F8 ? 1 : 2;
  constexpr uint32_t kAtomB = kTok * RB;          // one K atom of a key tile
  constexpr uint32_t kStageB = kAtomB * ATOMS;
  constexpr int kKsteps = RB / 32;                // 32 bytes of K per MMA

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sb = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = lay.stages, NQ = lay.nq, HP = lay.hp, NMAX = lay.n_max, NACC = lay.nacc;
  constexpr int kParts = F8 ? 2 : 1;              // fp8: hi and lo query terms
  const uint32_t qpartB = static_cast<uint32_t>(NMAX) * RB * ATOMS;
  const uint32_t qbufB = qpartB * kParts;
  const uint32_t stage0 = base;
  const uint32_t q0 = base + lay.off_q;
  float *wbuf = reinterpret_cast<float *>(sb + lay.off_w);            // [NQ][NMAX]
  int *prefix = reinterpret_cast<int *>(sb + lay.off_prefix);         // [R + 1] tiles before each block
  int *cprefix = prefix + (p.max_rows + 1);                            // [R + 1] their cost before each block
  const uint32_t bar0 = base + lay.off_bar;
  // barrier map: full[S] empty[S] qfull[2] qempty[2] tfull[4] tempty[4] done
  auto FULL = [&](int s) { return bar0 + 8u * s; };
  auto EMPTY = [&](int s) { return bar0 + 8u * (S + s); };
  auto QFULL = [&](int q) { return bar0 + 8u * (2 * S + q); };
  auto QEMPTY = [&](int q) { return bar0 + 8u * (2 * S + 2 + q); };
  auto TFULL = [&](int a) { return bar0 + 8u * (2 * S + 4 + a); };
  auto TEMPTY = [&](int a) { return bar0 + 8u * (2 * S + 8 + a); };
  const uint32_t DONE = bar0 + 8u * (2 * S + 12);
  int *misc = reinterpret_cast<int *>(sb + lay.off_misc);  // [0] tmem base [1] abort [2..33] scan
  volatile int *abort_flag = misc + 1;

  pdl_launch_dependents();  // the top-k kernel may be scheduled as SMs free up

  // ---- tile counts per score block, prefix-summed (every CTA, redundantly)
  const int R = p.max_rows;
  for (int b = tid; b < R; b += kThreads) {
    int nt = 0, cost = 0;
    const int nrows = p.block_nrows[b];
    if (nrows > 0) {
      const int first = p.block_first[b];
      bool ok = nrows <= p.block_rows && first >= 0 && first + nrows <= R;
      const int req = ok ? p.row_req[first] : 0;
      ok = ok && req >= 0 && req < p.max_reqs;
      int lmax = 0, nin = 0;
      for (int i = 0; i < nrows && ok; ++i) {  // checked over the whole block
        const int L = p.row_len[first + i];
        if (p.row_req[first + i] != req || L < 0 || L > p.score_width) ok = false;
        if (first + i >= p.row_lo && first + i < p.row_hi) {  // rows scored here
          lmax = max(lmax, L);
          ++nin;
        }
      }
      if (!ok) {
        if (blockIdx.x == 0) flag_status(p.status, DSA_DEV_BAD_BLOCK);
      } else {
        nt = (lmax + kTok - 1) / kTok;  // 0 for a block outside the window
        cost = nt * (kTileCost0 + nin);
      }
    }
    prefix[b + 1] = nt;
    cprefix[b + 1] = cost;
  }
  if (tid == 0) {
    prefix[0] = 0;
    cprefix[0] = 0;
    misc[1] = 0;
  }
  __syncthreads();
  // inclusive scans of both (in place)
  auto scan = [&](int *arr) {
    const int per = (R + kThreads - 1) / kThreads;
    const int lo = 1 + tid * per, hi = min(R + 1, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += arr[i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) misc[2 + warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w2 = 0; w2 < warp; ++w2) run += misc[2 + w2];
    for (int i = lo; i < hi; ++i) {
      run += arr[i];
      arr[i] = run;
    }
    __syncthreads();
  };
  scan(prefix);
  scan(cprefix);
  // The CTA's tiles: an equal share of the total cost.  A tile of a score
  // block with n rows costs kTileCost0 + n units: a block's rows share its
  // key tiles, but each row adds MMA columns and epilogue sums, so equal
  // tile counts left the CTAs holding 4-row prefill blocks ~50% longer than
  // those holding decode rows (per-CTA end times, mixed and 1M prefill
  // steps; a 4-row tile at 1.6 decode tiles balanced both within a few
  // percent).  Tile t of block b starts at cost cprefix[b] + t * w_b; the
  // CTA takes the tiles whose start falls in its share, so the shares tile
  // the row order without gaps or overlaps.  Decode-only steps (every block
  // one row) keep equal tile counts.
  const int total = prefix[R];
  const int ctotal = cprefix[R];
  auto tile_at = [&](int c) {  // the first tile whose cost start is >= c
    if (c >= ctotal) return total;
    const int b = find_block(cprefix, R, c);
    const int nt = prefix[b + 1] - prefix[b];
    const int w = (cprefix[b + 1] - cprefix[b]) / nt;
    return prefix[b] + (c - cprefix[b] + w - 1) / w;
  };
  const int beg = tile_at(static_cast<int>((static_cast<long long>(blockIdx.x) * ctotal) / gridDim.x));
  const int end = tile_at(static_cast<int>((static_cast<long long>(blockIdx.x + 1) * ctotal) / gridDim.x));
  if (beg >= end) return;  // uniform across the CTA
  BlockCache bc;
  bc.tab = reinterpret_cast<int *>(sb + lay.off_blk);
  bc.b_lo = find_block(prefix, R, beg);
  {
    const int nb = find_block(prefix, R, end - 1) - bc.b_lo + 1;
    bc.n = nb < kBlkCache ? nb : kBlkCache;
    for (int i = tid; i < bc.n; i += kThreads) {
      const int b = bc.b_lo + i;
      if (prefix[b + 1] > prefix[b]) {  // only blocks with tiles passed the checks above
        const BlockInfo bi = load_block(p, b);
        *reinterpret_cast<int4 *>(const_cast<int *>(bc.tab) + i * 8) = make_int4(bi.first, bi.nrows, bi.req, bi.lmax);
        *reinterpret_cast<int4 *>(const_cast<int *>(bc.tab) + i * 8 + 4) =
            make_int4(bi.lens[0], bi.lens[1], bi.lens[2], bi.lens[3]);
      }
    }
  }

  // ---- barriers and tensor memory
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(FULL(s), 1);
      tc::mbar_init(EMPTY(s), 1);
    }
    for (int q = 0; q < 2; ++q) {
      tc::mbar_init(QFULL(q), 1);
      tc::mbar_init(QEMPTY(q), 1 + 8);  // MMA commit + 8 epilogue warps
    }
    for (int a = 0; a < 4; ++a) {
      tc::mbar_init(TFULL(a), 1);
      tc::mbar_init(TEMPTY(a), 4);      // the 4 warps of the owning warpgroup
    }
    tc::mbar_init(DONE, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&kmap);
    if constexpr (!F8) tc::tma_prefetch_desc(&qmap);
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&misc[0]), static_cast<uint32_t>(lay.tmem_cols));
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  // fp8 queries of the CTA's first NQ score blocks: quantised now by warps
  // 1..9 (warp 0, the producer, starts streaming keys meanwhile), so the
  // producer does not do it alone while its key ring drains
  int npre = 0;
  if constexpr (F8) {
    int b = bc.b_lo;
    for (int j = 0; j < NQ && b < R && prefix[b] < end; ++j) {
      if (warp != 0)
        stage_q_fp8<RB>(p, bc.get(p, b), sb + lay.off_q + j * qbufB, qpartB, wbuf + j * NMAX, NMAX, HP, tid - 32,
                        kThreads - 32);
      ++npre;
      do {  // the next block with tiles
        ++b;
      } while (b < R && prefix[b + 1] == prefix[b]);
    }
    if (warp != 0) {
      tc::fence_proxy_async_smem();
      asm volatile("bar.sync 1, %0;\n" ::"r"(kThreads - 32) : "memory");  // warps 1..9 only
      if (tid == 32)
        for (int j = 0; j < npre; ++j) tc::mbar_arrive(QFULL(j));
    }
  }

  Walker wk;
  wk.start(prefix, R, beg, end);

  if (warp == 0) {
    // ======================================================== producer
    const uint64_t policy = tc::l2_evict_first_policy();
    const uint64_t qpolicy = tc::l2_evict_last_policy();
    int cur = -1, qcount = -1, issued = 0;
    int ps = 0, pphase = 0;  // ring position and phase of the next tile
    int qstaged = 0;         // query stagings issued
    int win_base = 0, win_page = -1;  // page ids win_base + lane, held by lane
    int nxt_base = -64, nxt_page = -1;  // the following window, loaded ahead
    BlockInfo bi{};
    const int32_t *pt = nullptr;
    const int P = p.page_size;
    const int npg = kTok / P;  // pages per tile: 1, 2, 4 or 8
    int np_blk = 0;            // pages of the current block up to its longest row
    for (; wk.valid(); wk.next()) {
      if (wk.block != cur) {
        cur = wk.block;
        ++qcount;
        bi = bc.get(p, cur);
        pt = p.page_table + static_cast<size_t>(bi.req) * p.max_pages_per_req;
        np_blk = (bi.lmax + P - 1) / P;
        win_base = -64;  // force a window load for the new block
        nxt_base = -64;
        const int qb = qcount % NQ;
        if (qcount >= npre) {  // (the first npre were staged by the whole CTA before the loop)
          if (!warp_wait(QEMPTY(qb), ((qcount / NQ) & 1) ^ 1, abort_flag)) {
            if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
            break;
          }
          // stage the block's queries (B operand) and head weights
          uint8_t *qdst = sb + lay.off_q + qb * qbufB;
          float *wdst = wbuf + qb * NMAX;
          if constexpr (!F8) {
            // bf16: one TMA box per (row, K atom) writes the swizzled operand
            // directly; when the head count needs no padding the block's weight
            // rows are contiguous and one bulk copy brings them on the same
            // barrier, else the lanes load them (the producer then waits for
            // those loads)
            const bool wbulk = p.idx_heads == HP;
            if (!wbulk) {
              for (int n = lane; n < NMAX; n += 32) {
                const int rr = n / HP, h = n % HP;
                const bool live = rr < bi.nrows && h < p.idx_heads;
                wdst[n] = live ? p.w[static_cast<size_t>(bi.first + rr) * p.idx_heads + h] : 0.f;
              }
              __syncwarp();
            }
            if (lane == 0) {
              const uint32_t wbytes = wbulk ? static_cast<uint32_t>(bi.nrows * HP) * 4u : 0u;
              tc::mbar_arrive_expect_tx(QFULL(qb), static_cast<uint32_t>(bi.nrows) * ATOMS * HP * RB + wbytes);
              if (wbulk)
                tc::bulk_load(smem_u32(wdst), p.w + static_cast<size_t>(bi.first) * p.idx_heads, wbytes, QFULL(qb),
                              qpolicy);
              for (int rr = 0; rr < bi.nrows; ++rr)
#pragma unroll
                for (int a = 0; a < ATOMS; ++a)
                  tc::tma_load_2d(q0 + qb * qbufB + a * NMAX * RB + rr * HP * RB, &qmap, a * (RB / kElem),
                                  (bi.first + rr) * p.idx_heads, QFULL(qb), qpolicy);
            }
          } else {
            // fp8: each query head becomes hi + lo e4m3 terms with one scale
            stage_q_fp8<RB>(p, bi, qdst, qpartB, wdst, NMAX, HP, lane, 32);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(QFULL(qb));
          }
        }
        ++qstaged;
      }
      {
        const int s = ps;
        if (!warp_wait(EMPTY(s), pphase ^ 1, abort_flag)) {
          if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
          break;
        }
        // page ids of this tile from a 32-entry window the whole warp loads
        // at once (one L2 round trip per 32 pages instead of one per page);
        // lane k < npg resolves the tile's page k.  Windows start at
        // multiples of npg and 32 % npg == 0, so a tile never straddles two.
        const int pi0 = wk.tile() * npg;
        if (pi0 >= win_base + 32 || pi0 < win_base) {
          if (pi0 == nxt_base) {
            win_base = nxt_base;
            win_page = nxt_page;
          } else {
            win_base = pi0;
            win_page = win_base + lane < np_blk ? pt[win_base + lane] : -1;
          }
          // load the next window now: it is used 32 pages from here
          nxt_base = win_base + 32;
          nxt_page = nxt_base + lane < np_blk ? pt[nxt_base + lane] : -1;
        }
        const int pi = pi0 + (lane < npg ? lane : 0);
        const int pgl = __shfl_sync(0xFFFFFFFFu, win_page, pi - win_base);
        const bool inblk = lane < npg && pi < np_blk;
        const bool okp = inblk && pgl >= 0 && pgl < p.num_pages;
        const uint32_t okm = __ballot_sync(0xFFFFFFFFu, okp);
        if (__ballot_sync(0xFFFFFFFFu, inblk && !okp) != 0u && lane == 0) flag_status(p.status, DSA_DEV_BAD_PAGE);
        if (lane == 0)
          tc::mbar_arrive_expect_tx(FULL(s), static_cast<uint32_t>(__popc(okm)) * P * RB * ATOMS);
        __syncwarp();
        // one lane per (page, K atom) box: the boxes of a tile are issued in parallel
        {
          const int k = lane / ATOMS, a = lane % ATOMS;
          const int pg = __shfl_sync(0xFFFFFFFFu, pgl, k & 31);
          if (lane < npg * ATOMS && ((okm >> k) & 1u))
            tc::tma_load_2d(stage0 + s * kStageB + a * kAtomB + k * P * RB, &kmap, a * (RB / kElem), pg * P,
                            FULL(s), policy);
        }
        ++issued;
        if (++ps == S) { ps = 0; pphase ^= 1; }
      }
      __syncwarp();
    }
    // no copy may land after the CTA exits: wait for the last stages and
    // query buffers issued
    if (lane == 0) {
      for (int it = max(0, issued - S); it < issued; ++it)
        tc::mbar_wait(FULL(it % S), (it / S) & 1, nullptr, kWaitBudget);
      for (int qc = max(0, qstaged - NQ); qc < qstaged; ++qc)
        tc::mbar_wait(QFULL(qc % NQ), (qc / NQ) & 1, nullptr, kWaitBudget);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================================================ MMA
    // The whole warp runs the loop and one elected lane (always the same
    // one) issues the MMAs and commits, so the descriptors stay
    // warp-uniform: a lone issuing lane runs far slower beside the busy
    // epilogue warps on its scheduler.  The descriptors' start-address field
    // is linear in the shared-memory address (every operand lies below
    // 256 KiB), so they are formed once and advanced by adding offsets >> 4;
    // ring stage, accumulator and phases are running counters.
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    int cur = -1, qcount = -1, qb = 0;
    int ms = 0, msphase = 0, ma = 0, maphase = 0;  // ring stage and accumulator of the next tile
    const uint64_t adesc0 = make_desc<RB>(stage0);
    const uint32_t batomD = static_cast<uint32_t>(NMAX * RB) >> 4, qpartD = qpartB >> 4;
    uint64_t ad_s = adesc0, bd_q = 0;
    uint32_t d = tm, idesc = 0;
    bool any = false, stop = false;
    auto wait = [&](uint32_t bar, int parity) {
      if (!warp_wait(bar, static_cast<uint32_t>(parity), abort_flag)) stop = true;
      return !stop;
    };
    // test only: a wait on the MMA-completion barrier before any MMA is
    // issued, which nothing completes, so it runs out after a short budget
    const bool test_stop =
        p.test_timeout != 0 &&
        !__all_sync(0xFFFFFFFFu, tc::mbar_wait(DONE, 0, abort_flag, kTestWaitBudget));
    for (; wk.valid() && !test_stop; wk.next()) {
      const int s = ms, ab = ma;
      if (wk.block != cur) {
        cur = wk.block;
        ++qcount;
        qb = qcount % NQ;
        idesc = tc::idesc_m128(HP * bc.get(p, cur).nrows, F8);
        bd_q = make_desc<RB>(q0 + qb * qbufB);
        if (!wait(QFULL(qb), (qcount / NQ) & 1)) break;
      }
      if (!wait(TEMPTY(ab), maphase ^ 1)) break;
      if (!wait(FULL(s), msphase)) break;
      tc::tc_fence_after();
      if (tc::elect_one()) {
#pragma unroll
        for (int a = 0; a < ATOMS; ++a)
#pragma unroll
          for (int k = 0; k < kKsteps; ++k) {
            const uint64_t ad = ad_s + static_cast<uint32_t>((a * kAtomB + k * 32) >> 4);
#pragma unroll
            for (int part = 0; part < kParts; ++part) {
              const uint64_t bd = bd_q + (part * qpartD + a * batomD + static_cast<uint32_t>(k * 2));
              tc::mma<F8>(d, ad, bd, idesc, (a | k | part) != 0 ? 1u : 0u);
            }
          }
        tc::mma_commit(EMPTY(s));
        tc::mma_commit(TFULL(ab));
        if (wk.last_of_block()) tc::mma_commit(QEMPTY(qb));
      }
      __syncwarp();
      any = true;
      if (++ms == S) {
        ms = 0;
        msphase ^= 1;
        ad_s = adesc0;
      } else {
        ad_s += kStageB >> 4;
      }
      if (++ma == NACC) {
        ma = 0;
        maphase ^= 1;
        d = tm;
      } else {
        d += static_cast<uint32_t>(NMAX);
      }
    }
    if (wk.valid() && lane == 0) {
      *abort_flag = 1;
      flag_status(p.status, DSA_DEV_TIMEOUT);
    }
    if (any) {  // every MMA issued here has completed before TMEM is freed
      if (tc::elect_one()) tc::mma_commit(DONE);
      __syncwarp();
      if (lane == 0) tc::mbar_wait(DONE, 0, nullptr, kWaitBudget);
    }
    __syncwarp();
  } else {
    // ======================================================= epilogue
    const int wg = (warp - 2) >> 2;  // warpgroup: owns the accumulator buffers of parity wg
    const int quarter = warp & 3;    // TMEM lanes 32*quarter .. +31
    const int tl = quarter * 32 + lane;
    int cur = -1, qcount = -1, qb = 0;
    int ea = 0, eaphase = 0;  // accumulator buffer and phase of the next tile
    const uint64_t keep = tc::l2_evict_last_policy();
    BlockInfo bi{};
    const int32_t *pt = nullptr;
    for (; wk.valid(); wk.next()) {
      const int it = wk.item - beg;
      const int ab = ea;
      const int aphase = eaphase;
      if (++ea == NACC) { ea = 0; eaphase ^= 1; }
      if (wk.block != cur) {
        if (cur >= 0 && lane == 0) tc::mbar_arrive(QEMPTY(qb));  // done with the old weights
        cur = wk.block;
        ++qcount;
        qb = qcount % NQ;
        bi = bc.get(p, cur);
        pt = p.page_table + static_cast<size_t>(bi.req) * p.max_pages_per_req;
        if (!warp_wait(QFULL(qb), (qcount / NQ) & 1, abort_flag)) {
          if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
          break;
        }
      }
      if ((it & 1) != wg) continue;  // the other warpgroup's tile
      const int t = wk.tile() * kTok + tl;
      float sc = 1.f;
      if constexpr (F8) {
        // the key's scale (two dependent loads: page id, then scale) is
        // fetched before the wait for the accumulator, so its latency
        // overlaps the tile's MMA instead of following it
        sc = 0.f;
        if (t < bi.lmax) {
          const int pg = pt[t / p.page_size];
          if (pg >= 0 && pg < p.num_pages)
            sc = p.idx_scale[static_cast<size_t>(pg) * p.page_size + t % p.page_size];
        }
      }
      if (!warp_wait(TFULL(ab), aphase, abort_flag)) {
        if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
        break;
      }
      tc::tc_fence_after();
      const float *wq = wbuf + qb * NMAX;
      const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(ab * NMAX);
      // every row's weighted sum first, so the accumulator goes back to the
      // MMA before the stores and histogram atomics; with 64 heads the
      // accumulator is read in 32-column chunks, the next chunk's load in
      // flight while one is summed
      float sums[4] = {0.f, 0.f, 0.f, 0.f};
      if (HP == 64 && bi.nrows == 1) {  // one row: one load of its 64 heads
        float v[64];
        tc::tmem_ld64_sync(trow, v);
        const float4 *w4 = reinterpret_cast<const float4 *>(wq);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 ww = w4[i];
          s4[0] = fmaf(ww.x, fmaxf(v[4 * i], 0.f), s4[0]);
          s4[1] = fmaf(ww.y, fmaxf(v[4 * i + 1], 0.f), s4[1]);
          s4[2] = fmaf(ww.z, fmaxf(v[4 * i + 2], 0.f), s4[2]);
          s4[3] = fmaf(ww.w, fmaxf(v[4 * i + 3], 0.f), s4[3]);
        }
        sums[0] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      } else if (HP == 64) {
        // the same four chains per row as the one-load path, carried across
        // the row's two chunks, so a row's score has the same bits whatever
        // block (or window) it is scored in
        const int nch = 2 * bi.nrows;
        uint32_t ca[32], cb[32];
        float s4r[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int k = 0; k < 4; ++k) s4r[r][k] = 0.f;
        auto add = [&](const uint32_t (&v)[32], int c) {
          const float4 *w4 = reinterpret_cast<const float4 *>(wq + c * 32);
          float (&s4)[4] = s4r[c >> 1];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 ww = w4[i];
            s4[0] = fmaf(ww.x, fmaxf(__uint_as_float(v[4 * i]), 0.f), s4[0]);
            s4[1] = fmaf(ww.y, fmaxf(__uint_as_float(v[4 * i + 1]), 0.f), s4[1]);
            s4[2] = fmaf(ww.z, fmaxf(__uint_as_float(v[4 * i + 2]), 0.f), s4[2]);
            s4[3] = fmaf(ww.w, fmaxf(__uint_as_float(v[4 * i + 3]), 0.f), s4[3]);
          }
        };
        tc::tmem_ld32_nowait(trow, ca);
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
          if (c < nch) {
            tc::tmem_wait_ld32(ca);
            if (c + 1 < nch) tc::tmem_ld32_nowait(trow + (c + 1) * 32, cb);
            add(ca, c);
          }
          if (c + 1 < nch) {
            tc::tmem_wait_ld32(cb);
            if (c + 2 < nch) tc::tmem_ld32_nowait(trow + (c + 2) * 32, ca);
            add(cb, c + 1);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) sums[r] = (s4r[r][0] + s4r[r][1]) + (s4r[r][2] + s4r[r][3]);
      } else {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          if (rr >= bi.nrows) break;
          float sum = 0.f;
          for (int c = 0; c < HP; c += 16) {
            float v[16];
            tc::tmem_ld16_sync(trow + rr * HP + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) sum = fmaf(wq[rr * HP + c + i], fmaxf(v[i], 0.f), sum);
          }
          sums[rr] = sum;
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(TEMPTY(ab));  // the accumulator is read
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        if (rr >= bi.nrows) break;
        const int L = bi.lens[rr];
        const float score = sums[rr] * sc;
        if (t < L)  // kept in L2 for the top-k that reads them next (the key stream is evict-first)
          tc::st_global_hint(p.scores + static_cast<size_t>(bi.first + rr - p.row_lo) * p.score_width + t, score, keep);
        if (p.row_hist != nullptr) {
          // first-level histogram for the top-k that follows.  In a one-row
          // block the lanes with the same bin add their count with one
          // atomic (measured: the histogram costs the B64 indexer 2 us
          // instead of 6, the long-fp8 one 6 instead of 12); multi-row
          // blocks add key by key, which measured far cheaper there (the
          // mixed step's indexer: +5 us, against +51 with the matching)
          const bool live = t < L;
          if (bi.nrows == 1) {
            const uint32_t bin = live ? (order_key(score) >> 20) : 0xFFFFFFFFu;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bin);
            if (live && lane == __ffs(static_cast<int>(peers)) - 1)
              atomicAdd(p.row_hist + static_cast<size_t>(bi.first) * kKeyBins + bin,
                        static_cast<uint32_t>(__popc(peers)));
          } else if (live) {
            atomicAdd(p.row_hist + static_cast<size_t>(bi.first + rr) * kKeyBins + (order_key(score) >> 20), 1u);
          }
        }
      }
    }
  }

  // ---- teardown: every role is out of its loop and its async work is done
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, static_cast<uint32_t>(lay.tmem_cols));
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

constexpr int kSmemLimit1 = 232448;  // one CTA per SM: 227 KiB of dynamic shared memory
constexpr int kSmemLimit2 = 113 * 1024;  // two CTAs per SM

template <int RB, int ATOMS, bool F8>
cudaError_t launch_tc(const dsa_config_t &cfg, const IndexerParams &p, cudaStream_t st) {
  constexpr int kElem = F8 ? 1 : 2;
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  TcLayout lay;
  lay.hp = (cfg.idx_heads + 15) & ~15;
  lay.n_max = lay.hp * cfg.block_rows;
  if (lay.n_max > 256 || cfg.max_rows > kMaxRowsTc) return cudaErrorInvalidValue;
  // four accumulator buffers when they fit in TMEM: the MMA of tile i then
  // waits for the epilogue of tile i - 4, not i - 2
  lay.nacc = 4 * lay.n_max <= 512 ? 4 : 2;
  int cols = 32;
  while (cols < lay.nacc * lay.n_max) cols <<= 1;
  lay.tmem_cols = cols;
  // One CTA per SM: the deep key ring (as many stages as shared memory
  // holds: 6 of 32 KiB for bf16 keys, 12 of 16 KiB for fp8 keys) hides the
  // MMA/epilogue round trip; the floor keeps a second CTA (and a second TMEM
  // owner) off the SM.
  const int ctas_per_sm = 1;
  const int kSmemLimit = ctas_per_sm == 2 ? kSmemLimit2 : kSmemLimit1;
  const int kSmemFloor = ctas_per_sm == 2 ? 80 * 1024 : 120 * 1024;
  const uint32_t stageB = kTok * RB * ATOMS;
  const uint32_t qbufB = static_cast<uint32_t>(lay.n_max) * RB * ATOMS * (F8 ? 2 : 1);
  // everything but the stages and their two barriers each
  auto fixed = [&](int nq) {
    uint32_t off = nq * qbufB;                    // query buffers (after the stages)
    off += nq * lay.n_max * 4;                    // weights
    off += 2 * (cfg.max_rows + 1) * 4 + 16;       // tile and cost prefix tables
    off += kBlkCache * 8 * 4;                     // block cache
    off += 13 * 8;                                // the other barriers
    return off + 1024 + 34 * 4;                   // alignment slack, misc and scan scratch
  };
  lay.nq = 2;
  int stages = static_cast<int>((kSmemLimit - fixed(2)) / (stageB + 16));
  if (stages < 4) {
    lay.nq = 1;
    stages = static_cast<int>((kSmemLimit - fixed(1)) / (stageB + 16));
  }
  stages = stages > kMaxStages ? kMaxStages : stages;
  if (stages < 2) return cudaErrorInvalidValue;
  lay.stages = stages;
  uint32_t off = stages * stageB;
  lay.off_q = off;
  off += lay.nq * qbufB;
  lay.off_w = off;
  off += lay.nq * lay.n_max * 4;
  lay.off_prefix = off;
  off += 2 * (cfg.max_rows + 1) * 4;
  off = (off + 15u) & ~15u;
  lay.off_blk = off;
  off += kBlkCache * 8 * 4;
  lay.off_bar = off;
  off += (2 * stages + 13) * 8;
  lay.off_misc = off;
  off += 34 * 4;
  size_t smem = off + 1024;
  if (smem < static_cast<size_t>(kSmemFloor)) smem = kSmemFloor;
  if (smem > static_cast<size_t>(kSmemLimit)) return cudaErrorInvalidValue;

  CUtensorMap kmap;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cfg.idx_dim),
                              static_cast<cuuint64_t>(cfg.num_pages) * cfg.page_size};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cfg.idx_dim) * kElem};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(RB / kElem), static_cast<cuuint32_t>(cfg.page_size)};
  const cuuint32_t estride[2] = {1, 1};
  const CUtensorMapSwizzle swz = RB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : RB == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult cr = encode(&kmap, F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                       const_cast<uint8_t *>(p.idx_cache), gdim, gstride, box, estride,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;

  // queries (bf16 path): rows = (row, head), one box = one row's padded heads
  CUtensorMap qmap;
  memset(&qmap, 0, sizeof(qmap));
  if (!F8) {
    const cuuint64_t qdim[2] = {static_cast<cuuint64_t>(cfg.idx_dim),
                                static_cast<cuuint64_t>(cfg.max_rows) * cfg.idx_heads};
    const cuuint64_t qstride[1] = {static_cast<cuuint64_t>(cfg.idx_dim) * 2};
    const cuuint32_t qbox[2] = {static_cast<cuuint32_t>(RB / 2), static_cast<cuuint32_t>(lay.hp)};
    cr = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t *>(p.q_idx), qdim, qstride, qbox,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(indexer_tc_kernel<RB, ATOMS, F8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = ctas_per_sm * sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  indexer_tc_kernel<RB, ATOMS, F8><<<grid, kThreads, smem, st>>>(p, lay, kmap, qmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer_tc(const dsa_config_t &cfg, const IndexerParams &p, cudaStream_t st) {
  const bool f8 = cfg.idx_key_dtype == DSA_KEY_FP8_E4M3;
  if (f8) {
    switch (cfg.idx_dim) {
      case 32: return launch_tc<32, 1, true>(cfg, p, st);
      case 64: return launch_tc<64, 1, true>(cfg, p, st);
      case 128: return launch_tc<128, 1, true>(cfg, p, st);
    }
  } else {
    switch (cfg.idx_dim) {
      case 32: return launch_tc<64, 1, false>(cfg, p, st);
      case 64: return launch_tc<128, 1, false>(cfg, p, st);
      case 128: return launch_tc<128, 2, false>(cfg, p, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace dsa
