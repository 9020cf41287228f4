// Sparse attention for prefill row groups on the 5th-generation tensor cores:
// the rows of one request in a 16-row slot attend to the union of their
// selected keys, each row masked to its own selection.
//
// Megatron-LM PR #7211, commit message 5: prefill rows run in tiles in which
// a group of consecutive query tokens attends to the union of the group's
// selected keys with a per-token bitmask; commit message 1: all query heads
// of a KV group share the group's keys and the top-k slots are split across
// programs whose partial states are merged; commit message 8: probabilities
// enter the value reduction unrounded.
//
// group_union_kernel (one CTA per 16-row slot): the slot's member rows are
// its rows of the request with the most rows in it; a slot with at least
// kGroupMin members whose longest row is at most umax positions (four times
// the most a union of 16 top-k lists can hold) may form a group.  The
// members' selected positions (each row's list ascends, so each chunk's
// entries are found by binary search) are marked in a per-position mask
// (bit j = slot row j) and written out densely, chunk by chunk of the
// longest member's length, with the ascending list of the 128-position tiles
// that hold a selected position.  Positions outside a row's length and pages
// outside the pool are flagged and left out, as the decode kernel does.  The
// slot is a group only if the union fills at least a quarter of the longest
// prefix (else every row stays with the decode kernel, which then moves fewer
// bytes); its rows are marked so the decode kernel leaves them to this one.
//
// group_attn_kernel (persistent, one CTA per SM, 11 warps) walks (slot, KV
// head g, split s) items; split s takes the group's listed tiles
// [s*T/S, (s+1)*T/S) of its T tiles.  The 128 queries of an item are the
// slot's 16 rows x 8 query heads of g (query q = 8 * row + head), the MMA's
// M = 128; a tile's 128 positions are the MMA's N (and the K of P V):
//  * warp 0 (K producer): stages the item's queries with TMA tile loads,
//    then each listed tile's whole pages of K rows of head g (one box per
//    page and 64-element atom, 128-byte swizzle) plus the tile's row masks
//    into a 3-stage ring; warp 10 (V producer) streams the same tiles' V
//    rows into a 2-stage ring.  A prefill group's union covers most of its
//    prefix, so whole pages move with a handful of copies per tile where a
//    gather of the selected rows alone would need one copy per few rows;
//  * warp 1 (MMA; one elected lane issues): S = Q K^T (both K-major) into
//    tensor memory, and O += P V with P read from tensor memory as the A
//    operand and the page-major V tile read as an MN-major B operand;
//  * warps 2..9 (softmax): warpgroup w takes the item's tiles t = w, w + 2,
//    ... with its own S_w (P_w is written over it) and O_w in tensor memory,
//    thread = query.  A running maximum m moves only when a tile's row
//    maximum over the row's selected keys exceeds it by more than 2^8 (then
//    l and the row's O_w are scaled by 2^(m_old - m)); p = exp2(x - m) <= 256
//    (fp32) for the selected keys (0 for the rest) is summed into l and
//    written as two bf16 terms hi + lo (their sum is p to about 2^-17
//    relative), and the MMA runs P V once per term, so the probabilities are
//    not rounded to bf16 before the value reduction;
//  * after the item the two warpgroups combine their row states (exact
//    maximum, l and O scaled to it) and write the split's partial state
//    (m, l, acc) of their member rows, warpgroup w head dims [64w, 64w+64).
// Every wait is bounded; a wait that runs out sets DSA_DEV_TIMEOUT and an
// abort flag, the producers wait for their copies in flight and the MMA warp
// for its MMAs before tensor memory is freed.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "dsa_common.cuh"
#include "tc_ptx.cuh"

namespace dsa {
namespace {

constexpr int kGT = 128;                          // union positions per tile (MMA N of Q K^T, K of P V)
constexpr int kQ = kGroupRows * 8;                // queries per item (MMA M)
constexpr int kKStages = 3;                       // K tile (and row mask) ring
constexpr int kVStages = 2;                       // V tile ring
constexpr int kGWarps = 11;                       // K producer, MMA, 2 softmax warpgroups, V producer
constexpr int kGThreads = kGWarps * 32;
constexpr long long kGWaitBudget = 2000000000LL;  // SM cycles (about 1 s)
constexpr int kUnionThreads = 1024;
constexpr int kUnionSpan = 32768;                 // positions per pass (bitmasks in shared memory)
constexpr int kUnionScan = 16 * kUnionThreads;    // positions per scan step (16 per thread)
constexpr float kLn2G = 0.69314718055994530942f;

// tensor-memory columns, per softmax warpgroup w: S_w [128 x 128] fp32 at
// 128 w (P_w, two bf16 terms of [128 x 128], is written over it), O_w
// [128 x 128] fp32 at 256 + 128 w
constexpr uint32_t kColS = 0, kColO = 256, kTmemCols = 512;

// ------------------------------------------------------------ union kernel
struct SlotInfo {
  int n, req, lmax;
  uint32_t members;  // bit j: slot row j is a member
};

// Thread j < 16 of warp 0 looks at slot row j; the result is broadcast to
// the warp (warp 0 only).
__device__ __forceinline__ SlotInfo slot_members(const AttnParams &p, int slot, int lane, bool flag) {
  const int row = slot * kGroupRows + lane;
  int L = 0, req = -1;
  if (lane < kGroupRows && row < p.max_rows_attn) {
    L = p.row_len[row];
    req = p.row_req[row];
    if (L < 0 || L > p.score_width || (L > 0 && (req < 0 || req >= p.max_reqs))) {
      if (flag) flag_status(p.status, DSA_DEV_BAD_ROW);
      L = 0;
    }
  }
  // the request with the most live rows in the slot (ties: the lowest row's)
  const uint32_t same = __match_any_sync(0xFFFFFFFFu, L > 0 ? req : -1 - lane);
  int score = L > 0 ? (__popc(same) << 5) | (31 - lane) : -1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) score = max(score, __shfl_xor_sync(0xFFFFFFFFu, score, o));
  SlotInfo si;
  si.req = score >= 0 ? __shfl_sync(0xFFFFFFFFu, req, 31 - (score & 31)) : -1;
  si.members = score >= 0 ? __ballot_sync(0xFFFFFFFFu, L > 0 && req == si.req) : 0u;
  si.n = __popc(si.members);
  int lm = (si.members >> lane) & 1u ? L : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lm = max(lm, __shfl_xor_sync(0xFFFFFFFFu, lm, o));
  si.lmax = lm;
  return si;
}

__global__ void __launch_bounds__(kUnionThreads) group_union_kernel(const AttnParams p, const GroupParams gp) {
  extern __shared__ uint32_t mask2[];          // kUnionSpan / 2 words: two 16-bit row masks per word
  __shared__ uint32_t wsum[kUnionThreads / 32];
  __shared__ uint32_t wtiles[kUnionThreads / 32];  // per warp: its 4 tiles that hold a selected position
  __shared__ int s_info[4];                    // members, req, lmax, n
  __shared__ int s_n[kGroupRows], s_len[kGroupRows];  // each member's selected entries and length
  pdl_launch_dependents();
  const int slot = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (warp == 0) {
    const SlotInfo si = slot_members(p, slot, lane, true);
    if (lane == 0) {
      s_info[0] = static_cast<int>(si.members);
      s_info[1] = si.req;
      s_info[2] = si.lmax;
      s_info[3] = si.n;
    }
  }
  __syncthreads();
  const int req = s_info[1], lmax = s_info[2];
  // a group needs kGroupMin rows, and a prefix the union can fill to a
  // quarter at least (umax = 4 x the most a union of 16 top-k lists holds)
  uint32_t members = (s_info[3] >= kGroupMin && lmax <= gp.umax) ? static_cast<uint32_t>(s_info[0]) : 0u;
  const int tmax = gp.umax / kGT;
  int *tiles_out = gp.tiles + static_cast<size_t>(slot) * tmax;
  uint32_t *msk_out = gp.umask + static_cast<size_t>(slot) * (gp.umax / kGT) * 64;
  if (tid < kGroupRows) {
    const bool mem = (members >> tid) & 1u;
    const int L = mem ? p.row_len[slot * kGroupRows + tid] : 0;
    s_len[tid] = L;
    s_n[tid] = mem ? min(p.topk, L) : 0;
  }
  const int32_t *pt = p.page_table + static_cast<size_t>(max(req, 0)) * p.max_pages_per_req;
  // the page of this thread's first 16 positions (an input, not the top-k's
  // output): fetched before the wait, so the first scan does not wait on it
  constexpr int kPer = kUnionScan / kUnionThreads;
  const int pg_first = members != 0u && tid * kPer < lmax ? pt[(tid * kPer) >> p.page_shift] : -1;
  pdl_wait();  // the selection comes from the top-k kernel
  __syncthreads();
  const int K = p.topk;
  int ntile = 0, total = 0;  // tiles holding a selected position, selected positions
  for (int c0 = 0; c0 < lmax && members != 0u; c0 += kUnionSpan) {
    for (int i = tid; i < kUnionSpan / 2; i += kUnionThreads) mask2[i] = 0u;
    __syncthreads();
    // every member's entries (entry i of member j at j * K + i), 16 per
    // thread loaded before any is used, so the loads of all members are in
    // flight together
    for (int f0 = 0; f0 < kGroupRows * K; f0 += 16 * kUnionThreads) {
      int tv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int f = f0 + u * kUnionThreads + tid;
        const int j = f / K, i = f - j * K;
        tv[u] = f < kGroupRows * K && i < s_n[j]  // no member, or past its selected entries: none
                    ? p.topk_idx[static_cast<size_t>(slot * kGroupRows + j) * K + i]
                    : -1;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int f = f0 + u * kUnionThreads + tid;
        const int j = f / K, t = tv[u];
        if (t == -1) continue;
        if (t < 0 || t >= s_len[j]) {
          if (c0 == 0) flag_status(p.status, DSA_DEV_BAD_INDEX);
          continue;
        }
        if (t >= c0 && t < c0 + kUnionSpan) atomicOr(&mask2[(t - c0) >> 1], (1u << j) << (16 * ((t - c0) & 1)));
      }
    }
    __syncthreads();
    for (int s0 = c0; s0 < min(c0 + kUnionSpan, lmax); s0 += kUnionScan) {
      // thread t: positions s0 + 16t .. +15 (8 threads per 128-position tile);
      // a selected position on a page outside the pool is flagged and left out
      constexpr int per = kPer;  // 16, all on one page (page_size >= 16)
      int cnt = 0;
      uint32_t m16[per];  // per position: its 16 row bits
      uint32_t any = 0u;
#pragma unroll
      for (int k = 0; k < per; k += 2) {
        const uint32_t w = mask2[(s0 - c0 + tid * per + k) >> 1];
        m16[k] = w & 0xFFFFu;
        m16[k + 1] = w >> 16;
        any |= w;
      }
      if (any != 0u) {
        const int pg = s0 == 0 ? pg_first : pt[(s0 + tid * per) >> p.page_shift];
        const bool bad = pg < 0 || pg >= p.num_pages;
        if (bad) flag_status(p.status, DSA_DEV_BAD_PAGE);
#pragma unroll
        for (int k = 0; k < per; ++k) {
          if (bad) m16[k] = 0u;
          cnt += m16[k] != 0u ? 1 : 0;
        }
      }
      // stored per tile and row: row j's 128 bits (4 words, bit b of word w =
      // position 32 w + b of the tile); threads 2i and 2i+1 hold the two
      // halves of one word, the even one stores rows 0..7, the odd one 8..15
      {
        const int ti = (s0 >> 7) + (tid >> 3), wd = (tid >> 1) & 3;
        const bool odd = (tid & 1) != 0;
        // transpose the 16 x 16 bit matrix (m16[e] bit j -> m16[j] bit e)
        // by swapping 8-, 4-, 2- and 1-wide blocks
        auto swap_blocks = [&](auto sw_c, uint32_t msk) {
          constexpr int sw = decltype(sw_c)::value;
#pragma unroll
          for (int i = 0; i < per; ++i)
            if ((i & sw) == 0) {
              const uint32_t t = ((m16[i] >> sw) ^ m16[i + sw]) & msk;
              m16[i + sw] ^= t;
              m16[i] ^= t << sw;
            }
        };
        swap_blocks(std::integral_constant<int, 8>{}, 0x00FFu);
        swap_blocks(std::integral_constant<int, 4>{}, 0x0F0Fu);
        swap_blocks(std::integral_constant<int, 2>{}, 0x3333u);
        swap_blocks(std::integral_constant<int, 1>{}, 0x5555u);
#pragma unroll
        for (int j = 0; j < kGroupRows; ++j) {
          const uint32_t h = m16[j];  // row j's bits of this thread's 16 positions
          const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, h, 1);
          const uint32_t word = odd ? (other | (h << 16)) : (h | (other << 16));
          if ((j >= 8) == odd && ti < gp.umax / kGT) msk_out[(static_cast<size_t>(ti) * kGroupRows + j) * 4 + wd] = word;
        }
      }
      // the warp's 4 tiles: lanes 8i .. 8i+7 hold tile i
      const uint32_t nz = __ballot_sync(0xFFFFFFFFu, cnt > 0);
      int wcnt = cnt;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wcnt += __shfl_xor_sync(0xFFFFFFFFu, wcnt, o);
      if (lane == 0) {
        wtiles[warp] = ((nz & 0xFFu) ? 1u : 0u) | ((nz & 0xFF00u) ? 2u : 0u) | ((nz & 0xFF0000u) ? 4u : 0u) |
                       ((nz & 0xFF000000u) ? 8u : 0u);
        wsum[warp] = static_cast<uint32_t>(wcnt);
      }
      __syncthreads();
      // the step's tiles with a selected position, in ascending order
      int before = 0, ctiles = 0, csum = 0;
      for (int w = 0; w < kUnionThreads / 32; ++w) {
        const int nt = __popc(wtiles[w]);
        if (w < warp) before += nt;
        ctiles += nt;
        csum += static_cast<int>(wsum[w]);
      }
      if (lane < 4 && ((wtiles[warp] >> lane) & 1u)) {
        const int at = ntile + before + __popc(wtiles[warp] & ((1u << lane) - 1u));
        const int ti = (s0 >> 7) + warp * 4 + lane;
        if (at < tmax) tiles_out[at] = ti;
      }
      ntile += ctiles;
      total += csum;
      __syncthreads();  // every read of mask2, wsum and wtiles is done before the next step
    }
  }
  if (members != 0u && total * 4 < lmax) members = 0u;  // too sparse: the decode kernel does better
  if (tid < kGroupRows && slot * kGroupRows + tid < p.max_rows_attn)
    gp.grouped[slot * kGroupRows + tid] = (members >> tid) & 1u;
  if (tid == 0) gp.ntiles[slot] = members != 0u ? min(ntile, tmax) : 0;
}

// ------------------------------------------------------- attention kernel
struct GroupLayout {
  uint32_t off_q, off_k, off_v, off_mask, off_xch, off_bar, off_misc;
};

// K-major operand, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}
// MN-major operand, 128-byte swizzle: 64-element atoms along MN `lbo` bytes
// apart, 8-row groups along K `sbo` bytes apart.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// D[tmem] (+)= A[tmem] * B[smem desc], bf16 inputs.
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// An empty statement that the registers pass through (orders their uses
// after the wait that precedes it).
__device__ __forceinline__ void tmem_fence_regs32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                 "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// 32 lanes x 16 columns of 32-bit values stored from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {"
      "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// 2^x by the MUFU approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
// Splits (x0, x1) into two bf16x2 terms hi + lo whose sum is the pair to
// about 2^-17 relative (each term rounds to nearest).
__device__ __forceinline__ void split2_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 r = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t *>(&h);
  lo = *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ bool gwarp_wait(uint32_t bar, uint32_t parity, const volatile int *abort_flag) {
  const bool ok = tc::mbar_wait(bar, parity, abort_flag, kGWaitBudget);
  return __all_sync(0xFFFFFFFFu, ok);
}

// The union tiles of item `it`: slot, KV head, split, first tile and count.
struct GItem {
  int slot, g, s, t0, nt, count;
};
__device__ __forceinline__ GItem group_item(const AttnParams &p, const GroupParams &gp, int it) {
  GItem x;
  const int S = p.num_splits, H = p.num_kv_heads;
  x.slot = it / (H * S);
  x.g = (it / S) % H;
  x.s = it % S;
  x.count = gp.ntiles[x.slot];  // 0: the slot is no group
  const int T = x.count;
  x.t0 = static_cast<int>((static_cast<long long>(x.s) * T) / S);
  x.nt = static_cast<int>((static_cast<long long>(x.s + 1) * T) / S) - x.t0;
  return x;
}

__global__ void __launch_bounds__(kGThreads, 1)
    group_attn_kernel(const AttnParams p, const GroupParams gp, const GroupLayout lay,
                      const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sb = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t q0 = base + lay.off_q;
  const uint32_t bar0 = base + lay.off_bar;
  // barriers: kfull[3] kempty[3] vfull[2] vempty[2] sfull[2] pfull[2] qfull
  // qempty ofull oempty done xsum
  auto KFULL = [&](int s) { return bar0 + 8u * s; };
  auto KEMPTY = [&](int s) { return bar0 + 8u * (kKStages + s); };
  auto VFULL = [&](int s) { return bar0 + 8u * (2 * kKStages + s); };
  auto VEMPTY = [&](int s) { return bar0 + 8u * (2 * kKStages + kVStages + s); };
  auto SFULL = [&](int w) { return bar0 + 8u * (2 * kKStages + 2 * kVStages + w); };
  auto PFULL = [&](int w) { return bar0 + 8u * (2 * kKStages + 2 * kVStages + 2 + w); };
  const uint32_t QFULL = bar0 + 8u * (2 * kKStages + 2 * kVStages + 4), QEMPTY = QFULL + 8, OFULL = QFULL + 16,
                 OEMPTY = QFULL + 24, DONE = QFULL + 32, XSUM = QFULL + 40;
  int *misc = reinterpret_cast<int *>(sb + lay.off_misc);  // [0] tmem base [1] abort
  volatile int *abort_flag = misc + 1;
  const int Hq = p.num_q_heads;
  const int nitems = gp.nslots * p.num_kv_heads * p.num_splits;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(KFULL(s), 1);
      tc::mbar_init(KEMPTY(s), 1 + 4);  // the QK commit + the owning softmax warpgroup (it reads the masks)
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(VFULL(s), 1);
      tc::mbar_init(VEMPTY(s), 1);  // the P V commit
    }
    for (int w = 0; w < 2; ++w) {
      tc::mbar_init(SFULL(w), 1);  // S of warpgroup w's tile is in tensor memory
      tc::mbar_init(PFULL(w), 4);  // its 4 warps wrote P (and rescaled O)
    }
    tc::mbar_init(QFULL, 1);
    tc::mbar_init(QEMPTY, 1);
    tc::mbar_init(OFULL, 1);
    tc::mbar_init(OEMPTY, 8);
    tc::mbar_init(DONE, 1);
    tc::mbar_init(XSUM, 8);  // both warpgroups' row states are written
    misc[1] = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&kmap);
    tc::tma_prefetch_desc(&vmap);
    tc::tma_prefetch_desc(&qmap);
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&misc[0]), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);
  pdl_wait();  // the union and the selection come from the kernels before

  if (warp == 0 || warp == kGWarps - 1) {
    // ========================================================== producers
    // warp 0 stages each item's queries, then its tiles' K rows and row
    // masks into the K ring; the last warp stages the tiles' V rows into
    // the V ring.  Apart, each runs as far ahead as its own ring allows, so
    // the K stream (and the next item's queries) never waits behind V.
    const bool vrole = warp == kGWarps - 1;
    const uint64_t policy = tc::l2_evict_first_policy();
    const uint64_t qpolicy = tc::l2_evict_last_policy();
    int kn = 0, vn = 0, qn = 0;  // K tiles, V tiles and query sets issued
    bool stop = false;
    const int kcol0 = 0, vcol0 = p.kv_interleaved ? p.num_kv_heads * 128 : 0;
    auto wait = [&](uint32_t bar, int parity) {
      if (!gwarp_wait(bar, static_cast<uint32_t>(parity), abort_flag)) {
        if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
        stop = true;
      }
      return !stop;
    };
    for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
      const GItem x = group_item(p, gp, it);
      if (x.nt <= 0) continue;
      const int32_t *pt = p.page_table;
      {
        // the item's request (the union kernel's) from its first member row
        const int row0 = x.slot * kGroupRows + __ffs(static_cast<int>(
                                                   __ballot_sync(0xFFFFFFFFu, lane < kGroupRows &&
                                                                 x.slot * kGroupRows + lane < p.max_rows_attn &&
                                                                 gp.grouped[x.slot * kGroupRows + lane] != 0))) - 1;
        pt += static_cast<size_t>(p.row_req[row0 < 0 ? 0 : row0]) * p.max_pages_per_req;
      }
      if (!vrole) {
        // queries: rows (16 slot rows x 8 heads of g) of the [R * Hq, D] view
        if (!wait(QEMPTY, (qn & 1) ^ 1)) break;
        if (lane == 0) tc::mbar_arrive_expect_tx(QFULL, kQ * 256u);
        __syncwarp();
        if (lane < 2 * kGroupRows) {
          const int j = lane >> 1, a = lane & 1;
          tc::tma_load_2d(q0 + a * (kQ * 128u) + j * 1024u, &qmap, a * 64,
                          (x.slot * kGroupRows + j) * Hq + x.g * 8, QFULL, qpolicy);
        }
        ++qn;
      }
      const int32_t *tiles = gp.tiles + static_cast<size_t>(x.slot) * (gp.umax / kGT);
      const uint32_t *umask = gp.umask + static_cast<size_t>(x.slot) * (gp.umax / kGT) * 64;
      const int P = p.page_size, npg = kGT / P;  // pages per tile: 1, 2, 4 or 8
      for (int t = 0; t < x.nt; ++t) {
        // the tile's 128 positions are npg whole pages: lane 2k + a loads
        // page k's rows of head g, atom a
        const int ti = tiles[x.t0 + t];
        const int k = lane >> 1, a = lane & 1;
        int rowc = -P;  // a page outside the pool (or past the table) reads zeros
        if (lane < 2 * npg) {
          const int pi = ((ti * kGT) >> p.page_shift) + k;
          const int pg = pi < p.max_pages_per_req ? pt[pi] : -1;
          if (pg >= 0 && pg < p.num_pages) rowc = pg * P;
        }
        if (!vrole) {  // K rows and the tile's row masks
          const int ks = kn % kKStages;
          if (!wait(KEMPTY(ks), ((kn / kKStages) & 1) ^ 1)) break;
          if (lane == 0) {
            tc::mbar_arrive_expect_tx(KFULL(ks), kGT * 256u + kGT * 2u);
            tc::bulk_load(base + lay.off_mask + ks * kGT * 2u, umask + static_cast<size_t>(ti) * 64, kGT * 2u,
                          KFULL(ks), qpolicy);
          }
          __syncwarp();
          if (lane < 2 * npg)
            tc::tma_load_2d(base + lay.off_k + ks * (kGT * 256u) + a * (kGT * 128u) + k * P * 128u, &kmap,
                            kcol0 + x.g * 128 + a * 64, rowc, KFULL(ks), policy);
          ++kn;
        } else {  // V rows
          const int vs = vn % kVStages;
          if (!wait(VEMPTY(vs), ((vn / kVStages) & 1) ^ 1)) break;
          if (lane == 0) tc::mbar_arrive_expect_tx(VFULL(vs), kGT * 256u);
          __syncwarp();
          if (lane < 2 * npg)
            tc::tma_load_2d(base + lay.off_v + vs * (kGT * 256u) + a * (kGT * 128u) + k * P * 128u, &vmap,
                            vcol0 + x.g * 128 + a * 64, rowc, VFULL(vs), policy);
          ++vn;
        }
      }
    }
    // no copy may land after the CTA exits
    if (lane == 0) {
      for (int i = max(0, kn - kKStages); i < kn; ++i)
        tc::mbar_wait(KFULL(i % kKStages), (i / kKStages) & 1, nullptr, kGWaitBudget);
      for (int i = max(0, vn - kVStages); i < vn; ++i)
        tc::mbar_wait(VFULL(i % kVStages), (i / kVStages) & 1, nullptr, kGWaitBudget);
      if (qn > 0) tc::mbar_wait(QFULL, (qn - 1) & 1, nullptr, kGWaitBudget);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA
    // The whole warp runs the loop with warp-uniform descriptors and one
    // elected lane (always the same one) issues the MMAs and their commits:
    // a lone issuing thread loses most of the tensor rate to the busy
    // softmax warps that share its scheduler.
    const uint32_t tm = __shfl_sync(0xFFFFFFFFu, tmem, 0);
    const uint32_t idesc_qk = tc::idesc_m128(kGT, false);               // S[q][t]: N = 128 tokens
    const uint32_t idesc_pv = tc::idesc_m128(128, false) | (1u << 16);  // O[q][d]: B (V) MN-major
    const uint64_t dq = desc_kmajor(q0), dk0 = desc_kmajor(base + lay.off_k),
                   dv0 = desc_mnmajor(base + lay.off_v, kGT * 128u, 1024u);
    constexpr uint64_t kAtom = (kGT * 128u) >> 4, kTile = (kGT * 256u) >> 4;  // descriptor address units
    int kn = 0, vn = 0, qn = 0, on = 0, pn[2] = {0, 0};
    bool stop = false, any = false;
    auto wait = [&](uint32_t bar, int parity) {
      if (!gwarp_wait(bar, static_cast<uint32_t>(parity), abort_flag)) stop = true;
      return !stop;
    };
    auto commit = [&](uint32_t bar) {
      if (tc::elect_one()) tc::mma_commit(bar);
      __syncwarp();
    };
    // S_w = Q K^T of the next K tile over the 128 head dims (2 swizzle
    // atoms x 4 k-steps); S_w is free: the P V that read P_w (the same
    // columns) was issued before, and tcgen05 MMAs run in issue order
    auto qk = [&](int w) {
      const int ks = kn % kKStages;
      if (!wait(KFULL(ks), (kn / kKStages) & 1)) return;
      const uint64_t dk = dk0 + ks * kTile;
      if (tc::elect_one()) {
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma<false>(tm + kColS + w * 128, dq + a * ((kQ * 128u) >> 4) + k * 2, dk + a * kAtom + k * 2,
                           idesc_qk, (a | k) != 0 ? 1u : 0u);
        tc::mma_commit(KEMPTY(ks));
        tc::mma_commit(SFULL(w));
      }
      __syncwarp();
      ++kn;
    };
    for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
      const GItem x = group_item(p, gp, it);
      if (x.nt <= 0) continue;
      if (!wait(QFULL, qn & 1)) break;
      ++qn;
      any = true;
      // tile t goes to softmax warpgroup w = t & 1: S_w, P_w (in S_w's
      // columns) and O_w are its own, so the two warpgroups never wait on
      // one another inside the item
      qk(0);
      if (x.nt > 1 && !stop) qk(1);
      if (x.nt <= 2) commit(QEMPTY);  // the item's last S: its queries may go
      if (stop || !wait(OEMPTY, (on & 1) ^ 1)) break;  // the last item's O is read
      tc::tc_fence_after();
      for (int t = 0; t < x.nt && !stop; ++t) {
        const int w = t & 1;
        if (!wait(PFULL(w), pn[w] & 1)) break;
        ++pn[w];
        const int vs = vn % kVStages;
        if (!wait(VFULL(vs), (vn / kVStages) & 1)) break;
        tc::tc_fence_after();  // P_w was written by the softmax warps' tensor-memory stores
        const uint64_t dv = dv0 + vs * kTile;
        // O_w += P_w V: the 128 keys as 8 k-steps of 16 (keys 32 c .. +31
        // have their two bf16 terms at columns 32 c and 32 c + 16)
        if (tc::elect_one()) {
#pragma unroll
          for (int term = 0; term < 2; ++term)
#pragma unroll
            for (int k = 0; k < kGT / 16; ++k)
              mma_tmem_a(tm + kColO + w * 128, tm + kColS + w * 128 + (k >> 1) * 32 + term * 16 + (k & 1) * 8,
                         dv + k * ((16u * 128u) >> 4), idesc_pv, (t >= 2 || term || k) ? 1u : 0u);
          tc::mma_commit(VEMPTY(vs));
        }
        __syncwarp();
        ++vn;
        if (t + 2 < x.nt) {
          qk(w);
          if (t + 3 == x.nt) commit(QEMPTY);
        }
      }
      if (stop) break;
      commit(OFULL);
      ++on;
    }
    if (stop && lane == 0) {
      *abort_flag = 1;
      flag_status(p.status, DSA_DEV_TIMEOUT);
    }
    if (any) {  // every MMA issued here has completed before tensor memory is freed
      commit(DONE);
      if (lane == 0) tc::mbar_wait(DONE, 0, nullptr, kGWaitBudget);
    }
    __syncwarp();
  } else {
    // =========================================================== softmax
    // Two warpgroups: warpgroup w takes the item's tiles t = w, w + 2, ...
    // for all 128 queries (a warp reads the tensor-memory lanes of its
    // quarter), with its own S/P and O accumulator; the two row states are
    // combined once per item.
    const int w = (warp - 2) >> 2;          // softmax warpgroup
    const int quarter = warp & 3;           // tensor-memory lanes 32*quarter .. +31
    const int q = quarter * 32 + lane;      // this thread's query
    const int j = q >> 3, hh = q & 7;       // slot row and query head within the KV group
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t colS = tmem + lane_off + kColS + w * 128, colO = tmem + lane_off + kColO + w * 128;
    const float c = p.sm_scale_log2;
    float *xch = reinterpret_cast<float *>(sb + lay.off_xch);  // [2][3][128]: m, l, exact max per warpgroup
    int kbase = 0, sn = 0, on = 0, xn = 0;  // K tiles of earlier items, S tiles taken, items finished
    bool stop = false;
    auto wait = [&](uint32_t bar, int parity) {
      if (!gwarp_wait(bar, static_cast<uint32_t>(parity), abort_flag)) {
        if (lane == 0) { *abort_flag = 1; flag_status(p.status, DSA_DEV_TIMEOUT); }
        stop = true;
      }
      return !stop;
    };
    const uint32_t *masks_s = reinterpret_cast<const uint32_t *>(sb + lay.off_mask);
    for (int it = blockIdx.x; it < nitems && !stop; it += gridDim.x) {
      const GItem x = group_item(p, gp, it);
      const int row = x.slot * kGroupRows + j;
      if (x.count == 0) continue;  // not a group: the decode kernel has these rows
      const bool member = row < p.max_rows_attn && gp.grouped[row] != 0;
      const size_t rh = (static_cast<size_t>(row) * Hq + x.g * 8 + hh) * p.num_splits + x.s;
      if (x.nt <= 0) {  // an empty split of a group row
        if (member) {
          if (w == 0) {
            p.part_m[rh] = -INFINITY;
            p.part_l[rh] = 0.f;
          }
          for (int d = 64 * w; d < 64 * w + 64; d += 4)
            *reinterpret_cast<float4 *>(p.part_acc + rh * 128 + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      // running maximum m over the tiles: it moves (and l and O_w are scaled
      // by 2^(m_old - m)) only when a tile's row maximum exceeds it by more
      // than 2^8, so p = 2^(x - m) <= 256 and O_w is rarely touched
      float m = -INFINITY, l = 0.f, mtrue = -INFINITY;  // mtrue: the exact maximum
      for (int t = w; t < x.nt && !stop; t += 2) {
        const int kt = kbase + t, ks = kt % kKStages;
        if (!wait(SFULL(w), sn & 1) || !wait(KFULL(ks), (kt / kKStages) & 1)) break;
        ++sn;
        tc::tc_fence_after();
        // this row's selected keys of the tile: bit b of sel[i] = key 32 i + b
        const uint4 sel = *reinterpret_cast<const uint4 *>(masks_s + ks * 64 + j * 4);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(KEMPTY(ks));  // the masks are in registers
        // the unscaled score maximum over them: two loads in flight at a
        // time, eight independent max chains
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll 1
        for (int ch = 0; ch < 4; ch += 2) {
          uint32_t sa[32], sb[32];
          tc::tmem_ld32_nowait(colS + 32 * ch, sa);
          tc::tmem_ld32_nowait(colS + 32 * ch + 32, sb);
          tc::tmem_wait_ld32(sa);
          tmem_fence_regs32(sb);
          const uint32_t wa = ch == 0 ? sel.x : sel.z, wb = ch == 0 ? sel.y : sel.w;
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) {
            if ((wa >> kk) & 1u) mx[kk & 7] = fmaxf(mx[kk & 7], __uint_as_float(sa[kk]));
            if ((wb >> kk) & 1u) mx[kk & 7] = fmaxf(mx[kk & 7], __uint_as_float(sb[kk]));
          }
        }
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float mn = mt * c;  // c > 0: the tile's row maximum of the scaled (log2-domain) scores
        mtrue = fmaxf(mtrue, mn);
        float alpha = 1.f;
        if (m == -INFINITY) {
          m = mn;  // the first selected key of the row (O_w holds no share of this row yet)
        } else if (mn > m + 8.f) {
          alpha = exp2f(m - mn);
          l *= alpha;
          m = mn;
        }
        if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
          // scale the rows' O_w: the P V that last wrote it was issued
          // before this tile's S and has completed with it
#pragma unroll 1
          for (int d0 = 0; d0 < 128; d0 += 16) {
            float o[16];
            tc::tmem_ld16_sync(colO + d0, o);
            uint32_t ob[16];
#pragma unroll
            for (int d = 0; d < 16; ++d) ob[d] = __float_as_uint(o[d] * alpha);
            tmem_st16(colO + d0, ob);
          }
        }
        const float mb = m == -INFINITY ? 0.f : -m;  // no selected key yet: every p is 0
        // keys 32 ch .. +31: P_w's two terms go to S_w's columns of these
        // keys (read just before), hi to 32 ch .. +15 and lo to 32 ch + 16 ..
        float la[4] = {0.f, 0.f, 0.f, 0.f};  // independent sum chains
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tc::tmem_ld32_nowait(colS + 32 * ch, v);
          tc::tmem_wait_ld32(v);
          const uint32_t sw = ch == 0 ? sel.x : ch == 1 ? sel.y : ch == 2 ? sel.z : sel.w;
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float x0 = ((sw >> (2 * k)) & 1u) ? __uint_as_float(v[2 * k]) : -INFINITY;
            const float x1 = ((sw >> (2 * k + 1)) & 1u) ? __uint_as_float(v[2 * k + 1]) : -INFINITY;
            const float p0 = ex2_approx(fmaf(x0, c, mb)), p1 = ex2_approx(fmaf(x1, c, mb));
            la[k & 3] += p0 + p1;
            split2_bf16x2(p0, p1, hi[k], lo[k]);
          }
          tmem_st16(colS + 32 * ch, hi);
          tmem_st16(colS + 32 * ch + 16, lo);
        }
        l += (la[0] + la[1]) + (la[2] + la[3]);
        tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(PFULL(w));  // this warp's rows of P_w are written
      }
      if (stop) break;
      kbase += x.nt;
      // combine the warpgroups' row states: M is the exact maximum, share
      // w of l and O scaled by 2^(m_w - M)
      xch[(w * 3 + 0) * kQ + q] = m;
      xch[(w * 3 + 1) * kQ + q] = l;
      xch[(w * 3 + 2) * kQ + q] = mtrue;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(XSUM);
      if (!wait(XSUM, xn & 1)) break;
      ++xn;
      const float m0 = xch[0 * kQ + q], l0 = xch[1 * kQ + q], t0 = xch[2 * kQ + q];
      const float m1 = xch[3 * kQ + q], l1 = xch[4 * kQ + q], t1 = xch[5 * kQ + q];
      const float M = fmaxf(t0, t1);
      const bool has0 = l0 > 0.f, has1 = l1 > 0.f;  // O_1 is not written when the item has one tile
      const float f0 = has0 ? exp2f(m0 - M) : 0.f, f1 = has1 ? exp2f(m1 - M) : 0.f;
      const float L = l0 * f0 + l1 * f1;
      const bool empty = !(L > 0.f);
      // the split's partial state of this query: warpgroup w writes head
      // dims [64 w, 64 w + 64)
      if (!wait(OFULL, on & 1)) break;
      ++on;
      tc::tc_fence_after();
      const uint64_t keep = tc::l2_evict_last_policy();  // the merge reads them next
      if (member && w == 0) {
        tc::st_global_hint(p.part_m + rh, empty ? -INFINITY : M * kLn2G, keep);
        tc::st_global_hint(p.part_l + rh, empty ? 0.f : L, keep);
      }
      float *dst = p.part_acc + rh * 128 + 64 * w;
#pragma unroll 1
      for (int d0 = 0; d0 < 64; d0 += 16) {
        float oa[16], ob[16];
        tc::tmem_ld16_sync(tmem + lane_off + kColO + 64 * w + d0, oa);
        tc::tmem_ld16_sync(tmem + lane_off + kColO + 128 + 64 * w + d0, ob);
        if (member) {
#pragma unroll
          for (int d = 0; d < 16; d += 4) {
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!empty) {
              r.x = (has0 ? oa[d] * f0 : 0.f) + (has1 ? ob[d] * f1 : 0.f);
              r.y = (has0 ? oa[d + 1] * f0 : 0.f) + (has1 ? ob[d + 1] * f1 : 0.f);
              r.z = (has0 ? oa[d + 2] * f0 : 0.f) + (has1 ? ob[d + 2] * f1 : 0.f);
              r.w = (has0 ? oa[d + 3] * f0 : 0.f) + (has1 ? ob[d + 3] * f1 : 0.f);
            }
            *reinterpret_cast<float4 *>(dst + d0 + d) = r;
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(OEMPTY);
    }
  }

  // ---- teardown: every role is out of its loop and its async work is done
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 group_tensor_map_encoder() {
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

}  // namespace

bool group_path_enabled(const dsa_config_t &cfg) {
  return (cfg.flags & DSA_FLAG_NO_PREFILL_GROUPS) == 0 && cfg.block_rows > 1 &&
         cfg.num_kv_heads * 8 == cfg.num_q_heads && cfg.head_dim == 128 && cfg.max_rows >= kGroupRows;
}

int32_t group_union_capacity(const dsa_config_t &cfg) {
  // a union of 16 top-k lists holds at most 16 topk positions and must fill
  // a quarter of the group's span: spans past 64 topk never form a group
  const long long u = std::min<long long>(cfg.score_width, 4LL * kGroupRows * cfg.topk);
  return static_cast<int32_t>((u + kGT - 1) / kGT * kGT);
}

cudaError_t launch_group_union(const dsa_config_t &cfg, const AttnParams &p, const GroupParams &gp, cudaStream_t st) {
  (void)cfg;
  constexpr int smem = kUnionSpan / 2 * 4;
  cudaError_t e = cudaFuncSetAttribute(group_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(group_union_kernel, dim3(static_cast<unsigned>(gp.nslots)), dim3(kUnionThreads), smem, st, 1u, p, gp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_group_attn(const dsa_config_t &cfg, const AttnParams &p, const GroupParams &gp, cudaStream_t st) {
  auto encode = group_tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  GroupLayout lay;
  uint32_t off = 0;
  lay.off_q = off;
  off += kQ * 256u;                           // Q: 2 swizzle atoms of [128 queries x 128 B]
  lay.off_k = off;
  off += kKStages * kGT * 256u;               // K tiles: 2 swizzle atoms of [128 rows x 128 B]
  lay.off_v = off;
  off += kVStages * kGT * 256u;               // V tiles, the same
  lay.off_mask = off;
  off += kKStages * kGT * 2u;                 // per K tile: 16 rows x 128 bits
  lay.off_xch = off;
  off += 6 * kQ * 4u;                         // the warpgroups' row states
  lay.off_bar = off;
  off += (2 * kKStages + 2 * kVStages + 10) * 8u;
  lay.off_misc = off;
  off += 16u;
  const size_t smem = off + 1024;
  // K and V rows: 2-D views [num_pages * page_size rows, row elements], one
  // box = 64 elements (128 B) of one page's rows
  const cuuint64_t rows = static_cast<cuuint64_t>(cfg.num_pages) * cfg.page_size;
  const cuuint64_t row_elems = static_cast<cuuint64_t>(cfg.num_kv_heads) * cfg.head_dim * (p.kv_interleaved ? 2 : 1);
  const cuuint64_t gdim[2] = {row_elems, rows};
  const cuuint64_t gstride[1] = {row_elems * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(cfg.page_size)};
  const cuuint32_t es[2] = {1, 1};
  CUtensorMap kmap, vmap, qmap;
  CUresult cr = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t *>(p.k_cache), gdim, gstride,
                       box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // with the interleaved cache the V rows are columns Hkv*D.. of the same rows
  cr = encode(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<uint8_t *>(p.kv_interleaved ? p.k_cache : p.v_cache), gdim, gstride, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // queries: [max_rows * Hq rows, 128], one box = 8 heads x 64 elements
  const cuuint64_t qdim[2] = {128, static_cast<cuuint64_t>(cfg.max_rows) * cfg.num_q_heads};
  const cuuint64_t qstride[1] = {256};
  const cuuint32_t qbox[2] = {64, 8};
  cr = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t *>(p.q), qdim, qstride, qbox, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(group_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int items = gp.nslots * cfg.num_kv_heads * cfg.num_splits;
  const int grid = std::max(1, std::min(items, sms));
  e = launch_pdl(group_attn_kernel, dim3(grid), dim3(kGThreads), smem, st, 1u, p, gp, lay, kmap, vmap, qmap);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
