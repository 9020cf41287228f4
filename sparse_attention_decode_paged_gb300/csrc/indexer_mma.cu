// Lightning-indexer scores, warp-level tensor-core version (mma.sync).
//
//   scores[r, t] = s_t * sum_h w[r, h] * max(0, q_idx[r, h, :] . k_t),  t < row_len[r]
//
// Megatron-LM PR #7211, commit message 1: the indexer streams page-contiguous
// key tiles through tensor cores, and each request's programs stride over its
// row only up to its length; commit message 2: rows of one score block share
// each key tile.
//
// Grid: (ceil(W / chunk), max_rows block slots).  CTA (x, b) scores tokens
// [x*chunk, (x+1)*chunk) of score block b against all rows of the block;
// CTAs past the block's longest row exit at once, so the work follows the
// real lengths while the launch depends only on the static config.
//
// Per CTA: the block's indexer queries (<= 4 rows x H_I heads x D_I) sit in
// shared memory; key tiles of 128 tokens stream through a 3-stage cp.async
// ring (16-byte copies, addresses resolved through the page table; rows
// padded by 16 bytes so ldmatrix is conflict-free).  fp8 keys are widened to
// bf16 in shared memory (exact: every e4m3 value is a bf16 value) and the
// per-token scale multiplies the finished score.  Warp w owns tokens
// [16w, 16w+16) of a tile: A = keys (16 tokens x 16 dims per k-step, from
// ldmatrix), B = queries (8 heads per n-tile); the accumulator fragment holds
// q_h . k_t for 2 tokens x 2 heads per lane, which is ReLU'd, weighted and
// summed over heads in registers, then across the 4 lanes of a quad.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kTT = 128;         // tokens per key tile
constexpr int kWarps = 8;        // warp w owns tokens [16w, 16w+16) of a tile
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kChunkTiles = 16;  // key tiles per CTA
constexpr int kChunkTokens = kChunkTiles * kTT;

template <int DI, bool FP8>
struct Layout {
  static constexpr int kRowB = DI * 2 + 16;                  // padded bf16 row
  static constexpr int kSrcRowB = FP8 ? DI : DI * 2;         // bytes per token in the cache
  static constexpr int kRawRowB = kSrcRowB + 16;             // padded staged row
  static constexpr int kRawTileB = kTT * kRawRowB;
  static constexpr int kChunksPerRow = kSrcRowB / 16;
};

__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&h));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t *>(&b);
}

template <int DI, bool FP8>
__global__ void __launch_bounds__(kThreads, 1) indexer_mma_kernel(const IndexerParams p) {
  using Lay = Layout<DI, FP8>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.y;
  const int nrows = p.block_nrows[blk];
  if (nrows <= 0) return;
  const int first = p.block_first[blk];
  const int HP = (p.idx_heads + 7) & ~7;

  // ---- validate the score block (every thread reaches the same verdict)
  bool ok = nrows <= p.block_rows && first >= 0 && first + nrows <= p.max_rows;
  int req = 0, lmax = 0;
  int lens[4] = {0, 0, 0, 0};
  if (ok) {
    req = p.row_req[first];
    ok = req >= 0 && req < p.max_reqs;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i < nrows && ok) {
        const int L = p.row_len[first + i];
        if (p.row_req[first + i] != req || L < 0 || L > p.score_width) ok = false;
        lens[i] = L;
        lmax = max(lmax, L);
      }
    }
  }
  if (!ok) {
    if (tid == 0 && blockIdx.x == 0) flag_status(p.status, DSA_DEV_BAD_BLOCK);
    return;
  }
  const int t_begin = blockIdx.x * kChunkTokens;
  if (t_begin >= lmax) return;
  const int t_end = min(lmax, t_begin + kChunkTokens);
  const int ntiles = (t_end - t_begin + kTT - 1) / kTT;

  uint8_t *q_s = smem;
  float *w_s = reinterpret_cast<float *>(smem + p.block_rows * HP * Lay::kRowB);
  uint8_t *stage_s = smem + p.block_rows * HP * (Lay::kRowB + 4);
  uint8_t *conv_s = stage_s + kStages * Lay::kRawTileB;  // fp8 only

  // ---- the block's indexer queries and head weights
  constexpr int kQChunks = DI / 8;  // 16-byte pieces of one bf16 query row
  for (int i = tid; i < nrows * HP * kQChunks; i += kThreads) {
    const int c = i % kQChunks, hh = (i / kQChunks) % HP, rr = i / (kQChunks * HP);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (hh < p.idx_heads)
      v = *reinterpret_cast<const uint4 *>(
          p.q_idx + ((static_cast<size_t>(first + rr) * p.idx_heads + hh) * DI + c * 8) * 2);
    *reinterpret_cast<uint4 *>(q_s + (rr * HP + hh) * Lay::kRowB + c * 16) = v;
  }
  for (int i = tid; i < nrows * HP; i += kThreads) {
    const int hh = i % HP, rr = i / HP;
    w_s[i] = hh < p.idx_heads ? p.w[static_cast<size_t>(first + rr) * p.idx_heads + hh] : 0.f;
  }

  const int32_t *pt = p.page_table + static_cast<size_t>(req) * p.max_pages_per_req;
  const int P = p.page_size;

  auto load_tile = [&](int tile, int stage) {
    const int t0 = t_begin + tile * kTT;
    const uint32_t dst0 = smem_u32(stage_s + stage * Lay::kRawTileB);
    for (int i = tid; i < kTT * Lay::kChunksPerRow; i += kThreads) {
      const int j = i / Lay::kChunksPerRow, c = i % Lay::kChunksPerRow;
      const int t = t0 + j;
      const uint8_t *src = p.idx_cache;
      int bytes = 0;
      if (t < t_end) {
        const int page = pt[t / P];
        if (page >= 0 && page < p.num_pages) {
          src = p.idx_cache +
                (static_cast<size_t>(page) * P + (t % P)) * Lay::kSrcRowB + c * 16;
          bytes = 16;
        } else {
          flag_status(p.status, DSA_DEV_BAD_PAGE);
        }
      }
      cp_async_16(dst0 + j * Lay::kRawRowB + c * 16, src, bytes);
    }
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s, s);
    cp_async_commit();
  }

  for (int tile = 0; tile < ntiles; ++tile) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nt = tile + kStages - 1;
      if (nt < ntiles) load_tile(nt, nt % kStages);
      cp_async_commit();
    }
    const uint8_t *tile_s = stage_s + (tile % kStages) * Lay::kRawTileB;
    if constexpr (FP8) {
      for (int i = tid; i < kTT * (DI / 8); i += kThreads) {
        const int j = i / (DI / 8), c = i % (DI / 8);
        const uint2 raw = *reinterpret_cast<const uint2 *>(tile_s + j * Lay::kRawRowB + c * 8);
        uint4 o;
        o.x = e4m3x2_to_bf16x2(raw.x & 0xFFFFu);
        o.y = e4m3x2_to_bf16x2(raw.x >> 16);
        o.z = e4m3x2_to_bf16x2(raw.y & 0xFFFFu);
        o.w = e4m3x2_to_bf16x2(raw.y >> 16);
        *reinterpret_cast<uint4 *>(conv_s + j * Lay::kRowB + c * 16) = o;
      }
      __syncthreads();
      tile_s = conv_s;
    }
    const int tw = t_begin + tile * kTT + warp * 16;  // first token of this warp
    if (tw < t_end) {
      uint32_t a[DI / 16][4];
      const uint32_t abase =
          smem_u32(tile_s) + (warp * 16 + (lane & 15)) * Lay::kRowB + (lane >> 4) * 16;
#pragma unroll
      for (int ks = 0; ks < DI / 16; ++ks)
        ldmatrix_x4(abase + ks * 32, a[ks][0], a[ks][1], a[ks][2], a[ks][3]);

      // per-token scale of the two tokens this lane may write
      const int ta = tw + (lane >> 2), tb = ta + 8;
      float sc_a = 1.f, sc_b = 1.f;
      if (FP8 && (lane & 3) == 0) {
        sc_a = sc_b = 0.f;
        if (ta < t_end) {
          const int pg = pt[ta / P];
          if (pg >= 0 && pg < p.num_pages) sc_a = p.idx_scale[static_cast<size_t>(pg) * P + ta % P];
        }
        if (tb < t_end) {
          const int pg = pt[tb / P];
          if (pg >= 0 && pg < p.num_pages) sc_b = p.idx_scale[static_cast<size_t>(pg) * P + tb % P];
        }
      }
#pragma unroll 1
      for (int rr = 0; rr < nrows; ++rr) {
        float s0 = 0.f, s1 = 0.f;
        const uint32_t qbase =
            smem_u32(q_s + rr * HP * Lay::kRowB) + (lane & 7) * Lay::kRowB + (lane >> 3) * 16;
        const float *wr = w_s + rr * HP;
#pragma unroll 1
        for (int nt = 0; nt < HP / 8; ++nt) {
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int ks = 0; ks < DI / 16; ks += 2) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(qbase + nt * 8 * Lay::kRowB + ks * 32, b0, b1, b2, b3);
            mma_bf16_16816(acc, a[ks][0], a[ks][1], a[ks][2], a[ks][3], b0, b1);
            mma_bf16_16816(acc, a[ks + 1][0], a[ks + 1][1], a[ks + 1][2], a[ks + 1][3], b2, b3);
          }
          const int h0 = nt * 8 + 2 * (lane & 3);
          const float w0 = wr[h0], w1 = wr[h0 + 1];
          s0 += w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);
          s1 += w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);
        }
        s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 1);
        s0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 2);
        s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 1);
        s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 2);
        if ((lane & 3) == 0) {
          int L = lens[0];
#pragma unroll
          for (int i = 1; i < 4; ++i)
            if (rr == i) L = lens[i];
          float *srow = p.scores + static_cast<size_t>(first + rr) * p.score_width;
          if (ta < L) srow[ta] = s0 * sc_a;
          if (tb < L) srow[tb] = s1 * sc_b;
        }
      }
    }
  }
  cp_async_wait<0>();
}

template <int DI, bool FP8>
cudaError_t launch_t(const dsa_config_t &cfg, const IndexerParams &p, cudaStream_t st) {
  using Lay = Layout<DI, FP8>;
  const int HP = (cfg.idx_heads + 7) & ~7;
  const size_t smem = static_cast<size_t>(cfg.block_rows) * HP * (Lay::kRowB + 4) +
                      kStages * Lay::kRawTileB + (FP8 ? kTT * Lay::kRowB : 0);
  cudaError_t e = cudaFuncSetAttribute(indexer_mma_kernel<DI, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid((cfg.score_width + kChunkTokens - 1) / kChunkTokens, cfg.max_rows);
  indexer_mma_kernel<DI, FP8><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer(const dsa_config_t &cfg, const IndexerParams &p, cudaStream_t st) {
  const bool fp8 = cfg.idx_key_dtype == DSA_KEY_FP8_E4M3;
  switch (cfg.idx_dim) {
    case 32: return fp8 ? launch_t<32, true>(cfg, p, st) : launch_t<32, false>(cfg, p, st);
    case 64: return fp8 ? launch_t<64, true>(cfg, p, st) : launch_t<64, false>(cfg, p, st);
    case 128: return fp8 ? launch_t<128, true>(cfg, p, st) : launch_t<128, false>(cfg, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
