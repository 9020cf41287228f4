// Sparse GQA attention over the selected keys (split) and the split merge.
//
// Megatron-LM PR #7211, commit message 1: all query heads of a KV group are
// handled together so each selected key and value row is read once, and the
// top-k slots are split across programs whose slices are merged flash-decoding
// style; commit message 8: probabilities enter the value reduction in fp32.
//
// sparse_attn_kernel: grid (S splits, R rows), one warp per KV head g.  The
// warp walks its split's slots 16 at a time: lanes 0..15 resolve slot ->
// position -> page -> row offset (bounds-checked), every lane issues its
// 16-byte loads of two K rows (scores) and 8-byte loads of all 16 V rows
// before any arithmetic, so 8 KiB per warp are in flight.  Scores use the
// tensor cores (mma.sync m16n8k16, A = 16 keys x 16 dims, B = the group's <= 8
// query heads) with the head dim permuted identically on both operands so
// each lane's key bytes are one contiguous 16-byte load.  The online softmax
// runs in the log2 domain in fp32; p (fp32, never rounded) and the rescale
// factors go through shared memory and every lane accumulates its 4 (D=128)
// or 2 (D=64) value dims for all heads with fp32 FMA.
//
// merge_kernel: one warp per (row, head); combines the S partial states.
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kChunk = 16;       // selected keys per warp iteration
constexpr int kMaxKvHeads = 16;  // warps per CTA
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct VecV;
template <>
struct VecV<128> {
  using T = uint2;  // 4 bf16
  static constexpr int kN = 4;
  __device__ __forceinline__ static T load(const uint8_t *p) { return ldg_nc_v2(p); }
  __device__ __forceinline__ static void unpack(const T &v, float (&f)[4]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  }
  __device__ __forceinline__ static T zero() { return make_uint2(0u, 0u); }
};
template <>
struct VecV<64> {
  using T = uint32_t;  // 2 bf16
  static constexpr int kN = 2;
  __device__ __forceinline__ static T load(const uint8_t *p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];\n" : "=r"(r) : "l"(p));
    return r;
  }
  __device__ __forceinline__ static void unpack(const T &v, float (&f)[2]) {
    f[0] = bf16lo(v); f[1] = bf16hi(v);
  }
  __device__ __forceinline__ static T zero() { return 0u; }
};

template <int D>
__global__ void __launch_bounds__(32 * kMaxKvHeads) sparse_attn_kernel(const AttnParams p) {
  using V = VecV<D>;
  constexpr int KJ = D / 32;  // 16-byte pieces of a key row per lane quad
  constexpr int VN = V::kN;   // value dims per lane
  __shared__ float p_s[kMaxKvHeads][kChunk][8];
  __shared__ float a_s[kMaxKvHeads][8];

  const int s = blockIdx.x, r = blockIdx.y;
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c4 = lane & 3, g4 = lane >> 2;
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, G = Hq / Hkv, S = p.num_splits;
  const int K = p.topk, P = p.page_size;

  int L = p.row_len[r];
  const int req = p.row_req[r];
  const bool row_ok = L >= 0 && L <= p.score_width && (L == 0 || (req >= 0 && req < p.max_reqs));
  if (!row_ok) {
    if (lane == 0) flag_status(p.status, DSA_DEV_BAD_ROW);
    L = 0;
  }
  const int n = min(K, L);
  const int a = static_cast<int>((static_cast<long long>(s) * n) / S);
  const int b = static_cast<int>((static_cast<long long>(s + 1) * n) / S);

  // query heads of this group as the B operand (dims permuted, see header)
  uint4 qf[KJ];
#pragma unroll
  for (int j = 0; j < KJ; ++j) {
    qf[j] = make_uint4(0u, 0u, 0u, 0u);
    if (g4 < G)
      qf[j] = *reinterpret_cast<const uint4 *>(
          p.q + ((static_cast<size_t>(r) * Hq + g * G + g4) * D + 32 * j + 8 * c4) * 2);
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2c4, 2c4+1 (log2 domain)
  float acc[8][VN];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int d = 0; d < VN; ++d) acc[h][d] = 0.f;

  const int32_t *sel = p.topk_idx + static_cast<size_t>(r) * K;
  const int32_t *pt =
      p.page_table + static_cast<size_t>(L > 0 ? req : 0) * p.max_pages_per_req;
  const long long tok_stride = static_cast<long long>(Hkv) * D;  // elements per token

  for (int base = a; base < b; base += kChunk) {
    long long off = -1;  // element offset of row (t, g) in the caches; -1 = skip
    if (lane < kChunk) {
      const int i = base + lane;
      if (i < b) {
        const int t = sel[i];
        if (t != -1) {
          if (t < 0 || t >= L) {
            flag_status(p.status, DSA_DEV_BAD_INDEX);
          } else {
            const int page = pt[t / P];
            if (page < 0 || page >= p.num_pages)
              flag_status(p.status, DSA_DEV_BAD_PAGE);
            else
              off = (static_cast<long long>(page) * P + (t % P)) * tok_stride +
                    static_cast<long long>(g) * D;
          }
        }
      }
    }
    const long long ok0 = __shfl_sync(0xFFFFFFFFu, off, g4);
    const long long ok1 = __shfl_sync(0xFFFFFFFFu, off, g4 + 8);
    uint4 kf0[KJ], kf1[KJ];
#pragma unroll
    for (int j = 0; j < KJ; ++j) {
      kf0[j] = ok0 >= 0 ? ldg_nc_v4(p.k_cache + (ok0 + 32 * j + 8 * c4) * 2) : make_uint4(0u, 0u, 0u, 0u);
      kf1[j] = ok1 >= 0 ? ldg_nc_v4(p.k_cache + (ok1 + 32 * j + 8 * c4) * 2) : make_uint4(0u, 0u, 0u, 0u);
    }
    typename V::T vv[kChunk];
    bool vok[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const long long ov = __shfl_sync(0xFFFFFFFFu, off, i);
      vok[i] = ov >= 0;
      vv[i] = vok[i] ? V::load(p.v_cache + (ov + lane * VN) * 2) : V::zero();
    }

    // scores S^T[token][head] = K . Q^T
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < KJ; ++j) {
      mma_bf16_16816(c, kf0[j].x, kf1[j].x, kf0[j].y, kf1[j].y, qf[j].x, qf[j].y);
      mma_bf16_16816(c, kf0[j].z, kf1[j].z, kf0[j].w, kf1[j].w, qf[j].z, qf[j].w);
    }
    const float x0 = ok0 >= 0 ? c[0] * p.sm_scale_log2 : -INFINITY;
    const float x1 = ok0 >= 0 ? c[1] * p.sm_scale_log2 : -INFINITY;
    const float x2 = ok1 >= 0 ? c[2] * p.sm_scale_log2 : -INFINITY;
    const float x3 = ok1 >= 0 ? c[3] * p.sm_scale_log2 : -INFINITY;
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, o));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
    const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
    const float p0 = x0 == -INFINITY ? 0.f : exp2f(x0 - mn0);
    const float p1 = x1 == -INFINITY ? 0.f : exp2f(x1 - mn1);
    const float p2 = x2 == -INFINITY ? 0.f : exp2f(x2 - mn0);
    const float p3 = x3 == -INFINITY ? 0.f : exp2f(x3 - mn1);
    float ps0 = p0 + p2, ps1 = p1 + p3;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      ps0 += __shfl_xor_sync(0xFFFFFFFFu, ps0, o);
      ps1 += __shfl_xor_sync(0xFFFFFFFFu, ps1, o);
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
    m0 = mn0;
    m1 = mn1;
    p_s[g][g4][2 * c4] = p0;
    p_s[g][g4][2 * c4 + 1] = p1;
    p_s[g][g4 + 8][2 * c4] = p2;
    p_s[g][g4 + 8][2 * c4 + 1] = p3;
    if (g4 == 0) {
      a_s[g][2 * c4] = al0;
      a_s[g][2 * c4 + 1] = al1;
    }
    __syncwarp();
    {
      const float4 alo = *reinterpret_cast<const float4 *>(&a_s[g][0]);
      const float4 ahi = *reinterpret_cast<const float4 *>(&a_s[g][4]);
      const float al[8] = {alo.x, alo.y, alo.z, alo.w, ahi.x, ahi.y, ahi.z, ahi.w};
#pragma unroll
      for (int h = 0; h < 8; ++h)
#pragma unroll
        for (int d = 0; d < VN; ++d) acc[h][d] *= al[h];
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (!vok[i]) continue;
      const float4 plo = *reinterpret_cast<const float4 *>(&p_s[g][i][0]);
      const float4 phi = *reinterpret_cast<const float4 *>(&p_s[g][i][4]);
      const float pv[8] = {plo.x, plo.y, plo.z, plo.w, phi.x, phi.y, phi.z, phi.w};
      float vf[VN];
      V::unpack(vv[i], vf);
#pragma unroll
      for (int h = 0; h < 8; ++h)
#pragma unroll
        for (int d = 0; d < VN; ++d) acc[h][d] = fmaf(pv[h], vf[d], acc[h][d]);
    }
    __syncwarp();
  }

  // partial state of heads g*G .. g*G+G-1 for split s
  const size_t rh0 = static_cast<size_t>(r) * Hq + static_cast<size_t>(g) * G;
  if (g4 == 0) {
    const int h0 = 2 * c4, h1 = 2 * c4 + 1;
    if (h0 < G) {
      p.part_m[(rh0 + h0) * S + s] = m0 == -INFINITY ? -INFINITY : m0 * kLn2;
      p.part_l[(rh0 + h0) * S + s] = l0;
    }
    if (h1 < G) {
      p.part_m[(rh0 + h1) * S + s] = m1 == -INFINITY ? -INFINITY : m1 * kLn2;
      p.part_l[(rh0 + h1) * S + s] = l1;
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < G) {
      float *dst = p.part_acc + ((rh0 + h) * S + s) * D + lane * VN;
      if constexpr (VN == 4) {
        *reinterpret_cast<float4 *>(dst) = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      } else {
        *reinterpret_cast<float2 *>(dst) = make_float2(acc[h][0], acc[h][1]);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  constexpr int VN = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long rh = static_cast<long long>(blockIdx.x) * 8 + warp;  // (row, head)
  if (rh >= static_cast<long long>(p.max_rows) * p.num_q_heads) return;
  const int S = p.num_splits;
  const float *pm = p.part_m + rh * S, *pl = p.part_l + rh * S;
  float ms0 = -INFINITY, ms1 = -INFINITY, ls0 = 0.f, ls1 = 0.f;
  if (lane < S) { ls0 = pl[lane]; ms0 = ls0 > 0.f ? pm[lane] : -INFINITY; }
  if (lane + 32 < S) { ls1 = pl[lane + 32]; ms1 = ls1 > 0.f ? pm[lane + 32] : -INFINITY; }
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
  for (int s2 = 0; s2 < S; ++s2) {
    const float fs = __shfl_sync(0xFFFFFFFFu, s2 < 32 ? f0 : f1, s2 & 31);
    if (fs != 0.f) {
      const float *src = p.part_acc + (rh * S + s2) * D + lane * VN;
      if constexpr (VN == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        o[0] = fmaf(fs, v.x, o[0]); o[1] = fmaf(fs, v.y, o[1]);
        o[2] = fmaf(fs, v.z, o[2]); o[3] = fmaf(fs, v.w, o[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        o[0] = fmaf(fs, v.x, o[0]); o[1] = fmaf(fs, v.y, o[1]);
      }
    }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + rh * D + lane * VN;
#pragma unroll
  for (int d = 0; d < VN; d += 2)
    *reinterpret_cast<__nv_bfloat162 *>(dst + d) = __floats2bfloat162_rn(o[d] * inv, o[d + 1] * inv);
  if (p.lse && lane == 0) p.lse[rh] = lsum > 0.f ? mx + logf(lsum) : -INFINITY;
}

}  // namespace

cudaError_t launch_sparse_attn(const dsa_config_t &cfg, const AttnParams &p, cudaStream_t st) {
  const dim3 grid(cfg.num_splits, cfg.max_rows);
  const int threads = 32 * cfg.num_kv_heads;
  if (cfg.head_dim == 128) sparse_attn_kernel<128><<<grid, threads, 0, st>>>(p);
  else if (cfg.head_dim == 64) sparse_attn_kernel<64><<<grid, threads, 0, st>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_merge(const dsa_config_t &cfg, const MergeParams &p, cudaStream_t st) {
  const long long pairs = static_cast<long long>(cfg.max_rows) * cfg.num_q_heads;
  const unsigned blocks = static_cast<unsigned>((pairs + 7) / 8);
  if (cfg.head_dim == 128) merge_kernel<128><<<blocks, 256, 0, st>>>(p);
  else if (cfg.head_dim == 64) merge_kernel<64><<<blocks, 256, 0, st>>>(p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace dsa
