// Read-only stream probe: the bandwidth a plain read of given pages reaches
// on this GPU, the reference beside which the streaming kernels' rates are
// reported.  Not part of the DSA path (a separate library that only the
// benchmark loads).
//
// Each warp reads whole pages (in the caller's order, e.g. the page-table
// order a step visits them) with eight independent 16-byte loads per lane in
// flight and folds them into one word, so no byte can be skipped; one word
// per warp is written to `sink`.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void read_pages_kernel(const uint4 *base, const int32_t *order, int32_t npages, int32_t page_u4,
                                  uint32_t *sink) {
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  uint32_t acc = 0u;
  for (int pg = warp; pg < npages; pg += nwarps) {
    const int phys = order != nullptr ? order[pg] : pg;
    const uint4 *src = base + static_cast<size_t>(phys) * page_u4;
    for (int i = lane; i < page_u4; i += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = i + u * 32 < page_u4 ? __ldcs(src + i + u * 32) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 8; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0 && sink != nullptr) sink[warp] = acc;
}

}  // namespace

// Reads `npages` pages of `page_bytes` (a multiple of 16; `base` 16-byte
// aligned) in `order` (device int32 [npages] of page indices, or NULL for
// 0..npages-1).  `sink` receives one word per warp: blocks_per_sm * SMs *
// threads / 32 words.  Returns a cudaError_t value (0 on success).
extern "C" int dsa_probe_read_pages(const void *base, const int32_t *order, int32_t npages, int32_t page_bytes,
                                    uint32_t *sink, int32_t blocks_per_sm, int32_t threads, cudaStream_t stream) {
  if (base == nullptr || npages <= 0 || page_bytes <= 0 || (page_bytes & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(base) & 15) != 0 || threads <= 0 || (threads & 31) != 0 || blocks_per_sm <= 0)
    return static_cast<int>(cudaErrorInvalidValue);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return static_cast<int>(e);
  read_pages_kernel<<<blocks_per_sm * sms, threads, 0, stream>>>(static_cast<const uint4 *>(base), order, npages,
                                                                  page_bytes / 16, sink);
  return static_cast<int>(cudaGetLastError());
}
