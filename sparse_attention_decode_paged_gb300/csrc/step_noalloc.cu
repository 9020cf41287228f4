// dsa_step_noalloc: the fused step with library-owned scratch memory.
//
// Some callers cannot allocate device memory for the step's workspace: code
// that runs while a CUDA graph is being captured (cudaMalloc is not a
// capturable operation), runtimes whose device memory belongs to another
// allocator that must not be bypassed or fragmented, and plain C hosts that
// have no device allocator of their own.  This entry point gives them the
// step with its intermediates (status word, scores, top-k, split partials,
// prefill-group region, key histogram) in a fixed-size array that lives in
// this library's device image.  The caller still passes every input and
// output.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  Its
// device address is looked up once per device with cudaGetSymbolAddress on
// the first call made on that device (with the device current); that first
// call must therefore happen outside stream capture.  All calls on a device
// share the one array and it keeps the last call's contents.  The status word
// is cleared at the start of each call.  The key histogram must start at
// zero: a step leaves its own histogram region at zero (the top-k clears
// each row's counts after using them), but the region's offset and size
// follow the config, so a call whose layout differs from the previous
// call's on that device first clears its histogram region on `stream`.
// Scores, top-k, the prefill-group region and the partials are rewritten
// before they are read.
// Calls whose executions overlap on the GPU (different streams, or graphs
// replayed concurrently) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_step_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};
// key-histogram region (offset, bytes) of the last call on each device; a
// region of 0 bytes means unknown (no call yet, or a call that failed)
size_t g_hist_off[kMaxDevices] = {};
size_t g_hist_bytes[kMaxDevices] = {};

}  // namespace

extern "C" dsa_status_t dsa_step_noalloc(const dsa_config_t *cfg, const dsa_step_args_t *args,
                                         uint32_t *status_out, dsa_stream_t stream) {
  dsa_status_t st = dsa_validate_config(cfg);
  if (st != DSA_OK) return st;
  size_t need = 0;
  st = dsa_workspace_size(cfg, &need);
  if (st != DSA_OK) return st;
  if (need > kNoAllocScratchBytes) {
    return dsa::set_error(DSA_ERR_CAPACITY,
                          "dsa_step_noalloc: this config needs %zu bytes of scratch, the built-in "
                          "array holds %zu; use dsa_step with a caller workspace",
                          need, kNoAllocScratchBytes);
  }
  if (status_out != nullptr && (reinterpret_cast<uintptr_t>(status_out) & 3u) != 0)
    return dsa::set_error(DSA_ERR_INVALID_ARG, "status_out is not 4-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dsa::set_error(DSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return dsa::set_error(DSA_ERR_UNSUPPORTED, "device %d", dev);
  dsa_workspace_layout_t lay;
  st = dsa_workspace_layout(cfg, &lay);
  if (st != DSA_OK) return st;
  const size_t hist_bytes = lay.total - lay.key_hist;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_step_scratch);
    if (e != cudaSuccess)
      return dsa::set_error(DSA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  char *ws = static_cast<char *>(g_scratch_ptr[dev]);
  const bool same_layout = g_hist_bytes[dev] == hist_bytes && g_hist_off[dev] == lay.key_hist;
  g_hist_bytes[dev] = 0;  // unknown until this call has been queued in full
  e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream);  // the status word starts at zero
  if (e != cudaSuccess) return dsa::set_error(DSA_ERR_CUDA, "clear status: %s", cudaGetErrorString(e));
  if (!same_layout) {  // the new histogram region holds the previous call's other data
    e = cudaMemsetAsync(ws + lay.key_hist, 0, hist_bytes, stream);
    if (e != cudaSuccess) return dsa::set_error(DSA_ERR_CUDA, "clear histogram: %s", cudaGetErrorString(e));
  }
  st = dsa_step(cfg, args, ws, stream);
  if (st != DSA_OK) return st;
  if (status_out != nullptr) {
    e = cudaMemcpyAsync(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return dsa::set_error(DSA_ERR_CUDA, "copy status: %s", cudaGetErrorString(e));
  }
  g_hist_off[dev] = lay.key_hist;
  g_hist_bytes[dev] = hist_bytes;
  return DSA_OK;
}
