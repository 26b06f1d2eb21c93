// tree_attn_forward_noalloc: the tree attention entry point for callers that
// cannot allocate device memory.
//
// Who needs it: code embedded in a host framework that owns every byte of
// device memory through its own pool (it hands kernels inputs and outputs,
// never raw cudaMalloc scratch), and latency-critical loops where a
// cudaMalloc/cudaFree would implicitly synchronize the device and stall the
// stream.  Such callers cannot size and pass the workspace that
// tree_attn_forward takes.
//
// How: the split-KV scratch (partial outputs, their log-sum-exps and the
// device error word) lives in one file-scope device array of kScratchBytes.
// Every GPU that loads the library reserves it until the process exits.  Host
// code cannot use the array's name as a device address, so on the first call
// on each device (with that device current) the entry point looks the address
// up with cudaGetSymbolAddress and caches it; that first call should come
// before any stream capture.  The cache is not refreshed: after a
// cudaDeviceReset the module (and the array) may be loaded elsewhere, so this
// entry point must not be used on a device that has been reset.  The call
// then runs the ordinary tree_attn_forward path with the array as its
// workspace, choosing a split-KV CTA count small enough for the partials to
// fit.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (nullptr on failure).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" TS_API ts_status tree_attn_forward_noalloc(const ts_attn_args* args, void* stream) {
  if (args == nullptr) return TS_ERR_INVALID_ARG;
  void* scratch = scratch_address();
  if (scratch == nullptr) return TS_ERR_CUDA;
  ts_attn_args a = *args;
  size_t need = tree_attn_workspace_size(&a);
  if (need == 0) {
    const int path = tree_attn_selected_path(&a);
    return path < 0 ? static_cast<ts_status>(-path) : TS_ERR_INVALID_ARG;
  }
  if (need > kScratchBytes) {
    // fewer split-KV CTAs need fewer partial slots: take the largest count that fits
    int lo = 1, hi = a.num_ctas > 0 ? a.num_ctas : 4096;
    a.num_ctas = 1;
    if (tree_attn_workspace_size(&a) > kScratchBytes) return TS_ERR_UNSUPPORTED;  // too large even unsplit
    while (lo < hi) {
      const int mid = lo + (hi - lo + 1) / 2;
      a.num_ctas = mid;
      if (tree_attn_workspace_size(&a) <= kScratchBytes) lo = mid;
      else hi = mid - 1;
    }
    a.num_ctas = lo;
  }
  // The array keeps the previous call's contents; the error word must start
  // at zero (partial slots are written before they are read).
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t zero_bytes = ts::attn_zero_prefix_bytes(&a);
  if (zero_bytes == 0 || cudaMemsetAsync(scratch, 0, zero_bytes, s) != cudaSuccess) return TS_ERR_CUDA;
  return tree_attn_forward(&a, scratch, kScratchBytes, stream);
}
