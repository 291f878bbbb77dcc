// tv_tree_attn_verify_static: the attention call for callers that cannot
// allocate device memory.  The split partials live in one file-scope device
// array of TV_STATIC_SCRATCH_BYTES, whose device address is passed to
// tv_tree_attn_verify as the workspace.
#include <cuda_runtime.h>

#include "internal.h"
#include "treeverify.h"

namespace {

// In host code this name stands in for the array; only the address returned
// by cudaGetSymbolAddress (per device, with that device current) may be
// handed to a kernel.
static __device__ __align__(256) unsigned char g_static_scratch[TV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// the address the last uncaptured call found, per device, for calls made
// during a stream capture (where no lookup is made)
std::atomic<void*> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" {

tv_status tv_tree_attn_verify_static(const void* q, const void* k_cache, const void* v_cache,
                                     int64_t cap, int32_t prefix_len, int32_t n_nodes,
                                     const int32_t* parent, void* out, int32_t hq, int32_t hkv,
                                     int32_t d, int32_t dtype, float scale, int32_t* dev_status,
                                     tv_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TV_ERR_CUDA;
  const size_t need = tv_attn_workspace_size(n_nodes, hq, hkv, d, dtype, prefix_len);
  if (need > TV_STATIC_SCRATCH_BYTES) return TV_ERR_CAPACITY;
  cudaStreamCaptureStatus cap_status = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap_status) != cudaSuccess)
    return TV_ERR_CUDA;
  void* addr = nullptr;
  if (cap_status == cudaStreamCaptureStatusNone) {
    // a fresh lookup: a device reset or a new primary context since the
    // last call moves the array
    if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || addr == nullptr)
      return TV_ERR_CUDA;
    g_scratch_addr[dev].store(addr);
  } else {
    addr = g_scratch_addr[dev].load();
    if (addr == nullptr) return TV_ERR_CUDA;
  }
  return tv_tree_attn_verify(q, k_cache, v_cache, cap, prefix_len, n_nodes, parent, out, hq, hkv,
                             d, dtype, scale, addr, TV_STATIC_SCRATCH_BYTES, dev_status, stream);
}

}  // extern "C"
