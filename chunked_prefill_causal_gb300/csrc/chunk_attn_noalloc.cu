// chunk_attn_noalloc.cu -- chunk attention for callers that cannot allocate.
//
// Some callers may not call cudaMalloc (or any allocator) on their execution
// path and have no scratch buffer to hand over: for example a plug-in run by
// an inference runtime that owns all device memory and fixes the budget at
// start-up, or a binding that only exposes the plain signature.  For them,
// vpp_chunk_attn_noalloc keeps the float32 partials of a key-split chunk
// attention in a fixed file-scope device array instead of a caller workspace.
// The array is kNoallocScratchBytes (32 MiB); every GPU that loads this
// library holds it until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host the name
// is only a stand-in for the device object.  The device address is looked up
// once per device with cudaGetSymbolAddress, with that device current, on the
// first call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "vpp.h"

namespace vpp {
int run_chunk_attn(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                   const int32_t* block_table, int32_t num_blocks, int64_t prefix_len,
                   int64_t chunk_len, int heads, int kv_heads, int head_dim_qk, int head_dim_v,
                   float softmax_scale, int num_splits, void* out, float* lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);
}  // namespace vpp

namespace {

constexpr size_t kNoallocScratchBytes = static_cast<size_t>(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (set-up once per
// device, under a lock).  The library's kernels are built for compute
// capability 10.3 only, so any other device is refused before the lookup; a
// failed lookup clears the runtime's error state so that the caller's next
// cudaGetLastError does not report it a second time.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VPP_ERR_CUDA;
  if (dev < 0 || dev >= 64) return VPP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return VPP_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return VPP_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return VPP_ERR_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return VPP_OK;
}

// Scratch bytes that a call with this split request needs (q is bf16, so only
// the split partials), or a negative status.
int64_t scratch_need(int64_t P, int64_t C, int heads, int kv_heads, int dq, int dv, int splits) {
  const int s = vpp_chunk_attn_num_splits(P, C, heads, kv_heads, dq, dv, splits);
  if (s < 0) return s;
  return static_cast<int64_t>(
      vpp_chunk_attn_workspace_size(VPP_BF16, P, C, heads, kv_heads, dq, dv, splits));
}

}  // namespace

extern "C" int vpp_chunk_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_table, int32_t num_blocks,
                                      int64_t prefix_len, int64_t chunk_len, int heads,
                                      int kv_heads, int head_dim_qk, int head_dim_v,
                                      float softmax_scale, int num_splits, void* out, float* lse,
                                      void* stream) {
  if (prefix_len < 0 || chunk_len < 0 || num_splits < 0) return VPP_ERR_INVALID;
  if (chunk_len == 0) return VPP_OK;
  int64_t need = scratch_need(prefix_len, chunk_len, heads, kv_heads, head_dim_qk, head_dim_v,
                              num_splits);
  if (need < 0) return static_cast<int>(need);
  if (num_splits == 0 && need > static_cast<int64_t>(kNoallocScratchBytes)) {
    // The library's own choice of key ranges does not fit the array: take the
    // largest explicit count whose partials do (one range needs none).
    int s = vpp_chunk_attn_num_splits(prefix_len, chunk_len, heads, kv_heads, head_dim_qk,
                                      head_dim_v, 0);
    while (s > 1) {
      --s;
      need = scratch_need(prefix_len, chunk_len, heads, kv_heads, head_dim_qk, head_dim_v, s);
      if (need < 0) return static_cast<int>(need);
      if (need <= static_cast<int64_t>(kNoallocScratchBytes)) break;
    }
    num_splits = s;
    if (s == 1) need = 0;
  }
  if (need > static_cast<int64_t>(kNoallocScratchBytes)) return VPP_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    if (int r = scratch_address(&scratch)) return r;
  }
  // No value in the scratch needs to start at zero: for every (range, token,
  // head) row the merge reads, this call's attention kernel writes the
  // partial output and its LSE first.
  return vpp::run_chunk_attn(q, VPP_BF16, k_cache, v_cache, block_table, num_blocks, prefix_len,
                             chunk_len, heads, kv_heads, head_dim_qk, head_dim_v, softmax_scale,
                             num_splits, out, lse, scratch, need > 0 ? kNoallocScratchBytes : 0,
                             static_cast<cudaStream_t>(stream));
}
