// common.cuh -- types shared by the host launch code and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vpp {

constexpr int kBlockTokens = 64;    // paged KV block ("02 · 并行策略与 PP 切分" note, §1)
constexpr int kMaxBatch = 1024;     // sequences per mixed micro-batch (plan passed by value)

// Per-sequence description of a varlen batch, passed to kernels by value.
struct VarlenPlan {
  int32_t batch;
  int32_t max_blocks_per_seq;       // row stride of the block table
  int32_t cu_q[kMaxBatch + 1];      // packed query/new-token row offsets
  int32_t ctx[kMaxBatch];           // total keys of each sequence (incl. new tokens)
};

// Kernel launchers (defined in the .cu files, called from api.cu).
cudaError_t launch_kv_append(const void* k_new, const void* v_new, bool in_fp32, void* k_cache,
                             void* v_cache, const int32_t* block_table, int32_t num_blocks,
                             int64_t prefix_len, int64_t chunk_len, int kv_heads, int dq, int dv,
                             int* status, int num_sms, cudaStream_t stream);

cudaError_t launch_kv_append_varlen(const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* block_table,
                                    const VarlenPlan& plan, int32_t num_blocks, int kv_heads,
                                    int dq, int dv, int* status, int num_sms,
                                    cudaStream_t stream);

cudaError_t launch_convert_f32_bf16(const float* in, uint16_t* out, int64_t n, int num_sms,
                                    cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(int timeout_us, int* status, cudaStream_t stream);

}  // namespace vpp
