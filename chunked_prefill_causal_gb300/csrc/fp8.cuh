// fp8.cuh -- fp8 (E4M3) KV-cache launchers shared by api.cu and kv_fp8.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace vpp {

// Sequences whose cached keys 0 .. ctx-1 are widened to bf16: entry i reads
// block-table row table_row[i] and writes rows base[i] .. base[i+1]-1 of the
// contiguous output (base[i+1] - base[i] = that sequence's key count).
struct WidenPlan {
  int32_t n;
  int32_t max_blocks_per_seq;    // row stride of the block table
  int32_t table_row[kMaxBatch];
  int64_t base[kMaxBatch + 1];
};

cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                 const float* k_scale, const float* v_scale, const int32_t* block_table,
                                 int32_t num_blocks, int64_t prefix_len, int64_t chunk_len, int kv_heads,
                                 int dq, int dv, int* status, int num_sms, cudaStream_t stream);

cudaError_t launch_kv_append_fp8_varlen(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                        const float* k_scale, const float* v_scale,
                                        const int32_t* block_table, const VarlenPlan& plan,
                                        int32_t num_blocks, int kv_heads, int dq, int dv, int* status,
                                        int num_sms, cudaStream_t stream);

// block_table == nullptr: one contiguous cache [capacity][kv_heads][d] (n = 1).
cudaError_t launch_kv_widen_fp8(const void* k_cache, const void* v_cache, uint16_t* k_out, uint16_t* v_out,
                                int kv_heads, int dq, int dv, const int32_t* block_table,
                                int32_t num_blocks, const WidenPlan& plan, int* status, int num_sms,
                                cudaStream_t stream);

}  // namespace vpp
