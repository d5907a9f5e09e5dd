// decode.cuh -- parameters of the split-KV decode kernel (shared with api.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace vpp {

// One decode row of a mixed batch.
struct DecodeRow {
  int32_t b;      // sequence index (row of the block table)
  int32_t q_row;  // packed query row in q/out
  int32_t ctx;    // keys 0 .. ctx-1 (the row's own token included)
  int32_t item0;  // first work item (key range) of this row
};

struct DecodeParams {
  int32_t n_rows;
  int32_t heads;
  int32_t kv_heads;
  int32_t split_tokens;        // keys per work item (multiple of 16)
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  float scale_log2;
  int32_t n_items;             // work items of the launch (set by launch_decode)
  const uint16_t* q;           // bf16 [total_q][heads][d]
  const void* k_cache;         // [num_blocks][64][kv_heads][d], bf16 or E4M3 codes
  const void* v_cache;
  const float* k_scale;        // E4M3 cache: [kv_heads] factors (null for bf16)
  const float* v_scale;
  const int32_t* block_table;  // [batch][max_blocks_per_seq]
  uint16_t* out;               // bf16 [total_q][heads][d]
  float* lse;                  // [heads][lse_stride], may be null
  int64_t lse_stride;
  float* ws_o;                 // float32 [items][heads][d] partials
  float* ws_lse;               // [items][heads]
  int* status;
  // Top-k mode (topk_idx != null): query token i of one chunk (prefix
  // topk_prefix) attends the key positions topk_idx[i][0 .. topk_len[i]-1]
  // of the sequence in block-table row 0; rows[] and n_rows are unused.
  const int32_t* topk_idx;     // [n_tokens][topk]
  const int32_t* topk_len;     // [n_tokens]
  int32_t topk;                // row stride of topk_idx (the list capacity k)
  int32_t topk_splits;         // work items per token: ceil(k / split_tokens)
  int64_t topk_prefix;
  int64_t topk_tokens;
  DecodeRow rows[kMaxBatch];
};

// Keys per decode work item.
constexpr int kDecodeSplitTokens = 1024;

// True when the decode kernel handles this shape (dq = dv in {64, 128},
// kv_heads <= 8, heads / kv_heads in {1, 2, 4, 8}).
bool decode_supported(int head_dim_qk, int head_dim_v, int heads, int kv_heads);

// fp8: the cache holds E4M3 codes with per-kv-head k_scale / v_scale.
// topk: p.topk_idx rows instead of decode rows (items = tokens x topk_splits).
// ctas > 0: at most that many CTAs, each taking every ctas-th item (one
// resident CTA per SM on a bf16 cache, two on an fp8 one); 0: one CTA per
// item.
cudaError_t launch_decode(const DecodeParams& p, int items, int head_dim, bool fp8, bool topk, int num_sms,
                          int ctas, cudaStream_t stream);

}  // namespace vpp
